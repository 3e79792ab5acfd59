"""GPU parity of the e4m3 (FP8) forward, fa_forward_fp8, against the float64
oracle run on the exact dequantised inputs (code value x power-of-two descale).

Tolerance (stated, from the arithmetic): the inputs carry no error here (the
oracle sees the same values).  The path rounds each weight p_j to e4m3 (3
mantissa bits: relative error at most 2^-4) before P V, so for every row
|O - O_ref| <= 2^-4 * sum_j w_j |v_j| <= 2^-4 * max|V|, plus the bf16 rounding of
O (2^-8 |O|): that bound is the max-abs tolerance.  Where the weight is spread
over many keys the errors average out; the mean-abs tolerance is 8e-3 (4x the
bf16 path's).  LSE does not involve P: 1e-3 as for bf16.
"""
import numpy as np
import pytest
import torch

import oracle
from tiled_online_softmax_sm_gb300 import binding as fb
from tiled_online_softmax_sm_gb300 import inputs as I

from _helpers import assert_close, assert_lse_close, host

pytestmark = pytest.mark.gpu

FP8_MEAN_ABS = 8e-3


def _case(seed, B, H, Hkv, n, m, causal, hot=1.0):
    g = I.rng(seed, 81)
    x = [I.normal_f32(g, shp) for shp in ((B, n, H, 128), (B, m, Hkv, 128), (B, m, Hkv, 128))]
    x[0] *= np.float32(hot)
    x[1] *= np.float32(hot)
    return [I.Tensor.from_f32(t, "e4m3") for t in x], I.fp32_scale(128)


def _run(q, k, v, scale, causal, rows=None, what=""):
    dq, dk, dv_ = (torch.from_numpy(t.data).cuda() for t in (q, k, v))
    o, lse = fb.forward_fp8(dq, dk, dv_, scale, q.descale, k.descale, v.descale, causal)
    if rows is None:
        o_ref, lse_ref = oracle.attention(q.values, k.values, v.values, scale, causal)
        got_o, got_l = host(o), host(lse)
    else:
        o_ref, lse_ref = oracle.attention_rows(q.values, k.values, v.values, scale, causal, rows)
        oh, lh = host(o), host(lse)
        got_o = oh[rows[:, 0], rows[:, 2], rows[:, 1]]
        got_l = lh[rows[:, 0], rows[:, 1], rows[:, 2]]
    err = np.abs(got_o - o_ref)
    bound = 2.0 ** -4 * float(np.abs(v.values).max()) + 2.0 ** -8 * float(np.abs(o_ref).max())
    print(f"\n[fp8] {what}: max-abs {err.max():.3e} (bound {bound:.3e}) mean-abs {err.mean():.3e}")
    assert_close(got_o, o_ref, bound, FP8_MEAN_ABS, what=what)
    assert_lse_close(got_l, lse_ref, what=what)
    assert fb.fa_get_device_status() == 0


@pytest.mark.parametrize("shape", [(1, 2, 1, 300, 300, True), (2, 4, 2, 517, 517, False),
                                   (1, 2, 2, 1, 1, False), (1, 4, 2, 100, 700, True)])
def test_fp8_small(shape, capsys):
    B, H, Hkv, n, m, causal = shape
    (q, k, v), scale = _case(91, B, H, Hkv, n, m, causal)
    with capsys.disabled():
        _run(q, k, v, scale, causal, what=f"fp8 {shape}")


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_hot(causal, capsys):
    (q, k, v), scale = _case(92, 1, 2, 2, 640, 640, causal, hot=10.0)
    with capsys.disabled():
        _run(q, k, v, scale, causal, what=f"fp8 hot causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_batched_prefill_sampled(causal, capsys):
    """B=4, H=16, n=m=2048, d=128 (the batched-prefill shape), sampled rows."""
    (q, k, v), scale = _case(93, 4, 16, 16, 2048, 2048, causal)
    g = I.rng(94)
    rows = np.stack([g.integers(0, 4, 4096), g.integers(0, 16, 4096), g.integers(0, 2048, 4096)],
                    1).astype(np.int32)
    with capsys.disabled():
        _run(q, k, v, scale, causal, rows=rows, what=f"fp8 B4 H16 2048 causal={causal}")
