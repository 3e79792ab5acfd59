"""GPU parity of the fp32 forward (fa_forward_f32) against the float64 oracle.

Tolerances: max-abs 1e-5 on O, 1e-3 on LSE.  Inputs are seeded; the fp32 path
gets exactly the values the oracle reads.
"""
import numpy as np
import pytest

import oracle
from tiled_online_softmax_sm_gb300 import binding as fb
from tiled_online_softmax_sm_gb300 import inputs as I

from _helpers import F32_MAX_ABS, assert_close, assert_lse_close, dev, host

pytestmark = pytest.mark.gpu


def _run(case):
    o, lse = fb.forward_f32(dev(case.q), dev(case.k), dev(case.v), case.scale, case.causal)
    o_ref, lse_ref = oracle.attention(case.q.values, case.k.values, case.v.values, case.scale,
                                      case.causal)
    assert_close(host(o), o_ref, F32_MAX_ABS, what=case.name)
    assert_lse_close(host(lse), lse_ref, what=case.name)
    return host(o), o_ref


@pytest.mark.parametrize("hot", [False, True])
def test_c1_single_head_256(hot):
    """Single-head non-causal fp32, n=m=256, d=dv=64, scale 1/8 (+ x10 hot copy)."""
    _run(I.c1_fp32(hot=hot))


@pytest.mark.parametrize("shape", [
    # B, H, Hkv, n, m, d, dv, causal
    (2, 4, 2, 130, 130, 64, 64, True),
    (1, 3, 1, 77, 200, 128, 128, False),
    (2, 2, 2, 1, 1, 64, 128, False),
    (1, 2, 1, 97, 97, 128, 64, True),
    (1, 1, 1, 5, 333, 64, 64, False),
    (1, 2, 1, 40, 130, 64, 64, True),
    (2, 2, 2, 130, 40, 128, 128, True),
    # several key tiles per key group, ragged last tile; and the causal
    # diagonal crossing the groups' tiles
    (1, 2, 2, 64, 1000, 64, 64, False),
    (1, 2, 1, 700, 700, 64, 128, True),
])
def test_fp32_shapes(shape):
    B, H, Hkv, n, m, d, dv, causal = shape
    case = I.dense_case(123, B, H, n, m, d, dv=dv, Hkv=Hkv, dtype="f32", causal=causal,
                        name=f"f32_{shape}")
    _run(case)


def test_fp32_hot_causal():
    case = I.dense_case(7, 1, 2, 300, 300, 64, dtype="f32", causal=True, hot=10.0, name="f32_hot_causal")
    _run(case)


def test_fp32_no_keys_gives_zero_and_neg_inf():
    import torch
    q = torch.randn(1, 4, 1, 64, device="cuda")
    k = torch.empty(1, 0, 1, 64, device="cuda")
    v = torch.empty(1, 0, 1, 64, device="cuda")
    o, lse = fb.forward_f32(q, k, v, 0.125, False)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
