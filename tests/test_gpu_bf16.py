"""GPU parity of the bf16 tcgen05 forward (fa_forward, fa_forward_varlen).

Against the float64 oracle run on the same bf16-rounded inputs: O max-abs
2e-2 and mean-abs 2e-3, LSE max-abs 1e-3, on every output element, small
cases and full-size workloads alike (the full-size ones in the launch
configuration the bench times).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tiled_online_softmax_sm_gb300 import binding as fb
from tiled_online_softmax_sm_gb300 import inputs as I

from _helpers import BF16_MAX_ABS, BF16_MEAN_ABS, assert_close, assert_lse_close, dev, dev_i32, host

pytestmark = pytest.mark.gpu


def _gpu(case):
    return fb.forward(dev(case.q), dev(case.k), dev(case.v), case.scale, case.causal)


def _check_full(case):
    o, lse = _gpu(case)
    o_ref, lse_ref = oracle.attention(case.q.values, case.k.values, case.v.values, case.scale,
                                      case.causal)
    assert_close(host(o), o_ref, BF16_MAX_ABS, BF16_MEAN_ABS, what=case.name)
    assert_lse_close(host(lse), lse_ref, what=case.name)
    assert fb.fa_get_device_status() == 0


@pytest.mark.parametrize("shape", [
    # B, H, Hkv, n, m, d, causal
    (1, 2, 1, 300, 300, 128, True),
    (2, 3, 3, 517, 517, 64, True),
    (1, 2, 2, 200, 777, 128, False),
    (1, 1, 1, 1, 1, 128, False),
    (1, 1, 1, 1, 1, 64, True),
    (2, 4, 2, 256, 256, 128, False),
    (1, 2, 1, 129, 129, 64, False),
    (1, 2, 2, 384, 384, 128, True),
    (3, 2, 1, 640, 100, 64, False),
    # causal with n != m: bottom-right (queries are the last n key positions)
    (1, 2, 1, 100, 300, 128, True),
    (2, 4, 2, 300, 100, 64, True),
    (1, 2, 2, 129, 700, 128, True),
    (1, 8, 2, 64, 1000, 128, True),
    (1, 2, 1, 1, 513, 64, True),
])
def test_small_shapes(shape):
    B, H, Hkv, n, m, d, causal = shape
    _check_full(I.dense_case(31, B, H, n, m, d, Hkv=Hkv, causal=causal, name=f"bf16_{shape}"))


@pytest.mark.parametrize("shape", [
    # B, H, Hkv, n, m, d: pair units B*H*ceil(n/256) past the 152 SMs, so the
    # last wave runs as split units (one query tile, keys halved between the
    # two warpgroups, merged in the CTA)
    (1, 160, 160, 256, 300, 128),    # 160 units: 8 in the last wave
    (1, 158, 79, 200, 1000, 64),     # a ragged second query tile, grouped heads
    (2, 80, 40, 512, 129, 128),      # 320 units: 16 in the last wave, 2 K/V tiles each
    (1, 170, 170, 256, 1024, 64),    # 18 in the last wave
])
def test_last_wave_split_units(shape):
    B, H, Hkv, n, m, d = shape
    _check_full(I.dense_case(35, B, H, n, m, d, Hkv=Hkv, causal=False, name=f"split {shape}"))


@pytest.mark.parametrize("shape", [
    # B, H, Hkv, n, m, d, causal: pair units, and (last row) split units
    (1, 2, 1, 300, 300, 128, True),
    (2, 3, 3, 517, 517, 64, False),
    (1, 160, 160, 256, 300, 128, False),
])
def test_output_on_a_16_byte_boundary_gives_the_same_bits(shape):
    """O that starts 16 bytes past a 32-byte boundary is written with 16-byte
    stores instead of 32-byte ones: the bits must not change."""
    B, H, Hkv, n, m, d, causal = shape
    c = I.dense_case(36, B, H, n, m, d, Hkv=Hkv, causal=causal, name=f"o16 {shape}")
    q, k, v = dev(c.q), dev(c.k), dev(c.v)
    o_a, lse_a = fb.forward(q, k, v, c.scale, causal)
    numel = B * n * H * d
    buf = torch.empty(numel + 64, dtype=torch.bfloat16, device="cuda")
    off = (16 - buf.data_ptr() % 32) % 32 // 2   # elements to 16 bytes past a 32-byte boundary
    o_b = buf[off:off + numel].view(B, n, H, d)
    assert o_b.data_ptr() % 32 == 16
    lse_b = torch.empty_like(lse_a)
    fb.fa_forward(q, k, v, o_b, lse_b, B, H, Hkv, n, m, d, d, c.scale, causal)
    torch.cuda.synchronize()
    assert fb.fa_get_device_status() == 0
    assert torch.equal(o_a.view(torch.int16), o_b.view(torch.int16))
    assert torch.equal(lse_a, lse_b)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_hot_x10(causal, d):
    # at d=64 O's divisor comes from the P V MMA's extra columns of ones
    _check_full(I.dense_case(32, 1, 2, 640, 640, d, causal=causal, hot=10.0, name=f"hot d={d}"))


def test_no_keys_gives_zero_and_neg_inf():
    q = torch.randn(1, 5, 2, 128, device="cuda").bfloat16()
    k = torch.empty(1, 0, 2, 128, device="cuda").bfloat16()
    o, lse = fb.forward(q, k, k, 0.088, False)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


@pytest.mark.parametrize("variant", ["full", "causal", "hot"])
def test_c2_full_size_every_output(variant):
    """Batched prefill bf16: B=4, H=16, n=m=2048, d=dv=128 (non-causal, causal,
    x10 hot), every element of O and LSE."""
    _check_full(I.c2_bf16(causal=variant == "causal", hot=variant == "hot"))


def test_c3_full_size_every_output():
    """Long-context causal prefill bf16: B=1, H=32, n=m=8192, d=dv=128, every
    element of O and LSE."""
    _check_full(I.c3_bf16())


# ----------------------------------------------------------------- varlen
def _varlen_gpu(case):
    T = int(case.cu_seqlens[-1])
    cu = dev_i32(case.cu_seqlens)
    mx = int(case.lens.max()) if len(case.lens) else 0
    return fb.forward_varlen(dev(case.q), dev(case.k), dev(case.v), cu, cu, mx, mx, case.scale,
                             case.causal)


@pytest.mark.parametrize("d", [64, 128])
def test_varlen_small_full(d):
    lens = [1, 2, 127, 128, 129, 255, 256, 257, 5, 300]
    case = I.varlen_case(41, lens, H=4, d=d, Hkv=2)
    o, lse = _varlen_gpu(case)
    o_ref, lse_ref = oracle.varlen(case.q.values, case.k.values, case.v.values, case.cu_seqlens,
                                   case.cu_seqlens, case.scale, True)
    assert_close(host(o), o_ref, BF16_MAX_ABS, BF16_MEAN_ABS, what=f"varlen d={d}")
    assert_lse_close(host(lse), lse_ref, what=f"varlen d={d}")
    assert fb.fa_get_device_status() == 0


def test_varlen_noncausal_and_empty_sequence():
    lens = [40, 0, 200]
    case = I.varlen_case(42, lens, H=2, d=128, causal=False)
    o, lse = _varlen_gpu(case)
    o_ref, lse_ref = oracle.varlen(case.q.values, case.k.values, case.v.values, case.cu_seqlens,
                                   case.cu_seqlens, case.scale, False)
    assert_close(host(o), o_ref, BF16_MAX_ABS, BF16_MEAN_ABS)
    assert_lse_close(host(lse), lse_ref)


@pytest.mark.parametrize("d", [64, 128])
def test_c5_varlen_full_size_every_output(d):
    """Ragged causal varlen: 16 sequences, lengths uniform on [1, 4096], H=16,
    10% of Q and K rows x20; every element of O and LSE."""
    case = I.c5_varlen(d)
    o, lse = _varlen_gpu(case)
    o_ref, lse_ref = oracle.varlen(case.q.values, case.k.values, case.v.values, case.cu_seqlens,
                                   case.cu_seqlens, case.scale, True)
    assert_close(host(o), o_ref, BF16_MAX_ABS, BF16_MEAN_ABS, what=f"c5 d={d}")
    assert_lse_close(host(lse), lse_ref, what=f"c5 d={d}")
    assert fb.fa_get_device_status() == 0


@pytest.mark.parametrize("seed", [50, 51])
@pytest.mark.parametrize("d", [64, 128])
def test_ragged_hot_batches_of_other_seeds_every_output(seed, d):
    """The ragged workload's recipe (16 lengths uniform on [1, 4096], 10% of Q
    and K rows x20) with other seeds: rows that one hot key dominates, with V
    entries past 5, in other places."""
    lens = I.uniform_lengths(seed, 16, 1, 4096, stream=5, tensor=9)
    _varlen_full_check(lens, seed, H=16, d=d, what=f"ragged seed {seed} d={d}")


def test_varlen_offsets_outside_buffers_are_rejected_on_device():
    case = I.varlen_case(44, [10, 20], H=2, d=64)
    cu_bad = case.cu_seqlens.copy()
    cu_bad[-1] = 999                     # past the 30 rows of the buffers
    q, k, v = dev(case.q), dev(case.k), dev(case.v)
    o = torch.zeros((30, 2, 64), dtype=torch.bfloat16, device="cuda")
    fb.fa_forward_varlen(q, k, v, o, None, dev_i32(cu_bad), dev_i32(cu_bad), 2, 30, 30, 999, 999,
                         2, 2, 64, 64, case.scale, 1)
    assert fb.fa_get_device_status() == fb.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("d", [64, 128])
def test_varlen_causal_unequal_q_and_k_lengths(d):
    """Chunked-prefill shape: each sequence's queries are its last q_len key
    positions (bottom-right causal), with q_len < k_len, = k_len and > k_len."""
    q_lens = [50, 128, 200, 1, 300]
    k_lens = [400, 128, 120, 77, 1000]
    H, Hkv = 4, 2
    cu_q = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(k_lens)]).astype(np.int32)
    g = I.rng(45, d)
    q = I.Tensor.from_f32(I.normal_f32(g, (int(cu_q[-1]), H, d)), "bf16")
    k = I.Tensor.from_f32(I.normal_f32(g, (int(cu_k[-1]), Hkv, d)), "bf16")
    v = I.Tensor.from_f32(I.normal_f32(g, (int(cu_k[-1]), Hkv, d)), "bf16")
    scale = I.fp32_scale(d)
    o, lse = fb.forward_varlen(dev(q), dev(k), dev(v), dev_i32(cu_q), dev_i32(cu_k), max(q_lens),
                               max(k_lens), scale, True)
    o_ref, lse_ref = oracle.varlen(q.values, k.values, v.values, cu_q, cu_k, scale, True)
    assert_close(host(o), o_ref, BF16_MAX_ABS, BF16_MEAN_ABS, what=f"varlen q!=k d={d}")
    assert_lse_close(host(lse), lse_ref, what=f"varlen q!=k d={d}")
    assert fb.fa_get_device_status() == 0


def _varlen_full_check(lens, seed, H=2, d=64, causal=True, what="", hot_frac=0.10):
    case = I.varlen_case(seed, lens, H=H, d=d, causal=causal, hot_frac=hot_frac)
    o, lse = _varlen_gpu(case)
    o_ref, lse_ref = oracle.varlen(case.q.values, case.k.values, case.v.values, case.cu_seqlens,
                                   case.cu_seqlens, case.scale, causal)
    assert_close(host(o), o_ref, BF16_MAX_ABS, BF16_MEAN_ABS, what=what)
    assert_lse_close(host(lse), lse_ref, what=what)
    assert fb.fa_get_device_status() == 0
    return case, o, lse


def test_varlen_schedule_boundary_and_fallback():
    """512 (sequence, query pair) combinations take the persistent sorted
    schedule; 600 take one CTA per unit.  Both match the oracle on every row,
    with the ragged workload's hot rows (10% of Q and K rows x20)."""
    g = I.rng(46, 0)
    at_limit = g.integers(257, 513, size=256).tolist()     # 256 sequences x 2 pairs = 512
    _varlen_full_check(at_limit, 47, what="512 combinations")
    past = g.integers(1, 257, size=600).tolist()           # 600 sequences x 1 pair
    past[5] = 0                                              # an empty one among them
    _varlen_full_check(past, 48, what="600 combinations")


def test_varlen_result_does_not_depend_on_sequence_order():
    """Reordering the sequences of a packed batch changes which CTA runs which
    unit (the schedule sorts by size) but not a single output bit."""
    lens = [300, 17, 1000, 0, 129, 640, 1, 256]
    case = I.varlen_case(49, lens, H=4, d=128)
    o1, l1 = _varlen_gpu(case)
    perm = [6, 2, 0, 7, 4, 1, 5, 3]
    cu = case.cu_seqlens
    seg = lambda x, s: x[cu[s]:cu[s + 1]]
    q2 = np.concatenate([seg(case.q.data, s) for s in perm])
    k2 = np.concatenate([seg(case.k.data, s) for s in perm])
    v2 = np.concatenate([seg(case.v.data, s) for s in perm])
    lens2 = [lens[s] for s in perm]
    cu2 = np.concatenate([[0], np.cumsum(lens2)]).astype(np.int32)
    mx = max(lens)
    o2, l2 = fb.forward_varlen(dev(I.Tensor("bf16", q2, None)), dev(I.Tensor("bf16", k2, None)),
                               dev(I.Tensor("bf16", v2, None)), dev_i32(cu2), dev_i32(cu2), mx, mx,
                               case.scale, True)
    o1h, o2h = o1.view(torch.int16).cpu().numpy(), o2.view(torch.int16).cpu().numpy()
    l1h, l2h = l1.view(torch.int32).cpu().numpy(), l2.view(torch.int32).cpu().numpy()
    for j, s in enumerate(perm):
        assert np.array_equal(o1h[cu[s]:cu[s + 1]], o2h[cu2[j]:cu2[j + 1]]), f"sequence {s}"
        assert np.array_equal(l1h[:, cu[s]:cu[s + 1]], l2h[:, cu2[j]:cu2[j + 1]]), f"sequence {s}"


def test_varlen_sequence_with_65535_key_tiles_is_scheduled():
    """The sorted schedule's per-combination work count is 16 bits wide: one
    query row against 65535 * 128 keys makes 1 + 65535 tile steps, which must
    saturate rather than wrap to 0 (a combination with 0 work is skipped).
    Closed form: Q = 0 gives every key the same score, so O is the mean of V
    and LSE = ln m; V row t is (t mod 8) / 8 in every column, whose mean over
    whole periods is 7/16, and every partial sum the kernel forms is an
    integer multiple of 1/8 below 2^22, so the result is exact."""
    m = 65535 * 128
    d = 64
    q = torch.zeros((1, 1, d), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((m, 1, d), dtype=torch.bfloat16, device="cuda")
    v = ((torch.arange(m, device="cuda") % 8).to(torch.float32) / 8).to(torch.bfloat16)
    v = v[:, None, None].expand(m, 1, d).contiguous()
    o = torch.zeros((1, 1, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 1), dtype=torch.float32, device="cuda")
    cu_q = dev_i32([0, 1])
    cu_k = dev_i32([0, m])
    fb.fa_forward_varlen(q, k, v, o, lse, cu_q, cu_k, 1, 1, m, 1, m, 1, 1, d, d, d ** -0.5, 0)
    assert fb.fa_get_device_status() == 0
    assert torch.all(o.float() == 0.4375), o.float().unique()
    assert abs(float(lse[0, 0]) - math.log(m)) < 1e-5


# ------------------------------------------------- non-finite V next door
_BF16_INF = np.uint16(0x7F80)
_BF16_NAN = np.uint16(0x7FC0)


def _poison_rows(t, rows):
    """A copy of inputs.Tensor t with rows (first axis) set to inf and NaN
    alternately, bit patterns and oracle values alike."""
    data = t.data.copy()
    vals = t.values.copy()
    for n_, r in enumerate(rows):
        data[r] = _BF16_INF if n_ % 2 == 0 else _BF16_NAN
        vals[r] = np.inf if n_ % 2 == 0 else np.nan
    return I.Tensor("bf16", data, vals)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_dense_nonfinite_v_of_next_batch_element_stays_there(d, causal):
    """m = 300 is not a multiple of the 128-key tile, so element 0's last K/V
    tile covers 84 rows past its end.  Element 1's V rows there hold inf and
    NaN; their keys are masked for element 0 (weight exactly 0), and 0 * inf
    would be NaN ("S12 FlashAttention", 实现, the -inf/NaN note), so element 0
    must still match the oracle on every output."""
    case = I.dense_case(33, 2, 2, 300, 300, d, causal=causal, name="poisoned next element")
    v = case.v.data.copy()
    v[1, :84] = _BF16_NAN
    v[1, :84:3] = _BF16_INF
    vt = I.Tensor("bf16", v, I.bf16_bits_to_f32(v))
    o, lse = fb.forward(dev(case.q), dev(case.k), dev(vt), case.scale, causal)
    o_ref, lse_ref = oracle.attention(case.q.values[:1], case.k.values[:1], case.v.values[:1],
                                      case.scale, causal)
    assert_close(host(o)[:1], o_ref, BF16_MAX_ABS, BF16_MEAN_ABS, what="element 0")
    assert_lse_close(host(lse)[:1], lse_ref, what="element 0")
    assert fb.fa_get_device_status() == 0


@pytest.mark.parametrize("d", [64, 128])
def test_varlen_nonfinite_v_of_next_sequence_stays_there(d):
    """Packed sequences of 300, 200 and 77 tokens: the last K/V tile of
    sequence 0 covers the first rows of sequence 1, and sequence 1's of
    sequence 2.  Sequence 1's V rows are all inf or NaN; sequences 0 and 2
    must match the oracle on every output."""
    lens = [300, 200, 77]
    case = I.varlen_case(34, lens, H=4, d=d, Hkv=2)
    a, b = int(case.cu_seqlens[1]), int(case.cu_seqlens[2])
    vp = _poison_rows(case.v, range(a, b))
    cu = dev_i32(case.cu_seqlens)
    o, lse = fb.forward_varlen(dev(case.q), dev(case.k), dev(vp), cu, cu, max(lens), max(lens),
                               case.scale, True)
    o_ref, lse_ref = oracle.varlen(case.q.values, case.k.values, case.v.values, case.cu_seqlens,
                                   case.cu_seqlens, case.scale, True)
    oh, lh = host(o), host(lse)
    for s in (0, 2):
        lo, hi = int(case.cu_seqlens[s]), int(case.cu_seqlens[s + 1])
        assert_close(oh[lo:hi], o_ref[lo:hi], BF16_MAX_ABS, BF16_MEAN_ABS, what=f"sequence {s}")
        assert_lse_close(lh[:, lo:hi], lse_ref[:, lo:hi], what=f"sequence {s}")
    assert fb.fa_get_device_status() == 0
