"""Pins of the float64 oracle against facts that do not come from the oracle.

Each test names the passage (page title, section) or the mathematical fact it
pins.  A plausible slip anywhere in the oracle (dropped scale, wrong causal
direction or index, wrong grouped-head mapping, transposed operand, missing
max subtraction, wrong LSE) fails at least one of them; ``test_pins_discriminate``
checks that for a set of such slips.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from tiled_online_softmax_sm_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(seed, *shape, scale=1.0):
    return (I.normal_f32(I.rng(seed, 99, len(shape)), shape) * np.float32(scale)).astype(np.float32)


def _sdpa_f64(q, k, v, scale, causal):
    """Library routine (torch math backend, float64) on BSHD inputs; grouped
    heads are expanded by repeating each kv head over its query group."""
    B, n, H, d = q.shape
    Hkv = k.shape[2]
    g = H // Hkv
    qt = torch.from_numpy(q.astype(np.float64)).permute(0, 2, 1, 3)
    kt = torch.from_numpy(k.astype(np.float64)).permute(0, 2, 1, 3).repeat_interleave(g, dim=1)
    vt = torch.from_numpy(v.astype(np.float64)).permute(0, 2, 1, 3).repeat_interleave(g, dim=1)
    n_, m_ = qt.shape[-2], kt.shape[-2]
    # causal, bottom-right aligned: key j visible to query i iff j <= i + (m - n)
    mask = torch.ones(n_, m_, dtype=torch.bool).tril(diagonal=m_ - n_) if causal else None
    if mask is not None and not mask.any(dim=-1).all():
        # rows that see no key: the library routine returns NaN there, the
        # reading is O = 0, LSE = -inf; evaluate the others only
        o = torch.zeros(qt.shape[:-1] + (vt.shape[-1],), dtype=torch.float64)
        keep = mask.any(dim=-1)
        o[..., keep, :] = torch.nn.functional.scaled_dot_product_attention(
            qt[..., keep, :], kt, vt, attn_mask=mask[keep], scale=scale)
    else:
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    s = torch.einsum("bhid,bhjd->bhij", qt, kt) * scale
    if causal:
        s = s.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    return o.permute(0, 2, 1, 3).numpy(), lse.numpy()


# ----------------------------------------------------------------------------
# Closed forms
# ----------------------------------------------------------------------------
def test_q_zero_noncausal_is_mean_of_v():
    """Q = 0 makes every score 0: O is the plain mean of the V rows of the
    query head's kv head, and LSE = ln m ("手搓 Attention" §1: weights from a
    softmax of equal scores are uniform)."""
    B, H, Hkv, n, m, d, dv = 2, 4, 2, 5, 7, 8, 6
    q = np.zeros((B, n, H, d), np.float32)
    k = _rand(1, B, m, Hkv, d)
    v = _rand(2, B, m, Hkv, dv)
    o, lse = oracle.attention(q, k, v, 0.3, causal=False)
    for b in range(B):
        for h in range(H):
            want = v[b, :, h // (H // Hkv), :].astype(np.float64).mean(axis=0)
            for i in range(n):
                np.testing.assert_allclose(o[b, i, h], want, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, math.log(m), rtol=0, atol=1e-14)


def test_q_zero_causal_is_prefix_mean():
    """Causal (key j visible to query i iff j <= i): with Q = 0 row i is the
    mean of V[0..i] and LSE = ln(i+1)."""
    B, H, n, d, dv = 1, 2, 9, 4, 5
    q = np.zeros((B, n, H, d), np.float32)
    k = _rand(3, B, n, H, d)
    v = _rand(4, B, n, H, dv)
    o, lse = oracle.attention(q, k, v, 1.0, causal=True)
    for h in range(H):
        for i in range(n):
            want = v[0, : i + 1, h].astype(np.float64).mean(axis=0)
            np.testing.assert_allclose(o[0, i, h], want, rtol=0, atol=1e-14)
            assert abs(lse[0, h, i] - math.log(i + 1)) < 1e-14


@pytest.mark.parametrize("n,m", [(4, 9), (9, 4), (1, 7)])
def test_q_zero_causal_unequal_lengths_bottom_right(n, m):
    """Causal with n != m, read bottom-right: the n queries are the last n of
    the m key positions, so row i sees keys 0..i+(m-n); with Q = 0 it is the
    mean of those V rows and LSE = ln(count).  Rows that see none (n > m) get
    O = 0 and LSE = -inf."""
    H, d, dv = 2, 4, 3
    q = np.zeros((1, n, H, d), np.float32)
    k = _rand(41, 1, m, H, d)
    v = _rand(42, 1, m, H, dv)
    o, lse = oracle.attention(q, k, v, 1.0, causal=True)
    for h in range(H):
        for i in range(n):
            cnt = min(m, max(0, i + 1 + m - n))
            if cnt == 0:
                assert np.all(o[0, i, h] == 0) and np.isneginf(lse[0, h, i])
                continue
            want = v[0, :cnt, h].astype(np.float64).mean(axis=0)
            np.testing.assert_allclose(o[0, i, h], want, rtol=0, atol=1e-14)
            assert abs(lse[0, h, i] - math.log(cnt)) < 1e-14


def test_one_dominant_score_selects_its_value_row():
    """K[j*] = c*Q[i] with c large makes score j* exceed every other by
    thousands: the softmax is one-hot and O[i] = V[j*]."""
    B, H, n, m, d = 1, 1, 3, 11, 16
    q = _rand(5, B, n, H, d)
    k = _rand(6, B, m, H, d)
    v = _rand(7, B, m, H, d)
    for i, jstar in [(0, 4), (1, 10), (2, 0)]:
        k2 = k.copy()
        k2[0, jstar, 0] = 1000.0 * q[0, i, 0]
        o, lse = oracle.attention(q, k2, v, 0.25, causal=False)
        np.testing.assert_allclose(o[0, i, 0], v[0, jstar, 0].astype(np.float64), rtol=0, atol=1e-12)
        s_star = 0.25 * float(np.dot(q[0, i, 0].astype(np.float64), k2[0, jstar, 0].astype(np.float64)))
        assert abs(lse[0, 0, i] - s_star) < 1e-9


def test_weights_sum_to_one_and_respect_mask():
    """Instrumented mode: the softmax weights of every row sum to 1, are
    positive on visible keys and zero on masked ones."""
    B, H, n, m, d = 2, 3, 6, 6, 8
    q = _rand(8, B, n, H, d, scale=3.0)
    k = _rand(9, B, m, H, d, scale=3.0)
    v = _rand(10, B, m, H, d)
    rows = np.array([(b, h, i) for b in range(B) for h in range(H) for i in range(n)], np.int32)
    for causal in (False, True):
        o, lse, w = oracle.attention_rows(q, k, v, 0.35, causal, rows, with_weights=True)
        assert np.all(np.abs(w.sum(axis=1) - 1.0) < 1e-14)
        for r, (b, h, i) in enumerate(rows):
            vis = np.arange(m) <= i if causal else np.ones(m, bool)
            assert np.all(w[r, vis] > 0) and np.all(w[r, ~vis] == 0)
            # O is the weighted row sum of V with those weights
            np.testing.assert_allclose(o[r], w[r] @ v[b, :, h].astype(np.float64), rtol=0, atol=1e-13)


def _row_by_definition(q, k, v, scale, causal, b, h, i, kv_b=None, kv_h=None, q_i=None):
    """One output row from "手搓 Attention" §2 version 0 with §4's max
    subtraction, in numpy float64; kv_b, kv_h and q_i override the batch
    element and kv head whose K/V rows are read and the query row, to play
    the row-offset slips the selected-rows test must catch."""
    n, m = q.shape[1], k.shape[1]
    group = q.shape[2] // k.shape[2]
    kb = b if kv_b is None else kv_b
    hk = h // group if kv_h is None else kv_h
    qi = i if q_i is None else q_i
    vis = min(m, max(0, i + 1 + (m - n))) if causal else m
    if vis == 0:
        return np.zeros(v.shape[-1])
    s = scale * (k[kb, :vis, hk].astype(np.float64) @ q[b, qi, h].astype(np.float64))
    w = np.exp(s - s.max())
    return (w / w.sum()) @ v[kb, :vis, hk].astype(np.float64)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n, m", [(13, 13), (9, 21), (21, 9)])
def test_selected_rows_equal_the_full_definition(causal, n, m):
    """The selected-rows oracle (the checker of the full-size GPU tests and
    of the CPU baseline) gives, bit for bit, row (b, h, i) of the every-row
    oracle, which the closed forms above and the library SDPA pin; every
    (b, h, i) of a batch with B > 1, grouped heads and n != m is asked for,
    in shuffled order and with repeats ("手搓 Attention" §2 version 0: the
    definition every other version is checked against).  Row-offset slips
    (the wrong batch element, kv head or query row), written test-side, each
    fail the same comparison."""
    B, H, Hkv, d, dv = 3, 6, 2, 16, 8
    q = _rand(70, B, n, H, d, scale=2)
    k = _rand(71, B, m, Hkv, d, scale=2)
    v = _rand(72, B, m, Hkv, dv)
    scale = 0.37
    o, lse = oracle.attention(q, k, v, scale, causal)
    allrows = np.array([(b, h, i) for b in range(B) for h in range(H) for i in range(n)], np.int32)
    g = I.rng(73, n, m)
    rows = np.concatenate([allrows[g.permutation(len(allrows))],
                           allrows[g.integers(0, len(allrows), size=17)]])
    o_r, lse_r = oracle.attention_rows(q, k, v, scale, causal, rows)
    assert np.array_equal(o_r, o[rows[:, 0], rows[:, 2], rows[:, 1]])
    assert np.array_equal(lse_r, lse[rows[:, 0], rows[:, 1], rows[:, 2]])
    # the definition written out agrees with both
    for b, h, i in allrows[:: 7]:
        want = _row_by_definition(q, k, v, scale, causal, b, h, i)
        np.testing.assert_allclose(o[b, i, h], want, rtol=0, atol=1e-12)
    # slips: each reads the wrong rows somewhere and misses by far more than rounding
    for b, h, i in [(1, 5, n - 1), (2, 2, n - 3), (0, 3, n - 2)]:
        wrong_b = _row_by_definition(q, k, v, scale, causal, b, h, i, kv_b=(b + 1) % B)
        wrong_h = _row_by_definition(q, k, v, scale, causal, b, h, i, kv_h=(h // 3 + 1) % Hkv)
        wrong_i = _row_by_definition(q, k, v, scale, causal, b, h, i, q_i=(i + 1) % n)
        for bad in (wrong_b, wrong_h, wrong_i):
            assert np.abs(bad - o[b, i, h]).max() > 1e-3


# ----------------------------------------------------------------------------
# Invariants
# ----------------------------------------------------------------------------
def test_joint_kv_permutation_invariance():
    """Non-causal attention is a set function of the (K, V) row pairs."""
    B, H, Hkv, n, m, d, dv = 2, 4, 1, 7, 13, 8, 12
    q, k, v = _rand(11, B, n, H, d, scale=2), _rand(12, B, m, Hkv, d, scale=2), _rand(13, B, m, Hkv, dv)
    o1, l1 = oracle.attention(q, k, v, 0.4, False)
    perm = I.rng(14).permutation(m)
    o2, l2 = oracle.attention(q, k[:, perm], v[:, perm], 0.4, False)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


def test_key_shift_invariance():
    """Adding u to every K row adds scale*q.u to every score of a row: the
    softmax is unchanged and LSE moves by exactly that amount.  K is bf16-valued
    and u a multiple of 1/64, so K + u is exact in fp32."""
    B, H, n, m, d = 1, 2, 5, 9, 8
    q = I.round_to_bf16(_rand(15, B, n, H, d))
    k = I.round_to_bf16(_rand(16, B, m, H, d))
    v = _rand(17, B, m, H, d)
    u = (np.arange(d, dtype=np.float32) - 3.0) / np.float32(64.0)
    k2 = (k + u).astype(np.float32)
    assert np.array_equal(k2.astype(np.float64), k.astype(np.float64) + u.astype(np.float64))
    scale = 0.5
    o1, l1 = oracle.attention(q, k, v, scale, False)
    o2, l2 = oracle.attention(q, k2, v, scale, False)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    shift = scale * np.einsum("bihd,d->bhi", q.astype(np.float64), u.astype(np.float64))
    np.testing.assert_allclose(l2 - l1, shift, rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------
# Brute force against a library routine on tiny inputs
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 1, 1, 1, 1, 4, 4), (2, 4, 2, 9, 9, 8, 8),
                                   (1, 6, 3, 5, 12, 16, 8), (3, 2, 2, 16, 16, 4, 7),
                                   (1, 2, 1, 12, 5, 8, 8)])
def test_brute_force_vs_library_sdpa(shape, causal):
    B, H, Hkv, n, m, d, dv = shape
    q, k, v = _rand(20, B, n, H, d, scale=2), _rand(21, B, m, Hkv, d, scale=2), _rand(22, B, m, Hkv, dv)
    scale = 0.37
    o, lse = oracle.attention(q, k, v, scale, causal)
    o_ref, lse_ref = _sdpa_f64(q, k, v, scale, causal)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


def test_p3_worked_case_seed42():
    """"FlashAttention推理优化实战100例 01", 实现代码 and 运行与验证: seed 42,
    N=4, d=8, float64 inputs, no scale, block size 2: the block-wise
    recurrence and the standard attention agree within 1e-8."""
    with open(os.path.join(GOLDEN, "p3_seed42_n4_d8.json")) as f:
        spec = json.load(f)
    st = np.random.RandomState(spec["seed"])  # the page's legacy numpy generator
    N, d = spec["N"], spec["d"]
    Q = st.randn(N, d)
    K = st.randn(N, d)
    V = st.randn(N, d)
    # the oracle takes fp32 inputs: use the fp32-rounded copies on both sides
    Qf, Kf, Vf = (x.astype(np.float32) for x in (Q, K, V))
    o_def, _ = oracle.attention(Qf[None, :, None], Kf[None, :, None], Vf[None, :, None],
                                spec["scale"], False)
    o_rec, _ = oracle.online_recurrence(Qf, Kf, Vf, spec["scale"], False,
                                        q_block=spec["block_size"], kv_block=spec["block_size"])
    assert np.abs(o_def[0, :, 0] - o_rec).max() < spec["max_abs_diff"]
    o_lib, _ = _sdpa_f64(Qf[None, :, None], Kf[None, :, None], Vf[None, :, None], spec["scale"], False)
    assert np.abs(o_def - o_lib).max() < spec["max_abs_diff"]


# ----------------------------------------------------------------------------
# The recurrence equals the definition ("S12 FlashAttention", 动手观察: any
# tile size, including 1, gives the same answer)
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("kv_block", [1, 2, 16, 63, 64])
def test_recurrence_any_tile_equals_definition(kv_block, causal):
    n = m = 130
    q, k, v = _rand(30, n, 16, scale=3), _rand(31, m, 16, scale=3), _rand(32, m, 24)
    o_rec, l_rec = oracle.online_recurrence(q, k, v, 0.3, causal, q_block=64, kv_block=kv_block)
    o_def, l_def = oracle.attention(q[None, :, None], k[None, :, None], v[None, :, None], 0.3, causal)
    np.testing.assert_allclose(o_rec, o_def[0, :, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(l_rec, l_def[0, 0], rtol=0, atol=1e-12)


@pytest.mark.parametrize("n,m", [(40, 130), (130, 40)])
def test_recurrence_unequal_causal_equals_definition(n, m):
    q, k, v = _rand(36, n, 8, scale=2), _rand(37, m, 8, scale=2), _rand(38, m, 8)
    o_rec, l_rec = oracle.online_recurrence(q, k, v, 0.4, True, q_block=16, kv_block=32)
    o_def, l_def = oracle.attention(q[None, :, None], k[None, :, None], v[None, :, None], 0.4, True)
    np.testing.assert_allclose(o_rec, o_def[0, :, 0], rtol=0, atol=1e-12)
    assert np.array_equal(np.isneginf(l_rec), np.isneginf(l_def[0, 0]))
    fin = ~np.isneginf(l_rec)
    np.testing.assert_allclose(l_rec[fin], l_def[0, 0][fin], rtol=0, atol=1e-12)


def test_recurrence_guard_fully_masked_first_tiles():
    """"S12 FlashAttention", 实现: a first tile that is fully masked would give
    exp(-inf - -inf) = NaN.  Visiting the kv blocks last-first under a causal
    mask makes the first tiles fully masked for early rows; the guarded
    recurrence stays finite and equal to the definition."""
    n = m = 96
    q, k, v = _rand(33, n, 8), _rand(34, m, 8), _rand(35, m, 8)
    order = list(reversed(range(6)))  # kv blocks of 16, diagonal/future first
    o_rec, l_rec = oracle.online_recurrence(q, k, v, 0.5, True, q_block=16, kv_block=16,
                                            kv_order=order)
    assert np.isfinite(o_rec).all() and np.isfinite(l_rec).all()
    o_def, l_def = oracle.attention(q[None, :, None], k[None, :, None], v[None, :, None], 0.5, True)
    np.testing.assert_allclose(o_rec, o_def[0, :, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(l_rec, l_def[0, 0], rtol=0, atol=1e-12)


def test_unguarded_recurrence_reproduces_the_nan_trap():
    """Negative control for the guard above ("S12 FlashAttention", 实现 and 练习
    2): the same diagonal-first visit order with the textbook update
    m_new = max(m, tile max), alpha = exp(m - m_new), p = exp(s - m_new),
    written test-side without the guard, turns early rows into NaN."""
    n = m = 32
    q, k, v = _rand(33, n, 8), _rand(34, m, 8), _rand(35, m, 8)
    s = (q.astype(np.float64) @ k.astype(np.float64).T) * 0.5
    s[np.triu_indices(n, 1)] = -np.inf                  # causal: j <= i
    blocks = [slice(16, 32), slice(0, 16)]               # future block first
    m_run = np.full(n, -np.inf)
    l_run = np.zeros(n)
    acc = np.zeros((n, 8))
    with np.errstate(invalid="ignore"):
        for blk in blocks:
            st = s[:, blk]
            m_new = np.maximum(m_run, st.max(axis=1))
            alpha = np.exp(m_run - m_new)                # -inf - -inf = NaN for early rows
            p = np.exp(st - m_new[:, None])
            l_run = alpha * l_run + p.sum(axis=1)
            acc = alpha[:, None] * acc + p @ v[blk].astype(np.float64)
            m_run = m_new
    o_naive = acc / l_run[:, None]
    assert np.isnan(o_naive[:16]).all()                  # rows 0..15 see nothing in block 1
    o_rec, _ = oracle.online_recurrence(q, k, v, 0.5, True, q_block=16, kv_block=16, kv_order=[1, 0])
    assert np.isfinite(o_rec).all()


# ----------------------------------------------------------------------------
# Paged decode, split partials and their merge
# ----------------------------------------------------------------------------
def _dense_gather(case):
    """Test-side gather of each sequence's keys/values (numpy indexing)."""
    out = []
    for s, L in enumerate(case.seq_lens):
        P = (int(L) + case.page_size - 1) // case.page_size
        ids = case.block_table[s, :P]
        kk = case.k_cache.values[ids].transpose(0, 2, 1, 3).reshape(-1, case.Hkv, case.d)[:L]
        vv = case.v_cache.values[ids].transpose(0, 2, 1, 3).reshape(-1, case.Hkv, case.dv)[:L]
        out.append((kk, vv))
    return out


def test_paged_decode_matches_dense_library():
    case = I.decode_case(7, num_seqs=5, H=8, Hkv=2, d=16, dv=16, page_size=4,
                         lens=[1, 4, 5, 17, 30], max_blocks=9)
    o, lse = oracle.paged_decode(case.q.values, case.k_cache.values, case.v_cache.values,
                                 case.block_table, case.seq_lens, case.scale)
    assert np.isfinite(o).all() and np.isfinite(lse).all()  # poisoned slots never read
    for s, (kk, vv) in enumerate(_dense_gather(case)):
        o_ref, l_ref = _sdpa_f64(case.q.values[s][None, None], kk[None], vv[None], case.scale, False)
        np.testing.assert_allclose(o[s], o_ref[0, 0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[s], l_ref[0, :, 0], rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_paged_prefill_matches_dense_library(causal):
    """Several new tokens per sequence against the sequence's paged keys equal
    the library routine on the gathered keys with the bottom-right mask."""
    lens = [1, 4, 5, 17, 30]
    q_lens = [1, 3, 5, 7, 40]          # the last sequence has more queries than keys
    case = I.decode_case(12, num_seqs=5, H=4, Hkv=2, d=16, dv=16, page_size=4, lens=lens,
                         max_blocks=9)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = _rand(13, int(cu[-1]), 4, 16)
    o, lse = oracle.paged_prefill(q, cu, case.k_cache.values, case.v_cache.values,
                                  case.block_table, case.seq_lens, case.scale, causal)
    assert np.isfinite(o).all()   # poisoned slots never read
    for s, (kk, vv) in enumerate(_dense_gather(case)):
        a, b = cu[s], cu[s + 1]
        o_ref, l_ref = _sdpa_f64(q[None, a:b], kk[None], vv[None], case.scale, causal)
        np.testing.assert_allclose(o[a:b], o_ref[0], rtol=0, atol=1e-12)
        assert np.array_equal(np.isneginf(lse[:, a:b]), np.isneginf(l_ref[0]))
        fin = ~np.isneginf(l_ref[0])
        np.testing.assert_allclose(lse[:, a:b][fin], l_ref[0][fin], rtol=0, atol=1e-12)


def test_paged_prefill_single_token_is_decode():
    case = I.decode_case(14, num_seqs=3, H=4, Hkv=1, d=8, page_size=4, lens=[3, 9, 16],
                         max_blocks=4)
    cu = np.arange(4, dtype=np.int32)
    a = oracle.paged_prefill(case.q.values, cu, case.k_cache.values, case.v_cache.values,
                             case.block_table, case.seq_lens, case.scale, True)
    b = oracle.paged_decode(case.q.values, case.k_cache.values, case.v_cache.values,
                            case.block_table, case.seq_lens, case.scale)
    np.testing.assert_allclose(a[0], b[0], rtol=0, atol=1e-14)
    np.testing.assert_allclose(a[1].T, b[1], rtol=0, atol=1e-14)


def test_paged_decode_rejects_bad_block_ids():
    case = I.decode_case(8, num_seqs=2, H=2, Hkv=1, d=8, page_size=4, lens=[5, 3], max_blocks=2)
    bt = case.block_table.copy()
    bt[0, 1] = case.num_pages
    with pytest.raises(IndexError):
        oracle.paged_decode(case.q.values, case.k_cache.values, case.v_cache.values, bt,
                            case.seq_lens, case.scale)


@pytest.mark.parametrize("splits", [1, 2, 3, 4, 16])
def test_split_partials_merge_to_unsplit(splits):
    """"S12 FlashAttention", 它还解锁了什么 and 练习 1: keys split across workers,
    each runs the recurrence, the (m, l, o) triples merge with the same rescale;
    the merge equals the unsplit result (empty splits included at 16)."""
    case = I.decode_case(9, num_seqs=4, H=4, Hkv=2, d=16, dv=8, page_size=4,
                         lens=[2, 9, 23, 40], max_blocks=10)
    args = (case.q.values, case.k_cache.values, case.v_cache.values, case.block_table, case.seq_lens)
    pm, pl, po = oracle.decode_partials(*args, splits, case.scale)
    o, lse = oracle.split_combine(pm, pl, po)
    o_ref, lse_ref = oracle.paged_decode(*args, case.scale)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)
    if splits == 16:  # sequence 0 has one page: 15 empty splits
        assert np.sum(np.isneginf(pm[0, 0])) == 15 and np.all(pl[0, 0][np.isneginf(pm[0, 0])] == 0)


def test_split_combine_all_empty_is_zero_and_neg_inf():
    pm = np.full((1, 2, 3), -np.inf)
    pl = np.zeros((1, 2, 3))
    po = np.zeros((1, 2, 3, 4))
    o, lse = oracle.split_combine(pm, pl, po)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_varlen_matches_per_sequence_library():
    lens = [1, 5, 17, 3]
    case = I.varlen_case(11, lens, H=4, d=8, Hkv=2, hot_frac=0.25, hot=5.0)
    for causal in (False, True):
        o, lse = oracle.varlen(case.q.values, case.k.values, case.v.values, case.cu_seqlens,
                               case.cu_seqlens, case.scale, causal)
        for s in range(len(lens)):
            a, b = case.cu_seqlens[s], case.cu_seqlens[s + 1]
            o_ref, l_ref = _sdpa_f64(case.q.values[None, a:b], case.k.values[None, a:b],
                                     case.v.values[None, a:b], case.scale, causal)
            np.testing.assert_allclose(o[a:b], o_ref[0], rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[:, a:b], l_ref[0], rtol=0, atol=1e-10)


def test_empty_and_degenerate_rows():
    """m = 0: no key is visible, O = 0 and LSE = -inf (reading for l = 0)."""
    q = _rand(40, 1, 3, 1, 4)
    k = np.zeros((1, 0, 1, 4), np.float32)
    v = np.zeros((1, 0, 1, 4), np.float32)
    o, lse = oracle.attention(q, k, v, 1.0, False)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


# ----------------------------------------------------------------------------
# Hot inputs and the negative controls of "手搓 Attention"
# ----------------------------------------------------------------------------
def test_hot_inputs_stay_finite_and_naive_softmax_overflows():
    """§4: with Q, K x10 the scores reach the hundreds; a softmax without the
    max subtraction overflows in fp32 while the oracle stays finite."""
    c = I.c1_fp32(hot=True)
    o, lse = oracle.attention(c.q.values, c.k.values, c.v.values, c.scale, False)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    s = (c.q.values[0, :, 0] @ c.k.values[0, :, 0].T) * np.float32(c.scale)
    assert s.max() > 150.0
    with np.errstate(over="ignore", invalid="ignore"):
        e = np.exp(s.astype(np.float32))
        naive = e / e.sum(axis=-1, keepdims=True)
    assert (~np.isfinite(naive)).any()


def test_fp16_exp_overflow_threshold_from_page():
    """§4 reports that fp16 exp overflows once the score exceeds 11.1."""
    with open(os.path.join(GOLDEN, "p1_fp16_exp_overflow.json")) as f:
        spec = json.load(f)
    thr = spec["score_threshold"]
    with np.errstate(over="ignore"):
        assert np.isinf(np.exp(np.float16(thr)))
        assert np.isfinite(np.exp(np.float16(thr - 0.1)))


def test_per_block_softmax_is_wrong():
    """§6 version 3 normalises each block on its own and sums them; its weights
    add up to the number of blocks.  It must differ from the oracle by O(1)."""
    n = m = 64
    q, k, v = _rand(50, n, 16), _rand(51, m, 16), _rand(52, m, 16)
    o_def, _ = oracle.attention(q[None, :, None], k[None, :, None], v[None, :, None], 0.25, False)
    bad = np.zeros((n, 16))
    for j0 in range(0, m, 16):
        s = 0.25 * q.astype(np.float64) @ k[j0:j0 + 16].astype(np.float64).T
        w = np.exp(s - s.max(axis=1, keepdims=True))
        bad += (w / w.sum(axis=1, keepdims=True)) @ v[j0:j0 + 16].astype(np.float64)
    assert np.abs(bad - o_def[0, :, 0]).max() > 0.5


def test_pins_discriminate_plausible_slips():
    """Plausible slips, written test-side, each fail the comparison the pins use."""
    B, H, Hkv, n, m, d = 1, 4, 2, 6, 6, 8
    q, k, v = _rand(60, B, n, H, d, scale=2), _rand(61, B, m, Hkv, d, scale=2), _rand(62, B, m, Hkv, d)
    scale = 0.4
    o_ref, lse_ref = _sdpa_f64(q, k, v, scale, True)
    # dropped scale
    o_bad, _ = _sdpa_f64(q, k, v, 1.0, True)
    assert np.abs(o_bad - o_ref).max() > 1e-3
    # grouped-head mapping h % Hkv instead of h // group
    k_mod = k[:, :, [h % Hkv for h in range(H)]]
    v_mod = v[:, :, [h % Hkv for h in range(H)]]
    o_bad, _ = _sdpa_f64(q, k_mod, v_mod, scale, True)
    assert np.abs(o_bad - o_ref).max() > 1e-3
    # causal off by one (j < i visible, diagonal dropped): Q = 0 closed form fails
    v0 = v[0, :, 0].astype(np.float64)
    prefix_excl = np.array([v0[:i].mean(axis=0) if i else np.zeros(d) for i in range(n)])
    prefix_incl = np.array([v0[: i + 1].mean(axis=0) for i in range(n)])
    assert np.abs(prefix_excl - prefix_incl).max() > 1e-3
    # transposed operand (K used as V)
    o_bad, _ = _sdpa_f64(q, k, k, scale, True)
    assert np.abs(o_bad - o_ref).max() > 1e-3
    # the oracle itself matches the library on this case
    o, lse = oracle.attention(q, k, v, scale, True)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


def test_results_do_not_depend_on_the_thread_count():
    """The oracle's rows are each one thread's loop, so one thread and all of
    them give the same bits (the bench times it both ways)."""
    c = I.dense_case(12, 2, 3, 70, 90, 64, Hkv=1, causal=True)
    o_all, lse_all = oracle.attention(c.q.values, c.k.values, c.v.values, c.scale, True)
    prev = oracle.set_num_threads(1)
    try:
        assert oracle.num_threads() == 1
        o_one, lse_one = oracle.attention(c.q.values, c.k.values, c.v.values, c.scale, True)
    finally:
        oracle.set_num_threads(prev)
    assert oracle.num_threads() == prev
    assert np.array_equal(o_all, o_one) and np.array_equal(lse_all, lse_one)
