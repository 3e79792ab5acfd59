"""The seeded input generators (CPU).

Both the CUDA path and the oracle read the arrays these generators make, so
parity cannot see a mistake in them; these checks pin them to something
else: torch's own bf16 conversion (round to nearest, ties to even), and the
layout and poisoning rules stated for the workloads.
"""
import numpy as np
import torch

from tiled_online_softmax_sm_gb300 import inputs as I


def _torch_bf16_bits(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def test_bf16_rounding_matches_torch_including_ties():
    g = I.rng(1, 2, 3)
    x = np.concatenate([
        I.normal_f32(g, (4096,)) * np.float32(1e3),
        I.normal_f32(g, (1024,)) * np.float32(1e-39),           # subnormals
        np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, -3.3895314e38], np.float32),
    ]).astype(np.float32)
    # exact ties: the 16 dropped bits are 0x8000, with an even and an odd kept part
    hi = (g.integers(0x0080, 0x7F00, size=2048).astype(np.uint32) << np.uint32(16))
    ties = (hi | np.uint32(0x8000)).view(np.float32)
    odd = ((hi | np.uint32(0x10000)) | np.uint32(0x8000)).view(np.float32)
    x = np.concatenate([x, ties, odd, -ties])
    assert np.array_equal(I.f32_to_bf16_bits(x), _torch_bf16_bits(x))


def test_bf16_nan_stays_nan_and_widening_is_exact():
    bits = I.f32_to_bf16_bits(np.array([np.nan, -np.nan], np.float32))
    assert np.isnan(I.bf16_bits_to_f32(bits)).all()
    every = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    finite = every[np.isfinite(I.bf16_bits_to_f32(every))]
    wide = I.bf16_bits_to_f32(finite)
    assert np.array_equal(wide, torch.from_numpy(finite.view(np.int16)).view(torch.bfloat16)
                          .float().numpy())
    assert np.array_equal(I.f32_to_bf16_bits(wide), finite)   # widening loses nothing


def test_generators_are_reproducible_and_seeded():
    a = I.dense_case(7, 1, 2, 33, 40, 64)
    b = I.dense_case(7, 1, 2, 33, 40, 64)
    c = I.dense_case(8, 1, 2, 33, 40, 64)
    assert np.array_equal(a.q.data, b.q.data) and np.array_equal(a.v.data, b.v.data)
    assert not np.array_equal(a.q.data, c.q.data)
    assert np.array_equal(a.q.values, I.bf16_bits_to_f32(a.q.data))


def test_decode_pool_layout_and_poison():
    lens = [0, 1, 15, 16, 17, 40, 100]
    c = I.decode_case(3, num_seqs=len(lens), H=8, Hkv=2, d=128, lens=lens, max_blocks=8)
    pages = [(L + 15) // 16 for L in lens]
    used = sum(pages)
    assert c.num_pages == used + int(np.ceil(0.10 * used))
    ids = []
    for s, (L, p) in enumerate(zip(lens, pages)):
        row = c.block_table[s]
        assert (row[p:] == -1).all()
        assert ((row[:p] >= 0) & (row[:p] < c.num_pages)).all()
        ids.extend(row[:p].tolist())
    assert len(ids) == len(set(ids)) == used            # no page is shared
    kv = I.bf16_bits_to_f32(c.k_cache.data), I.bf16_bits_to_f32(c.v_cache.data)
    unused = sorted(set(range(c.num_pages)) - set(ids))
    for cache in kv:
        assert np.isnan(cache[unused]).all()
        for s, (L, p) in enumerate(zip(lens, pages)):
            for j in range(p):
                page = cache[c.block_table[s, j]]
                valid = min(16, L - 16 * j)
                assert np.isfinite(page[:, :valid]).all()
                assert np.isnan(page[:, valid:]).all()     # tail slots of the last page
    assert c.kv_bytes == sum(lens) * 2 * (128 + 128) * 2


def test_varlen_hot_rows_are_the_stated_tenth_times_twenty():
    lens = [5, 300, 77]
    hot = I.varlen_case(9, lens, H=2, d=64)
    cold = I.varlen_case(9, lens, H=2, d=64, hot_frac=0.0)
    T = sum(lens)
    assert len(hot.hot_rows_q) == len(hot.hot_rows_k) == round(0.10 * T)
    assert not np.array_equal(hot.hot_rows_q, hot.hot_rows_k)   # drawn independently
    raw_q = I.normal_f32(I.rng(9, 5, 0), (T, 2, 64))
    want = raw_q.copy()
    want[hot.hot_rows_q] *= np.float32(20.0)
    assert np.array_equal(hot.q.data, I.f32_to_bf16_bits(want))
    rest = np.setdiff1d(np.arange(T), hot.hot_rows_k)
    assert np.array_equal(hot.k.data[rest], cold.k.data[rest])
    assert np.array_equal(hot.v.data, cold.v.data)               # V is not scaled
    assert list(hot.cu_seqlens) == [0, 5, 305, 382]
