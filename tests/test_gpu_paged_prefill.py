"""GPU parity of the paged (chunked) prefill, fa_paged_prefill.

Against the float64 oracle on the same bf16 inputs: O max-abs 2e-2, mean-abs
2e-3, LSE 1e-3.  The page pool's unused pages and the slots past each
sequence's end hold NaN.  Block-table indexing is checked bit-exactly against
the packed varlen path on the same keys laid out contiguously.
"""
import numpy as np
import pytest
import torch

import oracle
from tiled_online_softmax_sm_gb300 import binding as fb
from tiled_online_softmax_sm_gb300 import inputs as I

from _helpers import BF16_MAX_ABS, BF16_MEAN_ABS, assert_close, assert_lse_close, dev, dev_i32, host

pytestmark = pytest.mark.gpu


def _case(seed, lens, q_lens, H, Hkv, d, max_blocks=None):
    kv = I.decode_case(seed, num_seqs=len(lens), H=H, Hkv=Hkv, d=d, lens=lens,
                       max_blocks=max_blocks)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = I.Tensor.from_f32(I.normal_f32(I.rng(seed, 51), (int(cu[-1]), H, d)), "bf16")
    return kv, q, cu


def _gpu(kv, q, cu, causal, table=None):
    bt = kv.block_table if table is None else table
    return fb.paged_prefill(dev(q), dev(kv.k_cache), dev(kv.v_cache), dev_i32(bt),
                            dev_i32(kv.seq_lens), dev_i32(cu), int(np.diff(cu).max()), kv.scale,
                            causal)


def _ref(kv, q, cu, causal):
    return oracle.paged_prefill(q.values, cu, kv.k_cache.values, kv.v_cache.values,
                                kv.block_table, kv.seq_lens, kv.scale, causal)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_paged_prefill_small(d, causal):
    # context lengths: partial pages, exact pages, a tile boundary, short and long
    lens = [1, 16, 17, 130, 300, 513, 64]
    q_lens = [1, 5, 17, 128, 40, 300, 100]   # the last has more queries than keys
    kv, q, cu = _case(61, lens, q_lens, H=8, Hkv=2, d=d)
    o, lse = _gpu(kv, q, cu, causal)
    o_ref, lse_ref = _ref(kv, q, cu, causal)
    assert_close(host(o), o_ref, BF16_MAX_ABS, BF16_MEAN_ABS, what=f"paged prefill d={d}")
    assert_lse_close(host(lse), lse_ref, what=f"paged prefill d={d}")
    assert fb.fa_get_device_status() == 0


def test_paged_prefill_bit_exact_vs_contiguous_varlen():
    """The same keys, laid out contiguously and read by the packed varlen path,
    give identical bits: the block table only changes where a page comes from."""
    lens = [40, 257, 1000, 129]
    q_lens = [40, 64, 300, 1]
    kv, q, cu = _case(62, lens, q_lens, H=8, Hkv=4, d=128)
    o1, l1 = _gpu(kv, q, cu, True)
    ks, vs = [], []
    for s, L in enumerate(kv.seq_lens):
        ids = kv.block_table[s, :(int(L) + 15) // 16]
        ks.append(kv.k_cache.data[ids].transpose(0, 2, 1, 3).reshape(-1, kv.Hkv, kv.d)[:L])
        vs.append(kv.v_cache.data[ids].transpose(0, 2, 1, 3).reshape(-1, kv.Hkv, kv.dv)[:L])
    kc = I.Tensor("bf16", np.ascontiguousarray(np.concatenate(ks)), None)
    vc = I.Tensor("bf16", np.ascontiguousarray(np.concatenate(vs)), None)
    cu_k = np.concatenate([[0], np.cumsum(kv.seq_lens)]).astype(np.int32)
    o2, l2 = fb.forward_varlen(dev(q), dev(kc), dev(vc), dev_i32(cu), dev_i32(cu_k),
                               int(np.diff(cu).max()), int(kv.seq_lens.max()), kv.scale, True)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


def test_paged_prefill_chunks_on_the_decode_pool():
    """Chunks of 512 new tokens for 16 sequences of the decode workload's pool
    (context lengths uniform on [512, 8192], 32 heads over 8 kv heads)."""
    lens = I.uniform_lengths(63, 16, 512, 8192)
    q_lens = np.minimum(lens, 512)
    kv, q, cu = _case(63, lens, q_lens, H=32, Hkv=8, d=128, max_blocks=512)
    o, lse = _gpu(kv, q, cu, True)
    oh, lh = host(o), host(lse)
    # every sequence, rows at the chunk's start, end and a sweep, all heads
    keep = np.zeros(int(cu[-1]), bool)
    for s in range(len(lens)):
        a, b = cu[s], cu[s + 1]
        keep[[a, a + 1, b - 2, b - 1]] = True
        keep[a:b:37] = True
    o_ref, lse_ref = _ref(kv, q, cu, True)
    assert_close(oh[keep], o_ref[keep], BF16_MAX_ABS, BF16_MEAN_ABS, what="paged chunks")
    assert_lse_close(lh[:, keep], lse_ref[:, keep], what="paged chunks")
    assert fb.fa_get_device_status() == 0


def test_paged_prefill_bad_block_id_sets_status():
    kv, q, cu = _case(64, [40, 40], [8, 8], H=4, Hkv=2, d=64, max_blocks=4)
    table = kv.block_table.copy()
    table[0, 1] = kv.num_pages + 3
    o, lse = _gpu(kv, q, cu, True, table=table)
    assert fb.fa_get_device_status() == fb.FA_ERR_BAD_BLOCK_TABLE
    o_ref, _ = _ref(kv, q, cu, True)
    assert_close(host(o)[8:], o_ref[8:], BF16_MAX_ABS, BF16_MEAN_ABS)   # sequence 1 untouched
