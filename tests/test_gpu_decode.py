"""GPU parity of the paged grouped-head split-KV decode and of the split merge.

Against the float64 oracle: O max-abs 2e-2 and mean-abs 2e-3, LSE 1e-3.
Block-table indexing is checked bit-exactly: the same kernel on the same KV
laid out contiguously behind an identity table must give identical bits, and
the decode's page walk gathered out to dense buffers (fa_paged_gather) must
equal a host gather bit for bit.
Unused pool pages and the tail slots of each last page hold NaN, so a stray
read shows up as NaN in O.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from tiled_online_softmax_sm_gb300 import binding as fb
from tiled_online_softmax_sm_gb300 import inputs as I

from _helpers import BF16_MAX_ABS, BF16_MEAN_ABS, assert_close, assert_lse_close, dev, dev_i32, host

pytestmark = pytest.mark.gpu


def _gpu_decode(case, splits, workspace=None):
    return fb.paged_decode(dev(case.q), dev(case.k_cache), dev(case.v_cache),
                           dev_i32(case.block_table), dev_i32(case.seq_lens), splits, case.scale,
                           workspace=workspace)


def _oracle(case):
    return oracle.paged_decode(case.q.values, case.k_cache.values, case.v_cache.values,
                               case.block_table, case.seq_lens, case.scale)


@pytest.mark.parametrize("splits", [1, 3, 4, 8, 16])
def test_decode_small_ragged(splits):
    # lengths: empty, 1 token, partial pages, exact pages, many pages
    lens = [0, 1, 15, 16, 17, 100, 257, 640]
    case = I.decode_case(5, num_seqs=len(lens), H=32, Hkv=8, d=128, lens=lens, max_blocks=48)
    o, lse = _gpu_decode(case, splits)
    o_ref, lse_ref = _oracle(case)
    assert_close(host(o), o_ref, BF16_MAX_ABS, BF16_MEAN_ABS, what=f"decode X={splits}")
    assert_lse_close(host(lse), lse_ref, what=f"decode lse X={splits}")
    assert fb.fa_get_device_status() == 0


@pytest.mark.parametrize("group", [1, 2, 4, 8, 16])
def test_decode_group_sizes(group):
    Hkv = 2
    case = I.decode_case(6, num_seqs=3, H=Hkv * group, Hkv=Hkv, d=128, lens=[33, 200, 511],
                         max_blocks=40)
    o, lse = _gpu_decode(case, 4)
    o_ref, lse_ref = _oracle(case)
    assert_close(host(o), o_ref, BF16_MAX_ABS, BF16_MEAN_ABS, what=f"group {group}")
    assert_lse_close(host(lse), lse_ref)


def test_decode_partials_match_oracle_partials():
    case = I.decode_case(8, num_seqs=4, H=8, Hkv=2, d=128, lens=[5, 64, 300, 129], max_blocks=24)
    X = 5
    need = fb.fa_paged_decode_workspace_size(4, 8, 128, X)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    _gpu_decode(case, X, workspace=ws)
    torch.cuda.synchronize()
    pm, pl, po = (host(t) for t in fb.decode_workspace_views(ws, 4, 8, 128, X))
    rm, rl, ro = oracle.decode_partials(case.q.values, case.k_cache.values, case.v_cache.values,
                                        case.block_table, case.seq_lens, X, case.scale)
    assert np.array_equal(np.isneginf(pm), np.isneginf(rm))
    fin = ~np.isneginf(rm)
    assert np.abs(pm[fin] - rm[fin]).max() < 1e-3
    # l and o are relative to each side's own m: compare after normalising
    assert np.abs(pl[fin] * np.exp(pm[fin] - rm[fin]) - rl[fin]).max() / rl[fin].max() < 2e-2
    on = po[fin] / pl[fin][:, None]
    rn = ro[fin] / rl[fin][:, None]
    assert np.abs(on - rn).max() < BF16_MAX_ABS
    assert np.all(pl[~fin] == 0) and np.all(po[~fin] == 0)


def test_block_table_bit_exact_vs_contiguous_layout():
    """Same kernel, same arithmetic: a random permutation table and an identity
    table over the same KV re-laid-out contiguously give identical bits."""
    case = I.decode_case(9, num_seqs=6, H=32, Hkv=8, d=128, lens=[3, 40, 77, 512, 1000, 1500],
                         max_blocks=100)
    o1, l1 = _gpu_decode(case, 4)
    # re-lay-out: sequence s's pages become consecutive physical pages
    used = [case.block_table[s, :(int(L) + 15) // 16] for s, L in enumerate(case.seq_lens)]
    order = np.concatenate(used)
    P = len(order)
    table = np.full_like(case.block_table, -1)
    off = 0
    for s, ids in enumerate(used):
        table[s, :len(ids)] = np.arange(off, off + len(ids))
        off += len(ids)
    kc = I.Tensor("bf16", np.ascontiguousarray(case.k_cache.data[order]), None)
    vc = I.Tensor("bf16", np.ascontiguousarray(case.v_cache.data[order]), None)
    o2, l2 = fb.paged_decode(dev(case.q), dev(kc), dev(vc), dev_i32(table), dev_i32(case.seq_lens),
                             4, case.scale)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))
    assert P > 0


def test_bad_block_id_sets_status_without_fault():
    case = I.decode_case(10, num_seqs=2, H=8, Hkv=2, d=128, lens=[40, 40], max_blocks=4)
    table = case.block_table.copy()
    table[1, 1] = case.num_pages + 7      # out of range
    o, lse = fb.paged_decode(dev(case.q), dev(case.k_cache), dev(case.v_cache), dev_i32(table),
                             dev_i32(case.seq_lens), 2, case.scale)
    assert fb.fa_get_device_status() == fb.FA_ERR_BAD_BLOCK_TABLE
    assert fb.fa_get_device_status() == 0  # read clears it
    # the untouched sequence is still right
    o_ref, _ = _oracle(case)
    assert_close(host(o)[0], o_ref[0], BF16_MAX_ABS, BF16_MEAN_ABS)


def test_out_of_range_seq_len_sets_status_and_reads_nothing():
    """A length past the block table's row (or below zero) is caught on the
    device: the sequence counts as empty (O = 0, LSE = -inf), the status word
    says FA_ERR_INVALID_ARG, and the other sequences are unaffected."""
    case = I.decode_case(11, num_seqs=3, H=8, Hkv=2, d=128, lens=[40, 40, 40], max_blocks=4)
    lens = case.seq_lens.copy()
    lens[1] = 4 * 16 + 1
    lens[2] = -5
    o, lse = fb.paged_decode(dev(case.q), dev(case.k_cache), dev(case.v_cache),
                             dev_i32(case.block_table), dev_i32(lens), 2, case.scale)
    assert fb.fa_get_device_status() == fb.FA_ERR_INVALID_ARG
    oh, lh = host(o), host(lse)
    assert (oh[1:] == 0).all() and np.isneginf(lh[1:]).all()
    o_ref, lse_ref = _oracle(case)
    assert_close(oh[0], o_ref[0], BF16_MAX_ABS, BF16_MEAN_ABS)
    assert_lse_close(lh[0], lse_ref[0])


# ---- the decode's page walk, gathered out: bit-exact against a host gather

_SENTINEL = 0x1234   # a finite bf16 pattern no gathered row is compared against


def _gpu_gather(case, splits):
    S, maxb = case.block_table.shape
    Hkv = case.k_cache.data.shape[1]
    ko = torch.full((S, maxb * 16, Hkv, 128), _SENTINEL, dtype=torch.int16, device="cuda")
    vo = torch.full_like(ko, _SENTINEL)
    fb.fa_paged_gather(dev(case.k_cache), dev(case.v_cache), dev_i32(case.block_table),
                       dev_i32(case.seq_lens), ko, vo, S, Hkv, 128, 16, case.num_pages, maxb,
                       splits)
    return ko, vo


def _host_gather(case, s):
    """Token t of sequence s is slot t % 16 of physical page block_table[s, t // 16]."""
    t = np.arange(int(case.seq_lens[s]))
    pages = case.block_table[s, t // 16]
    return case.k_cache.data[pages, :, t % 16, :], case.v_cache.data[pages, :, t % 16, :]


def _check_gathered(case, ko, vo, seqs):
    for s in seqs:
        L = int(case.seq_lens[s])
        k_ref, v_ref = _host_gather(case, s)
        kg = ko[s].cpu().numpy().view(np.uint16)
        vg = vo[s].cpu().numpy().view(np.uint16)
        assert np.array_equal(kg[:L], k_ref), f"K rows of sequence {s}"
        assert np.array_equal(vg[:L], v_ref), f"V rows of sequence {s}"
        assert (kg[L:] == _SENTINEL).all() and (vg[L:] == _SENTINEL).all(), f"rows past {L}"


@pytest.mark.parametrize("splits", [1, 3, 8, 64])
def test_gathered_rows_equal_host_gather(splits):
    """Split page ranges, page lookups, tensor-copy rows and the swizzled page
    layout of the decode give exactly the rows the block table names; nothing
    past seq_len (NaN-poisoned in the cache) is written."""
    lens = [0, 1, 15, 16, 17, 100, 257, 640]
    case = I.decode_case(5, num_seqs=len(lens), H=32, Hkv=8, d=128, lens=lens, max_blocks=48)
    ko, vo = _gpu_gather(case, splits)
    _check_gathered(case, ko, vo, range(len(lens)))
    assert fb.fa_get_device_status() == 0


def test_gathered_rows_full_size_pool():
    """The 64-sequence pool (contexts 512..8192) at 8 splits, sampled sequences."""
    case = I.c4_decode()
    ko, vo = _gpu_gather(case, 8)
    _check_gathered(case, ko, vo, [0, 17, 40, 63])
    assert fb.fa_get_device_status() == 0


@pytest.mark.parametrize("X, dv", [(6, 128), (1, 64), (33, 64), (64, 256), (40, 96)])
def test_split_combine_against_oracle_merge(X, dv):
    """Merge of arbitrary partials: splits past 32 (two per lane), the 64-split
    limit, and head dims that leave lanes idle (64, 96) or take two chunks."""
    rng = I.rng(11, X, dv)
    S, H = 3, 4
    pm = rng.normal(size=(S, H, X)) * 5
    pm[0, 0, :] = -np.inf                  # all empty
    pm[1, 2, ::2] = -np.inf                # some empty
    pl = np.where(np.isneginf(pm), 0.0, rng.uniform(0.5, 50, size=(S, H, X)))
    po = rng.normal(size=(S, H, X, dv)) * pl[..., None]
    po[np.isneginf(pm)] = 0.0
    pm32, pl32, po32 = (x.astype(np.float32) for x in (pm, pl, po))
    o, lse = fb.split_combine(torch.from_numpy(pm32).cuda(), torch.from_numpy(pl32).cuda(),
                              torch.from_numpy(po32).cuda())
    o_ref, lse_ref = oracle.split_combine(pm32, pl32, po32)
    assert_close(host(o), o_ref, BF16_MAX_ABS, BF16_MEAN_ABS)
    assert_lse_close(host(lse), lse_ref)


@pytest.mark.parametrize("splits", [4, 8, 16])
def test_c4_full_size(splits):
    """64 sequences, H=32, Hkv=8, d=128, page 16, lengths uniform on [512, 8192],
    block tables random slices of a shared pool, split into 4/8/16 chunks."""
    case = _c4()
    o, lse = _gpu_decode(case, splits)
    o_ref, lse_ref = _c4_ref()
    assert_close(host(o), o_ref, BF16_MAX_ABS, BF16_MEAN_ABS, what=f"c4 X={splits}")
    assert_lse_close(host(lse), lse_ref)
    assert fb.fa_get_device_status() == 0


_cache = {}


def _c4():
    if "case" not in _cache:
        _cache["case"] = I.c4_decode()
    return _cache["case"]


def _c4_ref():
    if "ref" not in _cache:
        _cache["ref"] = _oracle(_c4())
    return _cache["ref"]


def test_decode_step_replays_from_a_cuda_graph():
    """A decode step (split partials + merge) captured once in a CUDA graph and
    replayed gives the eager result bit for bit, also after the inputs change
    in place (pointers fixed, contents new)."""
    case = I.decode_case(12, num_seqs=8, H=32, Hkv=8, d=128,
                         lens=[17, 300, 1024, 5, 2048, 129, 700, 64], max_blocks=128)
    q, kc, vc = dev(case.q), dev(case.k_cache), dev(case.v_cache)
    bt, sl = dev_i32(case.block_table), dev_i32(case.seq_lens)
    S, X = 8, 8
    need = fb.fa_paged_decode_workspace_size(S, case.H, case.dv, X)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o = torch.empty((S, case.H, case.dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((S, case.H), dtype=torch.float32, device="cuda")

    def step(stream=None):
        fb.fa_paged_decode(q, kc, vc, bt, sl, o, lse, S, case.H, case.Hkv, case.d, case.dv,
                           case.page_size, case.num_pages, case.max_blocks, X, case.scale, ws,
                           need, stream)

    step()                       # eager: also does the one-time set-up
    torch.cuda.synchronize()
    o_eager, l_eager = o.clone(), lse.clone()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step(s)
    o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), o_eager.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), l_eager.view(torch.int32))
    # new query contents, same pointers: the replay follows them
    q.copy_(torch.flip(q, dims=[0]))
    step()
    torch.cuda.synchronize()
    o_eager2 = o.clone()
    o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), o_eager2.view(torch.int16))
    assert not torch.equal(o_eager2.view(torch.int16), o_eager.view(torch.int16))


def test_wait_timeout_sets_status_and_context_stays_usable(monkeypatch):
    """Failure detection without a fault: with the test hook set, each decode
    warp never requests its first page, its bounded wait runs out (~1 s), the
    kernel records FA_ERR_TIMEOUT and returns.  The next call, hook unset,
    runs normally on the same context."""
    case = I.decode_case(13, num_seqs=1, H=8, Hkv=2, d=128, lens=[100], max_blocks=8)
    monkeypatch.setenv("FA_TEST_FORCE_WAIT_TIMEOUT", "1")
    t0 = time.time()
    _gpu_decode(case, 1)
    assert fb.fa_get_device_status() == fb.FA_ERR_TIMEOUT
    assert time.time() - t0 < 30
    monkeypatch.delenv("FA_TEST_FORCE_WAIT_TIMEOUT")
    o, lse = _gpu_decode(case, 2)
    assert fb.fa_get_device_status() == 0
    o_ref, lse_ref = _oracle(case)
    assert_close(host(o), o_ref, BF16_MAX_ABS, BF16_MEAN_ABS)


# ------------------------------------------------------------ fused form
def _bits(x):
    return x.view(torch.int16 if x.dtype == torch.bfloat16 else torch.int32).cpu().numpy()


def _fused(case, splits, ws):
    return fb.paged_decode_fused(dev(case.q), dev(case.k_cache), dev(case.v_cache),
                                 dev_i32(case.block_table), dev_i32(case.seq_lens), splits,
                                 case.scale, workspace=ws)


def test_fused_decode_gives_the_two_launch_bits_across_calls():
    """fa_paged_decode_fused ("S12 FlashAttention", 接下来: fuse the
    small-batch decode) runs the same partials and, in the split that takes
    the last ticket, the same merge: O and LSE equal fa_paged_decode's bit for
    bit.  One workspace (zeroed once) serves every call, with the split count
    changing from call to call, so the ticket words must come back to zero."""
    lens = [0, 1, 15, 16, 17, 100, 257, 640]
    case = I.decode_case(5, num_seqs=len(lens), H=32, Hkv=8, d=128, lens=lens, max_blocks=48)
    need = fb.fa_paged_decode_workspace_size(len(lens), 32, 128, 64)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    o_ref, lse_ref = _oracle(case)
    for splits in (1, 3, 4, 8, 16, 64, 8, 5):
        o, lse = _fused(case, splits, ws)
        o2, lse2 = _gpu_decode(case, splits)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(o), _bits(o2)), f"O bits, X={splits}"
        assert np.array_equal(_bits(lse), _bits(lse2)), f"LSE bits, X={splits}"
        assert_close(host(o), o_ref, BF16_MAX_ABS, BF16_MEAN_ABS, what=f"fused X={splits}")
        assert_lse_close(host(lse), lse_ref, what=f"fused lse X={splits}")
        assert fb.fa_get_device_status() == 0


@pytest.mark.parametrize("group", [1, 4, 16])
def test_fused_decode_group_sizes(group):
    case = I.decode_case(6, num_seqs=3, H=2 * group, Hkv=2, d=128, lens=[33, 200, 511],
                         max_blocks=40)
    ws = torch.zeros(fb.fa_paged_decode_workspace_size(3, 2 * group, 128, 4), dtype=torch.uint8,
                     device="cuda")
    o, lse = _fused(case, 4, ws)
    o_ref, lse_ref = _oracle(case)
    assert_close(host(o), o_ref, BF16_MAX_ABS, BF16_MEAN_ABS, what=f"fused group {group}")
    assert_lse_close(host(lse), lse_ref)
    assert fb.fa_get_device_status() == 0


def test_fused_c4_full_size():
    """The 64-sequence workload at 4, 8 and 16 splits through one workspace:
    every output against the oracle and bit for bit against the two-launch form."""
    case = _c4()
    o_ref, lse_ref = _c4_ref()
    ws = torch.zeros(fb.fa_paged_decode_workspace_size(64, 32, 128, 16), dtype=torch.uint8,
                     device="cuda")
    for splits in (4, 8, 16):
        o, lse = _fused(case, splits, ws)
        o2, lse2 = _gpu_decode(case, splits)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(o), _bits(o2)) and np.array_equal(_bits(lse), _bits(lse2))
        assert_close(host(o), o_ref, BF16_MAX_ABS, BF16_MEAN_ABS, what=f"fused c4 X={splits}")
        assert_lse_close(host(lse), lse_ref)
    assert fb.fa_get_device_status() == 0


def test_fused_timeout_keeps_the_tickets_consistent(monkeypatch):
    """A fused call whose warps time out (test hook, no fault) still takes
    every ticket, so the next call on the same workspace merges correctly."""
    case = I.decode_case(13, num_seqs=2, H=8, Hkv=2, d=128, lens=[100, 300], max_blocks=24)
    ws = torch.zeros(fb.fa_paged_decode_workspace_size(2, 8, 128, 3), dtype=torch.uint8,
                     device="cuda")
    monkeypatch.setenv("FA_TEST_FORCE_WAIT_TIMEOUT", "1")
    _fused(case, 3, ws)
    assert fb.fa_get_device_status() == fb.FA_ERR_TIMEOUT
    monkeypatch.delenv("FA_TEST_FORCE_WAIT_TIMEOUT")
    o, lse = _fused(case, 3, ws)
    assert fb.fa_get_device_status() == 0
    o_ref, lse_ref = _oracle(case)
    assert_close(host(o), o_ref, BF16_MAX_ABS, BF16_MEAN_ABS)
    assert_lse_close(host(lse), lse_ref)
