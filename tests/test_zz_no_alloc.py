"""fa_paged_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (plugins whose host framework owns every device
allocation, serving loops that must not allocate once running).

It must give what fa_paged_decode gives on the same inputs, bit for bit (the
same kernels run on the same inputs; only where the split partials live
differs), also on the second of two calls in a row (the fixed scratch array
keeps the previous call's contents); its calls must leave the device's free
memory unchanged; and it must refuse problems whose partials exceed the array.
This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes when run on its own.
"""
import numpy as np
import pytest
import torch

from tiled_online_softmax_sm_gb300 import binding as fb
from tiled_online_softmax_sm_gb300 import build as fbuild
from tiled_online_softmax_sm_gb300 import inputs as I

from _helpers import dev, dev_i32


def _args(case):
    return (dev(case.q), dev(case.k_cache), dev(case.v_cache), dev_i32(case.block_table),
            dev_i32(case.seq_lens))


def _noalloc(case, splits, tensors):
    q, kc, vc, bt, sl = tensors
    S = len(case.seq_lens)
    o = torch.full((S, case.H, case.dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((S, case.H), float("nan"), dtype=torch.float32, device="cuda")
    fb.fa_paged_decode_noalloc(q, kc, vc, bt, sl, o, lse, S, case.H, case.Hkv, case.d, case.dv,
                               case.page_size, case.num_pages, case.max_blocks, splits, case.scale)
    return o, lse


def _bits(x):
    return x.view(torch.int16 if x.dtype == torch.bfloat16 else torch.int32).cpu().numpy()


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_two_calls_in_a_row():
    # first call: many splits; second call: a different problem with fewer,
    # so stale partials of the first call would show if they leaked
    first = I.decode_case(71, num_seqs=12, H=32, Hkv=8, d=128,
                          lens=[1, 16, 17, 300, 511, 1024, 2000, 64, 5, 999, 4096, 33],
                          max_blocks=256)
    second = I.decode_case(72, num_seqs=7, H=16, Hkv=4, d=128,
                           lens=[700, 3, 128, 129, 4000, 15, 2500], max_blocks=256)
    for case, splits in ((first, 16), (second, 5)):
        t = _args(case)
        o_ref, lse_ref = fb.paged_decode(*t, splits, case.scale)
        o, lse = _noalloc(case, splits, t)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(o), _bits(o_ref)), f"O bits differ at X={splits}"
        assert np.array_equal(_bits(lse), _bits(lse_ref)), f"LSE bits differ at X={splits}"
        assert fb.fa_get_device_status() == 0


@pytest.mark.gpu
def test_noalloc_calls_leave_free_device_memory_unchanged():
    """After a first call (which only looks up the array's address), further
    calls take no device memory: the free bytes the driver reports do not move."""
    case = I.decode_case(73, num_seqs=8, H=32, Hkv=8, d=128,
                         lens=[1, 300, 4096, 17, 2000, 64, 999, 5], max_blocks=256)
    t = _args(case)
    S = len(case.seq_lens)
    o = torch.empty((S, case.H, case.dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((S, case.H), dtype=torch.float32, device="cuda")
    call = lambda: fb.fa_paged_decode_noalloc(*t[:5], o, lse, S, case.H, case.Hkv, case.d, case.dv,
                                              case.page_size, case.num_pages, case.max_blocks, 8,
                                              case.scale)
    call()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        call()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    assert fb.fa_get_device_status() == 0


def test_noalloc_rejects_problems_beyond_the_fixed_scratch():
    fbuild.build()
    lib = fb.load()
    S, H, X = 64, 32, 64          # partials of 64 seqs x 32 heads x 64 splits: 68 MB > 16 MiB
    assert fb.fa_paged_decode_workspace_size(S, H, 128, X) > fb.FA_NOALLOC_SCRATCH_BYTES
    rc = lib.fa_paged_decode_noalloc(16, 16, 16, 16, 16, 16, 16, S, H, 8, 128, 128, 16, 100, 8, X,
                                     0.1, None)
    assert rc == fb.FA_ERR_WORKSPACE
    assert "fixed scratch" in fb.fa_last_error()
