"""Shared test helpers: moving seeded inputs to the GPU and comparing results."""
import numpy as np

BF16_MAX_ABS = 2e-2   # bf16 inputs, fp32 accumulation: max |O - oracle|
BF16_MEAN_ABS = 2e-3  # ... and mean |O - oracle|
F32_MAX_ABS = 1e-5    # fp32 path
LSE_ABS = 1e-3        # LSE, every path


def dev(t):
    """inputs.Tensor -> CUDA tensor of its storage type (bf16 from the bit patterns)."""
    import torch
    if t.dtype == "bf16":
        return torch.from_numpy(t.data.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(t.data).cuda()


def dev_i32(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def host(x):
    import torch
    return x.detach().float().cpu().numpy().astype(np.float64)


def assert_close(got, want, max_abs, mean_abs=None, what=""):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values in result"
    err = np.abs(got - want)
    mx = float(err.max()) if err.size else 0.0
    assert mx <= max_abs, f"{what}: max-abs {mx:.3e} > {max_abs:.1e} at {np.unravel_index(err.argmax(), err.shape)}"
    if mean_abs is not None and err.size:
        mn = float(err.mean())
        assert mn <= mean_abs, f"{what}: mean-abs {mn:.3e} > {mean_abs:.1e}"
    return mx


def assert_lse_close(got, want, what=""):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape
    both_inf = np.isneginf(got) & np.isneginf(want)
    assert np.array_equal(np.isneginf(got), np.isneginf(want)), f"{what}: -inf pattern differs"
    with np.errstate(invalid="ignore"):
        err = np.abs(np.where(both_inf, 0.0, got - want))
    assert np.isfinite(err).all(), f"{what}: non-finite LSE"
    mx = float(err.max()) if err.size else 0.0
    assert mx <= LSE_ABS, f"{what}: LSE max-abs {mx:.3e} > {LSE_ABS:.1e}"
    return mx
