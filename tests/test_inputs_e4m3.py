"""CPU pins of the e4m3 (FP8) input encoding used by the FP8 forward's tests:
every finite code round-trips, rounding is to nearest with ties to the even
code and saturates at 448, and it agrees with torch's float8_e4m3fn cast."""
import numpy as np
import torch

from tiled_online_softmax_sm_gb300 import inputs as I


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = I.e4m3_bits_to_f32(codes)
    back = I.f32_to_e4m3_bits(vals)
    assert np.array_equal(back, codes)
    assert np.nanmax(np.abs(vals)) == 448.0


def test_ties_and_library_agreement():
    codes = np.array([c for c in range(0, 0x7F)], np.uint8)
    v = I.e4m3_bits_to_f32(codes).astype(np.float64)
    mids = (v[:-1] + v[1:]) / 2          # exact halfway points between neighbours
    x = np.concatenate([mids, -mids, np.random.default_rng(1).normal(size=20000) * 80])
    x = x.astype(np.float32)
    ours = I.f32_to_e4m3_bits(x)
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, lib)
    got = I.e4m3_bits_to_f32(ours[: len(mids)])
    # ties go to the even code
    assert np.all(I.f32_to_e4m3_bits(got) % 2 == 0)


def test_saturation_and_power_of_two_descale():
    assert I.e4m3_bits_to_f32(I.f32_to_e4m3_bits(np.array([1e6, -1e6], np.float32))).tolist() == [448.0, -448.0]
    t = I.Tensor.from_f32(np.random.default_rng(2).normal(size=(64, 8)).astype(np.float32) * 3, "e4m3")
    assert t.descale == 2.0 ** round(np.log2(t.descale))
    assert np.array_equal(t.values, (I.e4m3_bits_to_f32(t.data) * np.float32(t.descale)))
