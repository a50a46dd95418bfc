"""Pins for the oracle's E4M3 codec against torch.float8_e4m3fn (an independent implementation)."""
import numpy as np
import pytest
import torch


def torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_encode(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_decode_all_256_codes(orc):
    codes = np.arange(256, dtype=np.uint8)
    ours = orc.e4m3_decode(codes)
    ref = torch_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert set(np.flatnonzero(nan)) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def test_round_trip_all_finite_codes(orc):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = orc.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(orc.e4m3_encode(vals), codes)


def test_encode_every_bf16_value_in_range(orc):
    bits = np.arange(65536, dtype=np.uint32) << 16
    x = bits.view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) <= 448.0)]
    assert np.array_equal(orc.e4m3_encode(x), torch_encode(x))


def test_encode_ties_go_to_even(orc):
    codes = np.arange(0, 126, dtype=np.uint8)
    lo = orc.e4m3_decode(codes)
    hi = orc.e4m3_decode(codes + 1)
    mid = ((lo + hi) / 2).astype(np.float32)       # exact in float32
    assert np.array_equal(mid.astype(np.float64), (lo + hi) / 2)
    got = orc.e4m3_encode(mid)
    want = np.where(codes % 2 == 0, codes, codes + 1).astype(np.uint8)
    assert np.array_equal(got, want)
    assert np.array_equal(got, torch_encode(mid))
    assert np.array_equal(orc.e4m3_encode(-mid), want | 0x80)


def test_encode_random_float32(orc):
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-12, 6, 200000))).astype(np.float32)
    x = x[np.abs(x) <= 448]
    assert np.array_equal(orc.e4m3_encode(x), torch_encode(x))


@pytest.mark.parametrize("v", [448.0, 448.5, 463.9, 464.0, 500.0, 1e6, 3e38])
def test_encode_saturates(orc, v):
    assert orc.e4m3_encode(np.array([v, -v], np.float32)).tolist() == [0x7E, 0xFE]


def test_encode_subnormals_and_zero(orc):
    x = np.array([0.0, -0.0, 2 ** -9, 2 ** -10, 3 * 2 ** -10, 2 ** -11, 7 * 2 ** -9, 2 ** -6],
                 np.float32)
    assert orc.e4m3_encode(x).tolist() == [0x00, 0x80, 0x01, 0x00, 0x02, 0x00, 0x07, 0x08]
