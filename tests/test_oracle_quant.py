"""Pins for the oracle's fine-grained quantisation (1x128 activation tiles, 128x128 weight blocks)."""
import numpy as np
import torch

from fine_grained_fp8_bias_b300 import workloads as wl


def bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16)


def bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def torch_quant_tiles(x32, rows, cols):
    """Library composition: scale = amax / 448 (torch float32 division), codes = cast(x / scale)."""
    x = torch.from_numpy(x32)
    M, D = x.shape
    t = x.reshape(M // rows, rows, D // cols, cols).permute(0, 2, 1, 3)
    amax = t.abs().amax(dim=(2, 3), keepdim=True)
    scale = torch.where(amax == 0, torch.ones_like(amax), amax / torch.tensor(448.0))
    q = (t / scale).to(torch.float8_e4m3fn).view(torch.uint8)
    q = torch.where(amax == 0, torch.zeros_like(q), q)
    q = q.permute(0, 2, 1, 3).reshape(M, D)
    return q.numpy(), scale.reshape(M // rows, D // cols).numpy()


def test_1x128_matches_library_composition(orc):
    u = wl.normal(wl.stream_key(7, 1), (37, 512), 1.0)
    u[3, :128] = 0.0                       # a zero tile
    u[5, 128:256] *= 1e-3                  # a small-scale tile
    ub = u.to(torch.bfloat16)
    q, s = orc.quant_1x128(bits(ub))
    qr, sr = torch_quant_tiles(ub.float().numpy(), 1, 128)
    assert np.array_equal(q, qr)
    assert np.array_equal(s, sr)


def test_1x128_float32_input(orc):
    x = wl.normal(wl.stream_key(7, 2), (9, 384), 3.0).numpy()
    q, s = orc.quant_1x128(x)
    qr, sr = torch_quant_tiles(x, 1, 128)
    assert np.array_equal(q, qr) and np.array_equal(s, sr)


def test_amax_element_maps_to_448_and_error_bound(orc):
    x = wl.normal(wl.stream_key(7, 3), (64, 256), 1.0).numpy()
    q, s = orc.quant_1x128(x)
    dec = orc.e4m3_decode(np.arange(256, dtype=np.uint8))
    for r in range(64):
        for b in range(2):
            tile = x[r, b * 128:(b + 1) * 128]
            qt = q[r, b * 128:(b + 1) * 128]
            j = np.argmax(np.abs(tile))
            assert qt[j] == (0xFE if tile[j] < 0 else 0x7E)
            assert s[r, b] == np.float32(np.abs(tile).max()) / np.float32(448.0)
            # every code is a nearest E4M3 neighbour of x / scale
            v = (tile / s[r, b]).astype(np.float64)
            err = np.abs(v - dec[qt])
            mag = np.abs(dec[qt])
            ulp = np.where(mag < 2 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(mag, 2 ** -6))) - 3))
            assert np.all(err <= ulp / 2 + 1e-12)


def test_zero_tile_reading(orc):
    q, s = orc.quant_1x128(np.zeros((2, 256), np.float32))
    assert np.all(q == 0) and np.all(s == 1.0)
    x = np.zeros((1, 128), np.float32)
    x[0, 0] = -0.0
    q, s = orc.quant_1x128(x)
    assert np.all(q == 0) and s[0, 0] == 1.0


def test_power_of_two_rescale_invariance(orc):
    x = wl.normal(wl.stream_key(7, 4), (4, 256), 1.0).numpy()
    q1, s1 = orc.quant_1x128(x)
    q2, s2 = orc.quant_1x128(x * np.float32(2.0 ** -7))
    assert np.array_equal(q1, q2)
    assert np.array_equal(s2, s1 * np.float32(2.0 ** -7))


def test_tiles_are_independent(orc):
    x = wl.normal(wl.stream_key(7, 5), (3, 384), 1.0).numpy()
    q, s = orc.quant_1x128(x)
    y = x.copy()
    y[:, 128:256] *= 5.0
    q2, s2 = orc.quant_1x128(y)
    assert np.array_equal(q[:, :128], q2[:, :128]) and np.array_equal(q[:, 256:], q2[:, 256:])
    assert np.array_equal(s[:, 0], s2[:, 0]) and np.array_equal(s[:, 2], s2[:, 2])


def test_128x128_matches_library_composition(orc):
    w = wl.normal(wl.stream_key(7, 6), (256, 384), 1 / 16).numpy()
    w[128:, 256:] = 0.0
    q, s = orc.quant_128x128(w)
    qr, sr = torch_quant_tiles(w, 128, 128)
    assert s.shape == (2, 3)
    assert np.array_equal(q, qr) and np.array_equal(s, sr)
