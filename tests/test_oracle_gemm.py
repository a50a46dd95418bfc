"""Pins for the oracle's block-scaled FP8 GEMM with FP32 promotion every 128 K."""
import numpy as np
import torch

from fine_grained_fp8_bias_b300 import workloads as wl


def int_codes(orc, shape, vmax, seed):
    rng = np.random.default_rng(seed)
    v = rng.integers(-vmax, vmax + 1, shape).astype(np.float32)
    return orc.e4m3_encode(v), v.astype(np.int64)


def pow2(shape, seed, lo=-6, hi=3):
    rng = np.random.default_rng(seed)
    return np.exp2(rng.integers(lo, hi, shape)).astype(np.float32)


def test_exact_integer_case(orc):
    M, N, K = 37, 200 // 8 * 8 + 56, 384          # N = 256
    qa, va = int_codes(orc, (M, K), 8, 1)
    qw, vw = int_codes(orc, (N, K), 8, 2)
    sa, sw = pow2((M, K // 128), 3), pow2((N // 128, K // 128), 4)
    out = orc.gemm_fp8(qa, sa, qw, sw)
    ref = np.zeros((M, N), np.float64)
    for kb in range(K // 128):
        sl = slice(kb * 128, (kb + 1) * 128)
        dot = va[:, sl] @ vw[:, sl].T                    # exact integers
        ref += dot * sa[:, kb:kb + 1] * np.repeat(sw[:, kb], 128)[None, :]
    assert np.array_equal(out.astype(np.float64), ref)


def test_random_case_against_dense_fp64(orc):
    M, N, K = 19, 256, 512
    a = wl.normal(wl.stream_key(9, 1), (M, K), 1.0).numpy()
    w = wl.normal(wl.stream_key(9, 2), (N, K), 0.05).numpy()
    qa, sa = orc.quant_1x128(a)
    qw, sw = orc.quant_128x128(w)
    out = orc.gemm_fp8(qa, sa, qw, sw).astype(np.float64)
    dec = lambda q: torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy()
    A = dec(qa) * np.repeat(sa, 128, 1)
    W = dec(qw) * np.repeat(np.repeat(sw, 128, 0), 128, 1)
    ref = A @ W.T
    bound = np.abs(A) @ np.abs(W).T
    assert np.all(np.abs(out - ref) <= 1e-6 * bound + 1e-30)
    # and the dequantised product approximates the unquantised one
    rel = np.linalg.norm(out - a.astype(np.float64) @ w.astype(np.float64).T) / np.linalg.norm(ref)
    assert rel < 0.05


def test_scale_placement(orc):
    # one nonzero slab and one nonzero weight block pick out exactly one scale pair
    M, N, K = 2, 256, 256
    qa = np.zeros((M, K), np.uint8)
    qw = np.zeros((N, K), np.uint8)
    qa[:, 128:] = orc.e4m3_encode(np.ones(128, np.float32))
    qw[128:, 128:] = orc.e4m3_encode(np.full(128, 2.0, np.float32))
    sa = np.array([[3.0, 0.5], [7.0, 0.25]], np.float32)
    sw = np.array([[11.0, 13.0], [17.0, 0.125]], np.float32)
    out = orc.gemm_fp8(qa, sa, qw, sw)
    assert np.all(out[:, :128] == 0)
    assert np.all(out[0, 128:] == np.float32(256 * 0.5 * 0.125))
    assert np.all(out[1, 128:] == np.float32(256 * 0.25 * 0.125))
