"""Pins of the oracle's weight gradients (reading R16).

- The 128x1 re-quantisation: the largest element of every column tile maps to
  +-448, every code is within half an E4M3 step of the dequantised value, tiles
  restart at each 128-row block, padding is code 0; and it equals the 1x128
  quantiser applied to the transposed float32 matrix (a different route to the
  same layout).
- The token-contracted GEMM: bit-exact against float64 numpy on small integers
  with power-of-two scales (every partial sum exact), so operand order, slab
  placement and scale indexing are fixed.
- The layer: the gradient's definition.  A central finite difference of the
  float64, unquantised loss  L(W) = sum_t dh_t . h'_t(W)  along the oracle's
  gradient, and the float64 backprop formulas entry by entry, agree with the
  oracle to FP8 accuracy; a transposed or missing term is off by O(1).
"""
import numpy as np
import pytest
import torch

from fine_grained_fp8_bias_b300 import workloads as wl
from tests.helpers import bits, oracle_weights

CFG = wl.TINY.with_(T=200)          # shared expert: 200 rows (a 128 + 72 block split)


def _rand_fp8(rng, shape, orc):
    x = rng.standard_normal(shape).astype(np.float32) * rng.choice([0.01, 1.0, 30.0], size=shape[:1])[:, None]
    q, s = orc.quant_1x128(x.astype(np.float32))
    return q, s


def _deq_rows(orc, q, s):
    """float32 dec(q) * s with one scale per 1x128 tile of a row."""
    d = orc.e4m3_decode(q).astype(np.float32)
    return d * np.repeat(s.astype(np.float32), 128, axis=1)


def test_requant_128x1_properties(orc):
    rng = np.random.default_rng(11)
    M, C = 300, 256
    q, s = _rand_fp8(rng, (M, C), orc)
    qt, st = orc.requant_128x1(q, s)
    assert qt.shape == (C, 384) and st.shape == (C, 3)
    x = _deq_rows(orc, q, s).T                       # [C, M] float32
    assert np.all(qt[:, M:] == 0)
    for b in range(3):
        blk = x[:, b * 128:min(M, b * 128 + 128)]
        amax = np.abs(blk).max(axis=1)
        assert np.array_equal(st[:, b], np.where(amax == 0, 1.0, amax / np.float32(448.0)).astype(np.float32))
        codes = qt[:, b * 128:b * 128 + blk.shape[1]]
        j = np.abs(blk).argmax(axis=1)
        top = codes[np.arange(C), j]
        assert np.all((top == 0x7E) | (top == 0xFE) | (amax == 0))
        v = blk / st[:, b:b + 1]
        dq = orc.e4m3_decode(codes)
        mag = np.maximum(np.abs(v), 2.0 ** -6)
        half = 2.0 ** (np.floor(np.log2(mag)) - 4)   # half an E4M3 step (3 mantissa bits)
        assert np.all(np.abs(v - dq) <= half * (1 + 1e-6))


def test_requant_128x1_equals_row_quantiser_on_the_transpose(orc):
    rng = np.random.default_rng(12)
    M, C = 257, 384
    q, s = _rand_fp8(rng, (M, C), orc)
    qt, st = orc.requant_128x1(q, s)
    xt = np.zeros((C, 384), np.float32)
    xt[:, :M] = _deq_rows(orc, q, s).T
    q2, s2 = orc.quant_1x128(xt)
    assert np.array_equal(qt, q2)
    assert np.array_equal(st, s2)


def test_requant_zero_column_tile(orc):
    q = np.zeros((130, 128), np.uint8)
    s = np.ones((130, 1), np.float32)
    q[129, 5] = 0x38                                  # 1.0 in the second block only
    qt, st = orc.requant_128x1(q, s)
    assert st[5, 0] == 1.0 and st[5, 1] == np.float32(1.0) / np.float32(448.0)
    assert np.all(qt[:, :128] == 0) and qt[5, 129] == 0x7E


def _int_codes(rng, shape, orc):
    v = rng.integers(-8, 9, size=shape).astype(np.float32)
    return orc.e4m3_encode(v), v.astype(np.float64)


def test_rowscaled_gemm_exact_on_integers(orc):
    rng = np.random.default_rng(13)
    Na, Nb, Kd = 256, 384, 384
    qa, a = _int_codes(rng, (Na, Kd), orc)
    qb, b = _int_codes(rng, (Nb, Kd), orc)
    # |slab sum| <= 128 * 64 = 2^13 and sa * sb in 2^[-4, 4]: every partial and
    # every float32 sum of three slabs fits 24 bits, so any order is exact
    sa = (2.0 ** rng.integers(-2, 3, size=(Na, Kd // 128))).astype(np.float32)
    sb = (2.0 ** rng.integers(-2, 3, size=(Nb, Kd // 128))).astype(np.float32)
    got = orc.gemm_fp8_rowscaled(qa, sa, qb, sb)
    ref = np.zeros((Na, Nb))
    for kb in range(Kd // 128):
        sl = slice(kb * 128, kb * 128 + 128)
        ref += (a[:, sl] @ b[:, sl].T) * sa[:, kb:kb + 1].astype(np.float64) * sb[:, kb].astype(np.float64)
    assert np.array_equal(got, ref.astype(np.float32))


def test_rowscaled_gemm_random_close_to_float64(orc):
    rng = np.random.default_rng(14)
    Na, Nb, Kd = 128, 256, 512
    qa, sa = _rand_fp8(rng, (Na, Kd), orc)
    qb, sb = _rand_fp8(rng, (Nb, Kd), orc)
    # one scale per row per slab on both sides: use the row-tile scales as such
    got = orc.gemm_fp8_rowscaled(qa, sa, qb, sb)
    ref = _deq_rows(orc, qa, sa).astype(np.float64) @ _deq_rows(orc, qb, sb).astype(np.float64).T
    err = np.abs(got - ref).max() / np.abs(ref).max()
    assert err < 1e-5


# ------------------------------------------------------------ the layer
def _setup(orc, cfg, seed=4, dh_zero=False, starve=None):
    inp = wl.small_inputs(cfg)
    bias = inp["bias"].numpy().copy()
    if starve is not None:
        bias[starve] = -10.0                           # nobody selects this expert
    r = orc.route(bits(inp["u"]), inp["centroids"].numpy(), bias, cfg.K)
    W = oracle_weights(orc, cfg, set(range(cfg.E + cfg.S)))
    dh = wl.normal(wl.stream_key(seed, 78), (cfg.T, cfg.d), 1.0).to(torch.bfloat16)
    if dh_zero:
        dh = torch.zeros_like(dh)
    return inp, r, W, dh


def _group_w(W, g):
    return W.gate[g], W.up[g], W.down[g]


def _deq_w(orc, q, s):
    return orc.e4m3_decode(q).astype(np.float64) * np.kron(s.astype(np.float64), np.ones((128, 128)))


def _rows(cfg, r, g):
    if g >= cfg.E:
        return np.arange(cfg.T), np.ones(cfg.T)
    t, k = np.nonzero(r["idx"] == g)
    return t, r["gate"][t, k].astype(np.float64)


def _loss(u, dh, gk, Wg, Wu, Wd):
    """float64 sum over the group's rows of dh_t . g_k y(u_t)."""
    G, U = u @ Wg.T, u @ Wu.T
    y = (G / (1 + np.exp(-G)) * U) @ Wd.T
    return float(np.sum(gk[:, None] * dh * y))


@pytest.mark.parametrize("g", [3, CFG.E])          # a routed expert, the shared expert
def test_layer_wgrad_matches_the_gradient(orc, g):
    cfg = CFG
    inp, r, W, dh = _setup(orc, cfg)
    dWg, dWu, dWd = orc.layer_backward_wgrad(bits(inp["u"]), r["idx"], r["gate"], _group_w(W, g),
                                             bits(dh), cfg.d, cfg.E, cfg.K, cfg.I, g)
    t, gk = _rows(cfg, r, g)
    assert len(t) > 0
    u = inp["u"].to(torch.float64).numpy()[t]
    dhf = dh.to(torch.float64).numpy()[t]
    Wg, Wu, Wd = (_deq_w(orc, *w) for w in _group_w(W, g))
    # float64 backprop, entry by entry
    G, U = u @ Wg.T, u @ Wu.T
    sg = 1 / (1 + np.exp(-G))
    h = G * sg * U
    dy = gk[:, None] * dhf
    dH = dy @ Wd
    ref_d = dy.T @ h
    ref_g = (dH * U * sg * (1 + G * (1 - sg))).T @ u
    ref_u = (dH * G * sg).T @ u
    errs = [np.linalg.norm(a - b) / np.linalg.norm(b) for a, b in
            ((dWg, ref_g), (dWu, ref_u), (dWd, ref_d))]
    print(f"group {g} rows {len(t)}: rel err gate {errs[0]:.3e} up {errs[1]:.3e} down {errs[2]:.3e}")
    # each product has both operands rounded to E4M3 twice (1x128, then 128x1):
    # about 2 x 3.6% relative, independent per element
    assert max(errs) < 0.1
    # the definition: a central difference of the float64 loss along the
    # oracle's own gradient gives <dW_true, dW> / <dW, dW>: 1 to FP8 accuracy,
    # near 0 for a transposed or misplaced gradient, negative for a sign error
    Ws = [Wg, Wu, Wd]
    for name, dW, which in (("gate", dWg, 0), ("up", dWu, 1), ("down", dWd, 2)):
        V = dW.astype(np.float64)
        eps = 1e-3 * np.linalg.norm(Ws[which]) / np.linalg.norm(V)
        hi = list(Ws); hi[which] = Ws[which] + eps * V
        lo = list(Ws); lo[which] = Ws[which] - eps * V
        fd = (_loss(u, dhf, gk, *hi) - _loss(u, dhf, gk, *lo)) / (2 * eps)
        got = float(np.sum(V * V))
        print(f"  {name}: <dW, dW> {got:.6e}  finite difference along dW {fd:.6e}")
        assert 0.9 < fd / got < 1.1


def test_layer_wgrad_zero_gradient_and_unused_expert(orc):
    cfg = CFG
    inp, r, W, dh = _setup(orc, cfg, dh_zero=True)
    for g in (0, cfg.E):
        out = orc.layer_backward_wgrad(bits(inp["u"]), r["idx"], r["gate"], _group_w(W, g), bits(dh),
                                       cfg.d, cfg.E, cfg.K, cfg.I, g)
        assert all(not np.any(x) for x in out)
    inp, r, W, dh = _setup(orc, cfg, starve=5)
    assert not np.any(r["idx"] == 5)
    out = orc.layer_backward_wgrad(bits(inp["u"]), r["idx"], r["gate"], _group_w(W, 5), bits(dh),
                                   cfg.d, cfg.E, cfg.K, cfg.I, 5)
    assert all(not np.any(x) for x in out)
