"""Pins of the oracle's input gradient (reading R15) against a float64 chain
built from library pieces: dequantised weights and activations, numpy matmuls,
and torch autograd for the gates' dependence on u.  The oracle quantises every
backward GEMM operand to E4M3, so the two agree to FP8 accuracy; a wrong
transpose, sign or missing term is off by O(1)."""
import numpy as np
import pytest
import torch

from fine_grained_fp8_bias_b300 import workloads as wl
from tests.helpers import bits, oracle_weights

CFG = wl.TINY.with_(T=12)


def _setup(orc, cfg, seed=3, zero_weights=False):
    inp = wl.small_inputs(cfg)
    u = inp["u"]
    r = orc.route(bits(u), inp["centroids"].numpy(), inp["bias"].numpy(), cfg.K)
    W = oracle_weights(orc, cfg, set(range(cfg.E + cfg.S)))
    if zero_weights:
        for g in range(cfg.E + cfg.S):
            W.set(g, (np.zeros_like(W.gate[g][0]), W.gate[g][1]), (np.zeros_like(W.up[g][0]), W.up[g][1]),
                  (np.zeros_like(W.down[g][0]), W.down[g][1]))
    dh = wl.normal(wl.stream_key(seed, 77), (cfg.T, cfg.d), 1.0).to(torch.bfloat16)
    return inp, r, W, dh


def _deq(orc, q, s, rows_blk, cols_blk):
    d = orc.e4m3_decode(q).astype(np.float64)
    return d * np.kron(s.astype(np.float64), np.ones((rows_blk, cols_blk)))


def _reference(orc, cfg, inp, r, W, dh, with_gate_term=True):
    """float64 du from the unquantised backward formulas."""
    E, K, S, d, I = cfg.E, cfg.K, cfg.S, cfg.d, cfg.I
    u = inp["u"].to(torch.float64).numpy()
    c = inp["centroids"].to(torch.float64).numpy()
    dhf = dh.to(torch.float64).numpy()
    qa, sa = orc.quant_1x128(bits(inp["u"]))
    a = _deq(orc, qa, sa, 1, 128)
    out = np.empty((cfg.T, d))
    for t in range(cfg.T):
        acc = dhf[t].copy()
        dg = np.zeros(K)
        groups = [(E + s, 1.0, None) for s in range(S)] + \
                 [(int(r["idx"][t, k]), float(r["gate"][t, k]), k) for k in range(K)]
        for g, gk, k in groups:
            Wg = _deq(orc, *W.gate[g], 128, 128)
            Wu = _deq(orc, *W.up[g], 128, 128)
            Wd = _deq(orc, *W.down[g], 128, 128)
            G, U = a[t] @ Wg.T, a[t] @ Wu.T
            sg = 1.0 / (1.0 + np.exp(-G))
            y = (G * sg * U) @ Wd.T
            dH = (gk * dhf[t]) @ Wd
            dG = dH * U * sg * (1 + G * (1 - sg))
            dU = dH * G * sg
            acc += dG @ Wg + dU @ Wu
            if k is not None:
                dg[k] = dhf[t] @ y
        if with_gate_term:
            ut = torch.tensor(u[t], requires_grad=True)
            sel = torch.tensor(c[r["idx"][t]])
            s_ = torch.sigmoid(sel @ ut)
            gates = s_ / s_.sum()
            (gates * torch.tensor(dg)).sum().backward()
            acc += ut.grad.numpy()
        out[t] = acc
    return out


def test_zero_weights_give_the_residual_exactly(orc):
    inp, r, W, dh = _setup(orc, CFG, zero_weights=True)
    du = orc.layer_backward_dgrad(bits(inp["u"]), r["idx"], r["gate"], W, inp["centroids"].numpy(),
                                  bits(dh), CFG.d, CFG.E, CFG.K, CFG.S, CFG.I, range(CFG.T))
    assert np.array_equal(du, dh.to(torch.float32).numpy())


def test_against_float64_chain(orc):
    inp, r, W, dh = _setup(orc, CFG)
    du = orc.layer_backward_dgrad(bits(inp["u"]), r["idx"], r["gate"], W, inp["centroids"].numpy(),
                                  bits(dh), CFG.d, CFG.E, CFG.K, CFG.S, CFG.I, range(CFG.T))
    ref = _reference(orc, CFG, inp, r, W, dh)
    resid = dh.to(torch.float64).numpy()
    # compare the part that is not the residual dh (the residual is exact)
    err = np.linalg.norm(du - ref) / np.linalg.norm(ref - resid)
    print(f"backward vs float64 chain: relative error {err:.3e} of |du - dh|")
    assert err < 0.08


def test_gate_term_is_there_with_its_sign(orc):
    inp, r, W, dh = _setup(orc, CFG)
    du = orc.layer_backward_dgrad(bits(inp["u"]), r["idx"], r["gate"], W, inp["centroids"].numpy(),
                                  bits(dh), CFG.d, CFG.E, CFG.K, CFG.S, CFG.I, range(CFG.T))
    with_g = _reference(orc, CFG, inp, r, W, dh, True)
    without = _reference(orc, CFG, inp, r, W, dh, False)
    gate_part = np.linalg.norm(with_g - without)
    print(f"gate term {gate_part:.3e}; oracle to reference {np.linalg.norm(du - with_g):.3e}; "
          f"to reference without it {np.linalg.norm(du - without):.3e}; "
          f"with it negated {np.linalg.norm(du - (2 * without - with_g)):.3e}")
    # the oracle's departure from the no-gate-term reference, projected on the
    # gate term: 1 when the term is there with its sign, 0 if missing, -1 if
    # negated (the FP8 error hardly projects on this one direction)
    gdir = (with_g - without).ravel()
    proj = float(np.dot((du - without).ravel(), gdir) / np.dot(gdir, gdir))
    print(f"projection on the gate term: {proj:.3f}")
    assert 0.85 < proj < 1.15
