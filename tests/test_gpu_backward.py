"""GPU parity of the layer's input gradient (moe_backward_dgrad, reading R15)
against the oracle, and of the transposed weight blocks it uses."""
import numpy as np
import pytest
import torch

from fine_grained_fp8_bias_b300 import workloads as wl
from tests.helpers import bits, oracle_weights, rel_fro, routing_agreement

pytestmark = pytest.mark.gpu

DU_REL = 5e-3      # relative Frobenius error of du - dh (the non-residual part)


def _layer(cfg):
    from fine_grained_fp8_bias_b300.layer import MoELayer
    return MoELayer.from_config(cfg, "cuda")


def test_transposed_weights_are_exact():
    cfg = wl.TINY
    L = _layer(cfg)
    L.prepare_backward()
    torch.cuda.synchronize()
    wdt, sdt, wgut, sgut = (t.cpu().numpy() for t in L._bwd_w)
    wd, sd = L.w_down.cpu().numpy(), L.s_down.cpu().numpy()
    wg, sg = L.w_gate.cpu().numpy(), L.s_gate.cpu().numpy()
    wu, su = L.w_up.cpu().numpy(), L.s_up.cpu().numpy()
    I = cfg.I
    assert np.array_equal(wdt, wd.transpose(0, 2, 1))
    assert np.array_equal(sdt, sd.transpose(0, 2, 1))
    assert np.array_equal(wgut[:, :, :I], wg.transpose(0, 2, 1))
    assert np.array_equal(wgut[:, :, I:], wu.transpose(0, 2, 1))
    assert np.array_equal(sgut[:, :, :I // 128], sg.transpose(0, 2, 1))
    assert np.array_equal(sgut[:, :, I // 128:], su.transpose(0, 2, 1))


def _run(cfg, zero=False, seed=5):
    L = _layer(cfg)
    if zero:
        for t in (L.w_gate, L.w_up, L.w_down):
            t.zero_()
    u = wl.tokens(cfg, "cuda")
    out = L.forward(u)
    dh = wl.normal(wl.stream_key(seed, 88), (cfg.T, cfg.d), 1.0, "cuda").to(torch.bfloat16)
    du = L.backward_dgrad(u, dh, out)
    torch.cuda.synchronize()
    assert L.status() == 0 and L.backward_status() == 0
    return L, u, out, dh, du


def test_zero_weights_give_the_residual():
    cfg = wl.TINY
    _, _, _, dh, du = _run(cfg, zero=True)
    assert torch.equal(du, dh.float())


def _check(orc, cfg, tokens=None):
    L, u, out, dh, du = _run(cfg)
    u_cpu = u.cpu()
    r = orc.route(bits(u_cpu), wl.centroids(cfg).numpy(), wl.bias(cfg).numpy(), cfg.K)
    gidx, ggate = out["idx"].cpu().numpy(), out["gate"].cpu().numpy()
    bad = routing_agreement(gidx, ggate, r, bias=wl.bias(cfg).numpy())
    toks = np.arange(cfg.T) if tokens is None else np.asarray(tokens)
    toks = np.array([t for t in toks if t not in set(bad.tolist())], np.int64)
    need = set(range(cfg.E, cfg.E + cfg.S)) | {int(e) for t in toks for e in gidx[t]}
    W = oracle_weights(orc, cfg, need)
    # the oracle differentiates the forward the GPU ran (its routing and gates)
    ref = orc.layer_backward_dgrad(bits(u_cpu), gidx, ggate, W, wl.centroids(cfg).numpy(),
                                   bits(dh.cpu()), cfg.d, cfg.E, cfg.K, cfg.S, cfg.I, toks)
    got = du.cpu().numpy()[toks]
    base = dh.float().cpu().numpy()[toks]
    err = rel_fro(got - base, ref - base)
    mx = float(np.abs(got - ref).max())
    print(f"{cfg.name}: tokens {len(toks)} backward rel_fro(du - dh) {err:.3e} max_abs {mx:.3e}")
    assert err <= DU_REL


def test_backward_tiny(orc):
    _check(orc, wl.TINY)


def test_backward_ragged(orc):
    _check(orc, wl.LayerConfig("ragged", T=301, d=640, E=24, K=3, S=2, I=384, seed=23),
           tokens=range(0, 301, 7))


def test_backward_v3_sampled(orc):
    _check(orc, wl.V3_PREFILL, tokens=[0, 4095])
