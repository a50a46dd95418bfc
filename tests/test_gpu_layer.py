"""GPU parity of the whole layer forward (moe_forward through the C ABI) against the oracle."""
import numpy as np
import pytest
import torch

from fine_grained_fp8_bias_b300 import workloads as wl
from tests.helpers import MAX_ABS, REL_FRO, bits, oracle_weights, rel_fro, routing_agreement

pytestmark = pytest.mark.gpu


def gpu_forward(cfg, step=0, layer=None):
    from fine_grained_fp8_bias_b300.layer import MoELayer
    L = layer or MoELayer.from_config(cfg, "cuda")
    u = wl.tokens(cfg, "cuda", step)
    out = L.forward(u)
    torch.cuda.synchronize()
    assert L.status() == 0
    return L, u, out


def check_layer(orc, cfg, tokens=None, layer=None):
    L, u, out = gpu_forward(cfg, layer=layer)
    u_cpu = u.cpu()
    r = orc.route(bits(u_cpu), wl.centroids(cfg).numpy(), wl.bias(cfg).numpy(), cfg.K)
    gidx = out["idx"].cpu().numpy()
    bad = routing_agreement(gidx, out["gate"].cpu().numpy(), r)
    toks = np.arange(cfg.T) if tokens is None else np.asarray(tokens)
    toks = np.array([t for t in toks if t not in set(bad.tolist())], np.int64)
    need = set(range(cfg.E, cfg.E + cfg.S))
    for t in toks:
        need.update(int(e) for e in r["idx"][t])
    W = oracle_weights(orc, cfg, need)
    ref = orc.layer_forward(bits(u_cpu), r["idx"], r["gate"], W, cfg.d, cfg.E, cfg.K, cfg.S, cfg.I, toks)
    got = out["h"].cpu().numpy()[toks]
    err_f, err_m = rel_fro(got, ref), float(np.abs(got - ref).max())
    print(f"{cfg.name}: tokens {len(toks)} rel_fro {err_f:.3e} max_abs {err_m:.3e} "
          f"flagged {int(r['tie'].sum())} mismatched {len(bad)}")
    assert err_f <= REL_FRO and err_m <= MAX_ABS
    # the routed part alone (h' - u) must also be close: u does not hide errors
    du = u_cpu.float().numpy()[toks]
    assert rel_fro(got - du, ref - du) <= 10 * REL_FRO
    if len(bad) == 0:
        assert np.array_equal(out["counts"].cpu().numpy(), r["counts"])
    return L, u, out, r


def test_tiny_full(orc):
    check_layer(orc, wl.TINY)


def test_ragged_small(orc):
    # T not a multiple of any tile, S = 2, I = 384 (3 N tiles), d = 640 (d % 256 = 128)
    cfg = wl.LayerConfig("ragged", T=301, d=640, E=12, K=3, S=2, I=384, seed=17)
    check_layer(orc, cfg)


def test_single_token_and_k1(orc):
    check_layer(orc, wl.LayerConfig("t1", T=1, d=256, E=16, K=1, S=1, I=128, seed=18))
    check_layer(orc, wl.LayerConfig("noshared", T=50, d=256, E=8, K=2, S=0, I=256, seed=19))


def test_mid_sampled(orc):
    check_layer(orc, wl.MID, tokens=[0, 1, 777, 2048, 4095])


def test_v3_prefill_sampled(orc):
    # the benchmark's workload and launch configuration, checked on sampled tokens
    check_layer(orc, wl.V3_PREFILL, tokens=[0, 4095])


@pytest.mark.parametrize("T", [1, 16])
def test_v3_decode(orc, T):
    cfg = wl.V3_DECODE.with_(T=T)
    check_layer(orc, cfg, tokens=[0, T - 1] if T > 1 else [0])


def test_forward_then_bias_update(orc):
    cfg = wl.TINY
    L, u, out, r = check_layer(orc, cfg)
    b0 = wl.bias(cfg).numpy()
    L.update_bias(out["counts"], cfg.T, cfg.gamma)
    torch.cuda.synchronize()
    assert np.array_equal(L.bias.cpu().numpy(), orc.update_bias(r["counts"], b0, cfg.T, cfg.K, cfg.gamma))


def test_zero_weights_identity():
    from fine_grained_fp8_bias_b300.layer import MoELayer
    cfg = wl.TINY
    L = MoELayer(cfg.d, cfg.E, cfg.K, cfg.S, cfg.I, "cuda")
    L.centroids.copy_(wl.centroids(cfg, "cuda"))
    u = wl.tokens(cfg, "cuda")
    out = L.forward(u)
    torch.cuda.synchronize()
    assert torch.equal(out["h"], u.float())


def test_forward_is_deterministic():
    from fine_grained_fp8_bias_b300.layer import MoELayer
    L = MoELayer.from_config(wl.TINY, "cuda")
    u = wl.tokens(wl.TINY, "cuda")
    a = L.forward(u)
    h1 = a["h"].clone()
    b = L.forward(u)
    torch.cuda.synchronize()
    assert torch.equal(h1, b["h"])
