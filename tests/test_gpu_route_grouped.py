"""GPU parity of group-limited routing (moe_route_grouped and moe_forward with
n_groups > 0) against the oracle's orc_route_grouped (reading R14)."""
import numpy as np
import pytest
import torch

from fine_grained_fp8_bias_b300 import workloads as wl
from tests.helpers import MAX_ABS, REL_FRO, bits, oracle_weights, rel_fro, routing_agreement

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    from fine_grained_fp8_bias_b300 import lib
    return lib


CASES = {
    "tiny": wl.TINY.with_(n_groups=4, topk_groups=2, group_topk=2),
    "mid": wl.MID.with_(n_groups=8, topk_groups=3, group_topk=2),
    "v3_small": wl.V3_GROUPED.with_(T=300),
    "odd": wl.LayerConfig("odd", T=77, d=384, E=96, K=5, S=0, I=128, seed=61, n_groups=12,
                          topk_groups=3, group_topk=3),
    "v3_skew": wl.V3_SKEW.with_(T=300, n_groups=8, topk_groups=4, group_topk=2),
}


def _check(L, orc, cfg, u=None, b=None):
    inp = wl.small_inputs(cfg)
    u = inp["u"] if u is None else u
    b = inp["bias"] if b is None else b
    g = L.moe_route_grouped(u.cuda(), inp["centroids"].cuda(), b.cuda(), cfg.K, cfg.n_groups,
                            cfg.topk_groups, cfg.group_topk)
    torch.cuda.synchronize()
    r = orc.route_grouped(bits(u), inp["centroids"].numpy(), b.numpy(), cfg.K, cfg.n_groups,
                          cfg.topk_groups, cfg.group_topk)
    gidx = g["idx"].cpu().numpy()
    bad = routing_agreement(gidx, g["gate"].cpu().numpy(), r, bias=b.numpy())
    gsz = cfg.E // cfg.n_groups
    assert all(len(set((row // gsz).tolist())) <= cfg.topk_groups for row in gidx)
    counts = g["counts"].cpu().numpy()
    assert np.array_equal(counts, np.bincount(gidx.ravel(), minlength=cfg.E))
    if len(bad) == 0:
        assert np.array_equal(counts, r["counts"])
    tie_g = g["tie"].cpu().numpy()
    assert (tie_g != r["tie"]).sum() <= max(2, cfg.T // 1000)
    print(f"{cfg.name}: flagged {int(r['tie'].sum())}, mismatched {len(bad)}")
    return g, r


@pytest.mark.parametrize("name", sorted(CASES))
def test_grouped_routing_matches_oracle(L, orc, name):
    _check(L, orc, CASES[name])


def test_grouped_routing_v3_prefill_full(L, orc):
    _check(L, orc, wl.V3_GROUPED)


def test_grouped_all_scores_equal(L, orc):
    # zero tokens: every score is 0.5; groups 0 .. topk_groups-1 are kept and the
    # lowest experts win; every group score ties, so every token is flagged
    cfg = CASES["mid"].with_(T=20)
    u = torch.zeros((cfg.T, cfg.d), dtype=torch.bfloat16)
    g, r = _check(L, orc, cfg, u=u, b=torch.zeros(cfg.E))
    assert np.array_equal(g["idx"].cpu().numpy(), np.tile(np.arange(cfg.K), (cfg.T, 1)))
    assert np.all(g["tie"].cpu().numpy() == 1)


def test_forward_with_group_routing(orc):
    from fine_grained_fp8_bias_b300.layer import MoELayer
    cfg = CASES["tiny"]
    layer = MoELayer.from_config(cfg, "cuda")
    u = wl.tokens(cfg, "cuda")
    out = layer.forward(u)
    torch.cuda.synchronize()
    assert layer.status() == 0
    u_cpu = u.cpu()
    r = orc.route_grouped(bits(u_cpu), wl.centroids(cfg).numpy(), wl.bias(cfg).numpy(), cfg.K,
                          cfg.n_groups, cfg.topk_groups, cfg.group_topk)
    bad = routing_agreement(out["idx"].cpu().numpy(), out["gate"].cpu().numpy(), r,
                            bias=wl.bias(cfg).numpy())
    toks = np.array([t for t in range(cfg.T) if t not in set(bad.tolist())], np.int64)
    need = set(range(cfg.E, cfg.E + cfg.S)) | {int(e) for t in toks for e in r["idx"][t]}
    W = oracle_weights(orc, cfg, need)
    ref = orc.layer_forward(bits(u_cpu), r["idx"], r["gate"], W, cfg.d, cfg.E, cfg.K, cfg.S,
                            cfg.I, toks)
    got = out["h"].cpu().numpy()[toks]
    assert rel_fro(got, ref) <= REL_FRO and float(np.abs(got - ref).max()) <= MAX_ABS
