"""GPU checks of moe_route's screening step: the tensor-core logit estimates
stay far inside the error bound the candidate band is built from, and the
inputs that defeat the screen (many equal scores, large token norms) still
route exactly as the oracle does."""
import numpy as np
import pytest
import torch

from fine_grained_fp8_bias_b300 import workloads as wl
from tests.helpers import bits, routing_agreement

pytestmark = pytest.mark.gpu

BOUND_GAMMA = 2.0 ** -11     # the router's bound: |l~_e - l_e| <= gamma |u_t| |c_e|


@pytest.fixture(scope="module")
def L():
    from fine_grained_fp8_bias_b300 import lib
    return lib


@pytest.mark.parametrize("name,n_sample", [("tiny", 256), ("mid", 512), ("v3_prefill", 384),
                                           ("v3_skew", 384)])
def test_estimate_error_far_inside_bound(L, name, n_sample):
    cfg = wl.CONFIGS[name]
    inp = wl.small_inputs(cfg)
    est, norms = L.moe_route_estimate_logits(inp["u"].cuda(), inp["centroids"].cuda())
    torch.cuda.synchronize()
    rng = np.random.default_rng(7)
    rows = np.sort(rng.choice(cfg.T, size=min(n_sample, cfg.T), replace=False))
    u = inp["u"][rows].to(torch.float64).numpy()
    c = inp["centroids"].to(torch.float64).numpy()
    exact = u @ c.T                                   # float64 reference logits
    got = est.cpu().numpy()[rows].astype(np.float64)
    norms_c = np.sqrt((c * c).sum(1))
    nk = norms.cpu().numpy().astype(np.float64)
    assert np.all(nk >= norms_c * (1 - 1e-6))
    scale = np.sqrt((u * u).sum(1))[:, None] * nk[None, :]
    ratio = float(np.max(np.abs(got - exact) / scale))
    print(f"{name}: max |l~_e - l_e| / (|u| |c_e|) = {ratio:.3e} (bound {BOUND_GAMMA:.3e})")
    # the estimate must sit well inside the bound the candidate band assumes
    assert ratio <= BOUND_GAMMA / 20


def _route_against_oracle(L, orc, u, c, b, K):
    g = L.moe_route(u.cuda(), c.cuda(), b.cuda(), K)
    torch.cuda.synchronize()
    r = orc.route(bits(u), c.numpy(), b.numpy(), K)
    bad = routing_agreement(g["idx"].cpu().numpy(), g["gate"].cpu().numpy(), r, bias=b.numpy())
    return g, r, bad


def test_all_scores_equal_takes_all_experts(L, orc):
    # zero tokens: every logit is 0, every score 0.5 -> more candidates than the
    # screen keeps, so every expert is recomputed; the lowest indices win
    T, d, E, K = 37, 256, 64, 6
    u = torch.zeros((T, d), dtype=torch.bfloat16)
    c = wl.normal(wl.stream_key(3, 9), (E, d), 1.0 / np.sqrt(d))
    b = torch.zeros(E)
    g, r, bad = _route_against_oracle(L, orc, u, c, b, K)
    idx = g["idx"].cpu().numpy()
    assert np.array_equal(idx, np.tile(np.arange(K), (T, 1)))
    assert np.allclose(g["gate"].cpu().numpy(), 1.0 / K, rtol=1e-6)
    assert np.all(g["tie"].cpu().numpy() == 1)


def test_bias_makes_a_block_of_equal_scores(L, orc):
    # a bias of +1 on 40 experts for half the tokens' worth of ties: the first
    # 40 experts share a large offset, so many near-equal biased scores sit at
    # the K-th place and the band holds more than 32 candidates for some tokens
    cfg = wl.LayerConfig("eqblock", T=200, d=512, E=128, K=8, S=0, I=128, seed=51)
    inp = wl.small_inputs(cfg)
    u = (inp["u"].float() * 1e-3).to(torch.bfloat16)      # tiny logits: s ~ 0.5 everywhere
    b = torch.zeros(cfg.E)
    b[:40] = 1.0
    g, r, bad = _route_against_oracle(L, orc, u, inp["centroids"], b, cfg.K)
    print(f"equal-block: flagged {int(r['tie'].sum())}, mismatched {len(bad)}")


@pytest.mark.parametrize("scale", [1.0 / 64, 64.0])
def test_large_and_small_token_norms(L, orc, scale):
    # the band scales with |u_t|; very large and very small tokens route exactly
    cfg = wl.LayerConfig("norm", T=300, d=1024, E=256, K=8, S=0, I=128, seed=52)
    inp = wl.small_inputs(cfg)
    u = (inp["u"].float() * scale).to(torch.bfloat16)
    g, r, bad = _route_against_oracle(L, orc, u, inp["centroids"], inp["bias"], cfg.K)
    print(f"scale {scale}: flagged {int(r['tie'].sum())}, mismatched {len(bad)}")


def test_route_v3_skew_full(L, orc):
    # 16 hot experts with long centroids take 40% of the selections: the
    # per-expert bounds keep the candidate band narrow for the other experts
    cfg = wl.V3_SKEW
    inp = wl.small_inputs(cfg)
    g, r, bad = _route_against_oracle(L, orc, inp["u"], inp["centroids"], inp["bias"], cfg.K)
    hot = float((g["idx"].cpu().numpy() < cfg.hot_experts).mean())
    print(f"v3_skew: hot fraction {hot:.3f}, flagged {int(r['tie'].sum())}, mismatched {len(bad)}")
    assert hot > 0.3
