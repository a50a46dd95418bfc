"""GPU parity of the whole layer forward (moe_forward through the C ABI) against the oracle."""
import numpy as np
import pytest
import torch

from fine_grained_fp8_bias_b300 import workloads as wl
from tests.helpers import (MAX_ABS, REL_FRO, bits, layer_forward_threaded, oracle_weights_threaded,
                           rel_fro, route_threaded, routing_agreement, tile_covering_tokens)

pytestmark = pytest.mark.gpu


def gpu_forward(cfg, step=0, layer=None, u=None):
    from fine_grained_fp8_bias_b300.layer import MoELayer
    L = layer or MoELayer.from_config(cfg, "cuda")
    u = wl.tokens(cfg, "cuda", step) if u is None else u
    out = L.forward(u)
    torch.cuda.synchronize()
    assert L.status() == 0
    return L, u, out


def check_layer(orc, cfg, tokens=None, layer=None, u=None, cover=(64, 256)):
    """Layer output of the CUDA path against the oracle on the listed tokens
    (all tokens when None; "cover": tokens whose dispatch rows reach every
    shared-expert M tile and the first, last and last-tile rows of cover[0]
    routed experts, cover[1] tokens in all)."""
    L, u, out = gpu_forward(cfg, layer=layer, u=u)
    u_cpu = u.cpu()
    r = route_threaded(orc, bits(u_cpu), wl.centroids(cfg).numpy(), wl.bias(cfg).numpy(), cfg.K)
    gidx = out["idx"].cpu().numpy()
    bad = routing_agreement(gidx, out["gate"].cpu().numpy(), r, bias=wl.bias(cfg).numpy())
    if isinstance(tokens, str) and tokens == "cover":
        toks, picked = tile_covering_tokens(r["idx"], cfg, n_groups=cover[0], total=cover[1])
    else:
        toks, picked = (np.arange(cfg.T) if tokens is None else np.asarray(tokens)), []
    toks = np.array([t for t in toks if t not in set(bad.tolist())], np.int64)
    need = set(range(cfg.E, cfg.E + cfg.S))
    for t in toks:
        need.update(int(e) for e in r["idx"][t])
    W = oracle_weights_threaded(orc, cfg, need)
    ref = layer_forward_threaded(orc, bits(u_cpu), r["idx"], r["gate"], W, cfg, toks)
    got = out["h"].cpu().numpy()[toks]
    err_f, err_m = rel_fro(got, ref), float(np.abs(got - ref).max())
    print(f"{cfg.name}: tokens {len(toks)} (experts {len(need)}, covered groups {len(picked)}) "
          f"rel_fro {err_f:.3e} max_abs {err_m:.3e} flagged {int(r['tie'].sum())} "
          f"mismatched {len(bad)}")
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


@pytest.fixture(scope="module")
def v3_layer():
    # V3 prefill and its skewed form share the weight seed: one device copy
    from fine_grained_fp8_bias_b300.layer import MoELayer
    L = MoELayer.from_config(wl.V3_PREFILL, "cuda")
    yield L
    del L
    torch.cuda.empty_cache()


def test_v3_prefill_sampled(orc, v3_layer):
    # the benchmark's workload and launch configuration, checked on >= 256 tokens
    # whose rows cover all 32 M tiles of the shared expert and the first, last and
    # ragged-last-tile rows of 64 routed experts plus the largest and smallest
    check_layer(orc, wl.V3_PREFILL, tokens="cover", layer=v3_layer)


def test_v3_skew_sampled(orc, v3_layer):
    # 16 hot experts take ~40% of the selections: their groups span many M tiles
    cfg = wl.V3_SKEW
    v3_layer.centroids.copy_(wl.centroids(cfg, "cuda"))
    try:
        _, _, out, r = check_layer(orc, cfg, tokens="cover", layer=v3_layer, cover=(64, 256))
        hot = r["counts"][:cfg.hot_experts].sum() / (cfg.T * cfg.K)
        assert hot > 0.3, hot
    finally:
        v3_layer.centroids.copy_(wl.centroids(wl.V3_PREFILL, "cuda"))


def with_outliers(cfg, u, n_tok=48, scale=100.0):
    """u with one isolated large activation (+-scale, i.e. >= 100 sigma of the
    N(0, 1) draw) in one 1x128 tile of each of n_tok tokens: the case 1x128
    tile scaling is for (the outlier sets only its own tile's scale)."""
    u = u.clone()
    rng = np.random.default_rng(cfg.seed + 1000)
    toks = rng.choice(cfg.T, size=min(n_tok, cfg.T), replace=False)
    cols = rng.integers(0, cfg.d, size=len(toks))
    sign = rng.choice([-1.0, 1.0], size=len(toks))
    for t, c, sg in zip(toks, cols, sign):
        u[int(t), int(c)] = float(sg * scale)
    return u, np.sort(toks)


def test_mid_outliers(orc):
    cfg = wl.MID
    u, toks = with_outliers(cfg, wl.tokens(cfg, "cuda"), n_tok=48)
    # every token with an outlier, plus a few without
    check_layer(orc, cfg, tokens=list(toks) + [0, 1, cfg.T - 1], u=u)


def test_v3_prefill_outliers(orc, v3_layer):
    cfg = wl.V3_PREFILL
    u, toks = with_outliers(cfg, wl.tokens(cfg, "cuda"), n_tok=48)
    check_layer(orc, cfg, tokens=list(toks) + [0, 1, cfg.T - 1], layer=v3_layer, u=u)


@pytest.mark.parametrize("T", [1, 16, 64, 255, 256])
def test_v3_decode(orc, T):
    # below 256 tokens the layer routes with the CUDA-core exact router, from 256 on
    # with the tensor-core screen
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


@pytest.mark.parametrize("T", [1, 16, 200])
def test_small_batch_forward_is_deterministic(T):
    # the small-batch router sums its split partial logits in a fixed order
    from fine_grained_fp8_bias_b300.layer import MoELayer
    cfg = wl.V3_DECODE.with_(T=T)
    L = MoELayer.from_config(wl.TINY.with_(d=1024, E=64, K=6), "cuda")
    u = wl.tokens(cfg.with_(d=1024), "cuda")
    outs = []
    for _ in range(3):
        o = L.forward(u)
        outs.append({k: v.clone() for k, v in o.items()})
    torch.cuda.synchronize()
    for o in outs[1:]:
        for k in ("h", "idx", "gate", "tie", "counts"):
            assert torch.equal(o[k], outs[0][k]), k


@pytest.mark.parametrize("name,n", [("tiny", 5), ("ragged", 4)])
def test_forward_host_pipeline_matches_sequential_calls(name, n):
    # moe_forward_host overlaps uploads, compute and downloads on three streams
    # with two device buffer sets; it must give exactly what moe_forward +
    # moe_update_bias give batch after batch (the bias moves between batches)
    from fine_grained_fp8_bias_b300.layer import MoELayer
    cfg = wl.TINY if name == "tiny" else wl.LayerConfig("ragged", T=301, d=640, E=24, K=3, S=2,
                                                        I=384, seed=23)
    gamma = 0.01
    seq = MoELayer.from_config(cfg, "cuda")
    pipe = MoELayer.from_config(cfg, "cuda")
    batches = [wl.tokens(cfg, "cpu", step=k) for k in range(n)]
    ref_h, ref_idx = [], []
    for u in batches:
        out = seq.forward(u.cuda())
        seq.update_bias(out["counts"], cfg.T, gamma)
        ref_h.append(out["h"].cpu())
        ref_idx.append(out["idx"].cpu())
    torch.cuda.synchronize()
    u_host = [wl.pinned_like(u) for u in batches]
    h_host = [torch.full((cfg.T, cfg.d), float("nan"), dtype=torch.float32, pin_memory=True)
              for _ in range(n)]
    bufs = pipe.forward_host(u_host, h_host, gamma)
    torch.cuda.synchronize()
    assert pipe.status() == 0
    for k in range(n):
        assert torch.equal(h_host[k], ref_h[k]), k
    # the last two batches' routing stays in the two buffer sets
    for k in (n - 2, n - 1):
        assert torch.equal(bufs[k % 2]["idx"].cpu(), ref_idx[k])
    assert torch.equal(pipe.bias, seq.bias)
    assert not torch.equal(pipe.bias, wl.bias(cfg).cuda())      # the bias did move
