"""GPU parity of the quantisers, the router and the dispatch against the oracle
(bit-exact for codes, scales, indices, counts and rows)."""
import numpy as np
import pytest
import torch

from fine_grained_fp8_bias_b300 import workloads as wl
from tests.helpers import bits, routing_agreement

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    from fine_grained_fp8_bias_b300 import lib
    return lib


def test_generator_cpu_and_cuda_agree():
    for cfg, which, g in ((wl.V3_PREFILL, "gate", 5), (wl.MID, "down", 65), (wl.TINY, "up", 0)):
        a = wl.master_weight(cfg, which, g, "cpu")
        b = wl.master_weight(cfg, which, g, "cuda").cpu()
        assert torch.equal(a, b)
    assert torch.equal(wl.tokens(wl.TINY, "cpu"), wl.tokens(wl.TINY, "cuda").cpu())
    assert torch.equal(wl.tokens(wl.V3_LONG.with_(T=64), "cpu"),
                       wl.tokens(wl.V3_LONG.with_(T=64), "cuda").cpu())
    assert torch.equal(wl.centroids(wl.V3_DECODE, "cpu"), wl.centroids(wl.V3_DECODE, "cuda").cpu())
    assert torch.equal(wl.bias(wl.TINY, "cpu"), wl.bias(wl.TINY, "cuda").cpu())


def test_e4m3_conversion_sweep(L, orc):
    # tiles led by 448 have scale exactly 1, so the codes are E4M3(x) itself
    allb = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    vals = allb[np.isfinite(allb) & (np.abs(allb) <= 448.0)]
    rows = (len(vals) + 126) // 127
    x = np.zeros((rows, 128), np.float32)
    x[:, 0] = 448.0
    flat = x[:, 1:].reshape(-1)
    flat[: len(vals)] = vals
    x[:, 1:] = flat.reshape(rows, 127)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    q, s = L.moe_quant_1x128(xb.cuda())
    torch.cuda.synchronize()
    assert torch.all(s.cpu() == 1.0)
    assert np.array_equal(q.cpu().numpy(), orc.e4m3_encode(xb.float().numpy()))


@pytest.mark.parametrize("M,d", [(1, 128), (37, 384), (300, 2048), (129, 7168)])
def test_quant_1x128_bit_exact(L, orc, M, d):
    x = wl.normal(wl.stream_key(31, M, d), (M, d), 1.0)
    x[0, :128] = 0.0                                   # zero tile
    if M > 2:
        x[1, 128:256] = x[1, 128:256] * 1e-4            # tiny tile
        x[2] = x[2] * 300.0                             # saturating-range tile
    xb = x.to(torch.bfloat16)
    q, s = L.moe_quant_1x128(xb.cuda())
    qo, so = orc.quant_1x128(bits(xb))
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(s.cpu().numpy(), so.T)        # GPU layout is [d/128, M]


def test_quant_1x128_gather_and_bad_index(L, orc):
    n, d = 50, 512
    xb = wl.normal(wl.stream_key(32), (n, d), 2.0).to(torch.bfloat16)
    gather = torch.tensor([3, 3, 49, 0, 17, 8, 8, 8], dtype=torch.int32)
    q, s = L.moe_quant_1x128(xb.cuda(), gather.cuda(), scale_ld=11)
    qo, so = orc.quant_1x128(bits(xb[gather.long()]))
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(s.cpu().numpy()[:, :8], so.T)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    bad = torch.tensor([1, 50, -1], dtype=torch.int32, device="cuda")
    L.moe_quant_1x128(xb.cuda(), bad, status=status)
    assert L.moe_check_device_status(status) == -7
    assert L.moe_check_device_status(status) == 0      # read clears it


@pytest.mark.parametrize("R,C", [(128, 128), (256, 384), (2048, 7168)])
def test_quant_128x128_bit_exact(L, orc, R, C):
    w = wl.normal(wl.stream_key(33, R, C), (R, C), 1.0 / np.sqrt(C))
    w[:128, :128] = 0.0
    q, s = L.moe_quant_128x128(w.cuda())
    qo, so = orc.quant_128x128(w.numpy())
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(s.cpu().numpy(), so)


def route_case(L, orc, cfg, T=None):
    cfg = cfg if T is None else cfg.with_(T=T)
    inp = wl.small_inputs(cfg)
    g = L.moe_route(inp["u"].cuda(), inp["centroids"].cuda(), inp["bias"].cuda(), cfg.K)
    torch.cuda.synchronize()
    r = orc.route(bits(inp["u"]), inp["centroids"].numpy(), inp["bias"].numpy(), cfg.K)
    bad = routing_agreement(g["idx"].cpu().numpy(), g["gate"].cpu().numpy(), r,
                            bias=inp["bias"].numpy())
    counts = g["counts"].cpu().numpy()
    assert np.array_equal(counts, np.bincount(g["idx"].cpu().numpy().ravel(), minlength=cfg.E))
    if len(bad) == 0:
        assert np.array_equal(counts, r["counts"])
    # the flag may differ only where the GPU's own gap is itself borderline
    tie_g = g["tie"].cpu().numpy()
    assert (tie_g != r["tie"]).sum() <= max(2, cfg.T // 1000)
    return r, g, bad


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_route_configs(L, orc, name):
    route_case(L, orc, wl.CONFIGS[name])


def test_route_v3_prefill_full(L, orc):
    r, g, bad = route_case(L, orc, wl.V3_PREFILL)
    print(f"v3 prefill: flagged {int(r['tie'].sum())} tokens, mismatched {len(bad)}")


@pytest.mark.parametrize("T", [1, 16, 64, 256])
def test_route_v3_decode(L, orc, T):
    route_case(L, orc, wl.V3_DECODE, T)


def test_route_edges(L, orc):
    # K = E, the largest E and K, and T not a multiple of any tile
    for cfg in (wl.LayerConfig("ke", T=33, d=128, E=8, K=8, S=0, I=128, seed=40),
                wl.LayerConfig("big", T=70, d=256, E=1024, K=32, S=0, I=128, seed=41),
                wl.LayerConfig("odd", T=131, d=384, E=100, K=7, S=0, I=128, seed=42)):
        route_case(L, orc, cfg)


# up to 1024 selections one block sorts them (T = 1, 16, 128 at K = 8; 32 x 32 over
# 1024 experts); beyond, the three chunked kernels
@pytest.mark.parametrize("T,K,E", [(1, 1, 1), (65, 3, 7), (300, 8, 256), (4096, 8, 256),
                                   (200, 32, 1024), (129, 6, 64), (1, 8, 256), (16, 8, 256),
                                   (128, 8, 256), (129, 8, 256), (32, 32, 1024), (5, 8, 1024)])
def test_permute_bit_exact(L, orc, T, K, E):
    rng = np.random.default_rng(T * 7 + E)
    pool = np.array([e for e in range(E) if e != 2 or E <= K + 1])   # expert 2 stays empty
    idx = np.stack([rng.choice(pool, K, replace=False) for _ in range(T)]).astype(np.int32)
    S = 2
    out = L.moe_permute(torch.from_numpy(idx).cuda(), E, S)
    torch.cuda.synchronize()
    o = orc.dispatch(idx, E)
    assert np.array_equal(out["offsets"].cpu().numpy(), o["offsets"])
    assert np.array_equal(out["perm_token"].cpu().numpy()[: T * K], o["perm_token"])
    assert np.array_equal(out["inv_row"].cpu().numpy(), o["inv_row"])
    # shared-expert groups: S blocks of T rows, one per token
    go = out["group_offsets"].cpu().numpy()
    assert np.array_equal(go[: E + 1], o["offsets"])
    assert np.array_equal(go[E:], T * K + T * np.arange(S + 1))
    assert np.array_equal(out["perm_token"].cpu().numpy()[T * K:], np.tile(np.arange(T), S))


def test_permute_bad_index_flagged(L):
    # the one-block sort (4 selections) and the chunked kernels (1600)
    idx = torch.tensor([[0, 1], [2, 9]], dtype=torch.int32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    L.moe_permute(idx, 4, status=status)
    assert L.moe_check_device_status(status) == -7
    big = torch.randint(0, 64, (200, 8), dtype=torch.int32, device="cuda")
    big[100, 3] = 64
    L.moe_permute(big, 64, status=status)
    assert L.moe_check_device_status(status) == -7


def test_update_bias_bit_exact(L, orc):
    E, T, K = 256, 4096, 8
    b = wl.bias(wl.V3_PREFILL)
    counts = np.random.default_rng(3).integers(100, 160, E).astype(np.int32)
    counts[:4] = T * K // E                                # exactly average
    bd = b.cuda()
    L.moe_update_bias(torch.from_numpy(counts).cuda(), bd, T, K, 1e-3)
    torch.cuda.synchronize()
    assert np.array_equal(bd.cpu().numpy(), orc.update_bias(counts, b.numpy(), T, K, 1e-3))


# The last two cases have at least 148 * 64 * 4 = 37888 256-wide steps, so the
# kernel takes four steps of a token per warp item; the last one's d (65 tiles
# of 128) leaves a partly filled final item.
@pytest.mark.parametrize("T,K,S,E,d", [(1, 1, 1, 4, 128), (97, 3, 2, 16, 384), (300, 8, 1, 64, 2048),
                                       (2600, 8, 1, 64, 4096), (1200, 2, 1, 16, 8320)])
def test_quant_dispatch_bit_exact(L, orc, T, K, S, E, d):
    rng = np.random.default_rng(T + d)
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    o = orc.dispatch(idx, E)
    x = wl.normal(wl.stream_key(34, T, d), (T, d), 1.5)
    x[0, :128] = 0.0
    xb = x.to(torch.bfloat16)
    q, s = L.moe_quant_1x128_dispatch(xb.cuda(), torch.from_numpy(o["inv_row"]).cuda(), K, S)
    torch.cuda.synchronize()
    qt, st = orc.quant_1x128(bits(xb))                # each token quantised once
    rows = np.concatenate([o["perm_token"], np.tile(np.arange(T), S)])
    assert np.array_equal(q.cpu().numpy(), qt[rows])
    assert np.array_equal(s.cpu().numpy(), st[rows].T)
