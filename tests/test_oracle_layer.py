"""Pins for the oracle's layer output h'_t = u_t + shared FFNs + sum_k g_k FFN_k(u_t)."""
import numpy as np
import pytest
import torch

from fine_grained_fp8_bias_b300 import workloads as wl

CFG = wl.LayerConfig("pin", T=40, d=256, E=8, K=2, S=1, I=256, seed=21)


def bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def dec(q):
    return torch.from_numpy(np.ascontiguousarray(q)).view(torch.float8_e4m3fn).double()


def weights(orc, cfg, zero_routed=False, zero_all=False):
    def fn(which, g):
        w = wl.master_weight(cfg, which, g).numpy()
        if zero_all or (zero_routed and g < cfg.E):
            w = np.zeros_like(w)
        return w
    return orc.quantised_weights(cfg, range(cfg.E + cfg.S), fn)


def library_ffn(qa, sa, W, g):
    """FFN of one expert from library routines: dense fp64 matmuls of the dequantised
    operands, torch SiLU, and torch's float8 cast for the 1x128 re-quantisation of h."""
    a = dec(qa) * torch.from_numpy(np.repeat(sa, 128, 1)).double()

    def deq(pair):
        q, s = pair
        return dec(q) * torch.from_numpy(np.repeat(np.repeat(s, 128, 0), 128, 1)).double()

    G = (a @ deq(W.gate[g]).T).float()
    U = (a @ deq(W.up[g]).T).float()
    h = torch.nn.functional.silu(G) * U
    M, I = h.shape
    t = h.view(M, I // 128, 128)
    amax = t.abs().amax(-1, keepdim=True)
    scale = torch.where(amax == 0, torch.ones_like(amax), amax / torch.tensor(448.0))
    qh = (t / scale).to(torch.float8_e4m3fn).double() * scale.double()
    return qh.view(M, I) @ deq(W.down[g]).T


@pytest.fixture(scope="module")
def setup(orc):
    u = wl.tokens(CFG)
    r = orc.route(bits(u), wl.centroids(CFG).numpy(), wl.bias(CFG).numpy(), CFG.K)
    return u, r


def fwd(orc, u, r, W, toks, cfg=CFG):
    return orc.layer_forward(bits(u), r["idx"], r["gate"], W, cfg.d, cfg.E, cfg.K, cfg.S, cfg.I, toks)


def test_all_zero_weights_give_identity(orc, setup):
    u, r = setup
    out = fwd(orc, u, r, weights(orc, CFG, zero_all=True), range(CFG.T))
    assert np.array_equal(out, u.float().numpy())


def test_shared_expert_always_applied(orc, setup):
    u, r = setup
    W = weights(orc, CFG, zero_routed=True)
    out = fwd(orc, u, r, W, range(CFG.T))
    # a different routing (any experts, any gates) changes nothing
    idx2 = (r["idx"] + 3) % CFG.E
    gate2 = np.full_like(r["gate"], 0.5)
    out2 = orc.layer_forward(bits(u), idx2, gate2, W, CFG.d, CFG.E, CFG.K, CFG.S, CFG.I, range(CFG.T))
    assert np.array_equal(out, out2)
    qa, sa = orc.quant_1x128(bits(u))
    ysh = library_ffn(qa, sa, W, CFG.E).numpy()
    delta = out.astype(np.float64) - u.float().double().numpy()
    assert np.abs(delta).max() > 0.05
    assert np.linalg.norm(delta - ysh) / np.linalg.norm(ysh) < 2e-3


def test_ffn_matches_library_chain(orc):
    W = weights(orc, CFG)
    u = wl.tokens(CFG)
    qa, sa = orc.quant_1x128(bits(u))
    for g in (0, 5, CFG.E):
        y = orc.expert_ffn(qa, sa, *W.gate[g], *W.up[g], *W.down[g])
        ref = library_ffn(qa, sa, W, g).numpy()
        assert np.linalg.norm(y - ref) / np.linalg.norm(ref) < 2e-3
        assert np.abs(y - ref).max() < 2e-2


def test_single_expert_layer_is_the_ffn(orc):
    cfg = CFG.with_(K=1, S=0)
    u = wl.tokens(cfg)
    W = weights(orc, cfg)
    r = orc.route(bits(u), wl.centroids(cfg).numpy(), wl.bias(cfg).numpy(), 1)
    assert np.all(r["gate"] == 1.0)
    out = fwd(orc, u, r, W, range(cfg.T), cfg)
    qa, sa = orc.quant_1x128(bits(u))
    ref = u.float().double().numpy().copy()
    for t in range(cfg.T):
        ref[t] += library_ffn(qa[t:t + 1], sa[t:t + 1], W, int(r["idx"][t, 0])).numpy()[0]
    delta, dref = out - u.float().numpy(), ref - u.float().double().numpy()
    assert np.linalg.norm(delta - dref) / np.linalg.norm(dref) < 2e-3


def test_gates_weight_the_routed_outputs(orc, setup):
    u, r = setup
    W = weights(orc, CFG)
    toks = [0, 7, 39]
    base = fwd(orc, u, r, W, toks)
    # doubling one gate adds that expert's output once more
    gate2 = r["gate"].copy()
    gate2[7, 1] *= 2
    out = orc.layer_forward(bits(u), r["idx"], gate2, W, CFG.d, CFG.E, CFG.K, CFG.S, CFG.I, toks)
    qa, sa = orc.quant_1x128(bits(u[7:8]))
    y = orc.expert_ffn(qa, sa, *W.gate[r["idx"][7, 1]], *W.up[r["idx"][7, 1]], *W.down[r["idx"][7, 1]])
    extra = out[1].astype(np.float64) - base[1]
    assert np.allclose(extra, r["gate"][7, 1] * y[0], atol=1e-5)
    assert np.array_equal(out[[0, 2]], base[[0, 2]])


def test_tokens_are_independent(orc, setup):
    u, r = setup
    W = weights(orc, CFG)
    a = fwd(orc, u, r, W, [3, 4, 5])
    b = fwd(orc, u, r, W, [5, 3])
    assert np.array_equal(a[2], b[0]) and np.array_equal(a[0], b[1])
