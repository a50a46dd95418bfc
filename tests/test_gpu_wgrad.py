"""GPU parity of the weight gradients (reading R16) against the oracle: the
128x1 re-quantisation (bit-exact), the token-contracted GEMM (bit-exact on
small integers, float32-close on random codes, zeros for empty groups), and
the layer's moe_backward_wgrad after a forward and input gradient."""
import numpy as np
import pytest
import torch

from fine_grained_fp8_bias_b300 import workloads as wl
from tests.helpers import bits, oracle_weights, rel_fro

pytestmark = pytest.mark.gpu

DW_REL = 5e-3      # relative Frobenius error of each weight gradient of a group


@pytest.fixture(scope="module")
def L():
    from fine_grained_fp8_bias_b300 import lib
    return lib


# ragged groups: empty ones, one row, a block boundary, a ragged tail
SIZES = [0, 1, 127, 128, 129, 0, 300, 64, 0, 256, 37]


def _offsets(sizes):
    return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)


def _pb(sizes):
    return np.concatenate([[0], np.cumsum([(m + 127) // 128 for m in sizes])]).astype(np.int64)


def _codes(rng, shape):
    c = rng.integers(0, 254, size=shape, dtype=np.int64)
    return np.where(c >= 0x7F, c + 1, c).astype(np.uint8)       # no NaN codes (0x7F, 0xFF)


def test_requant_128x1_bit_exact(L, orc):
    rng = np.random.default_rng(21)
    go = _offsets(SIZES)
    M, C = int(go[-1]), 384
    q = _codes(rng, (M, C))
    s = (rng.uniform(0.5, 2.0, size=(M, C // 128)) * 2.0 ** rng.integers(-20, 10, size=(M, 1))).astype(np.float32)
    q[5:9] = 0                                                   # an all-zero stretch of rows
    qt, st = L.moe_requant_128x1(torch.from_numpy(q).cuda(), torch.from_numpy(s.T.copy()).cuda(),
                                 torch.from_numpy(go).cuda())
    torch.cuda.synchronize()
    qt, st = qt.cpu().numpy(), st.cpu().numpy()
    pb = _pb(SIZES)
    assert qt.shape[1] == L.moe_wgrad_ld(M, len(SIZES)) and qt.shape[1] >= 128 * pb[-1]
    for g, m in enumerate(SIZES):
        if m == 0:
            continue
        rq, rs = orc.requant_128x1(q[go[g]:go[g + 1]], s[go[g]:go[g + 1]])
        cols = slice(128 * pb[g], 128 * pb[g + 1])
        assert np.array_equal(qt[:, cols], rq), f"group {g}"
        assert np.array_equal(st[pb[g]:pb[g + 1]].T, rs), f"group {g}"


def test_requant_128x1_many_quotients(L, orc):
    # 4 M quotients over scales spanning 2^-90 .. 2^20: the division-free
    # quotient must match the oracle's IEEE division everywhere
    rng = np.random.default_rng(31)
    sizes = [1000, 1, 2047, 129, 823]
    go = _offsets(sizes)
    M, C = int(go[-1]), 1024
    q = _codes(rng, (M, C))
    s = (rng.uniform(1.0, 2.0, size=(M, C // 128)) *
         2.0 ** rng.integers(-90, 20, size=(M, C // 128))).astype(np.float32)
    qt, st = L.moe_requant_128x1(torch.from_numpy(q).cuda(), torch.from_numpy(s.T.copy()).cuda(),
                                 torch.from_numpy(go).cuda())
    torch.cuda.synchronize()
    qt, st = qt.cpu().numpy(), st.cpu().numpy()
    pb = _pb(sizes)
    for g in range(len(sizes)):
        rq, rs = orc.requant_128x1(q[go[g]:go[g + 1]], s[go[g]:go[g + 1]])
        cols = slice(128 * pb[g], 128 * pb[g + 1])
        assert np.array_equal(qt[:, cols], rq), f"group {g}"
        assert np.array_equal(st[pb[g]:pb[g + 1]].T, rs), f"group {g}"


def _wgrad_case(rng, integers, orc):
    go = _offsets(SIZES)
    G = len(SIZES)
    M = int(go[-1])
    ld = int(_pb(SIZES)[-1]) * 128 + 256          # more room than needed
    Na, Nb, split = 384, 640, 256                 # a half column tile; two output blocks
    if integers:
        def codes(shape):
            return orc.e4m3_encode(rng.integers(-8, 9, size=shape).astype(np.float32))
        sa = (2.0 ** rng.integers(-2, 3, size=(ld // 128, Na))).astype(np.float32)
        sb = (2.0 ** rng.integers(-2, 3, size=(ld // 128, Nb))).astype(np.float32)
    else:
        codes = lambda shape: _codes(rng, shape)
        sa = rng.uniform(0.001, 0.01, size=(ld // 128, Na)).astype(np.float32)
        sb = rng.uniform(0.001, 0.01, size=(ld // 128, Nb)).astype(np.float32)
    At, Bt = codes((Na, ld)), codes((Nb, ld))
    return go, G, M, ld, Na, Nb, split, At, Bt, sa, sb


@pytest.mark.parametrize("integers", [True, False])
def test_wgrad_gemm(L, orc, integers):
    rng = np.random.default_rng(22 + integers)
    go, G, M, ld, Na, Nb, split, At, Bt, sa, sb = _wgrad_case(rng, integers, orc)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    o0, o1 = L.moe_wgrad_gemm_fp8(torch.from_numpy(At).cuda(), torch.from_numpy(sa).cuda(),
                                  torch.from_numpy(Bt).cuda(), torch.from_numpy(sb).cuda(),
                                  torch.from_numpy(go).cuda(), split=split, status=status)
    torch.cuda.synchronize()
    assert L.moe_check_device_status(status) == 0
    got = np.concatenate([o0.cpu().numpy(), o1.cpu().numpy()], axis=1)     # [G, Na, Nb]
    pb = _pb(SIZES)
    worst = 0.0
    for g, m in enumerate(SIZES):
        if m == 0:
            assert not np.any(got[g]), f"empty group {g} must get zeros"
            continue
        cols = slice(128 * pb[g], 128 * pb[g + 1])
        ref = orc.gemm_fp8_rowscaled(At[:, cols], sa[pb[g]:pb[g + 1]].T.copy(), Bt[:, cols],
                                     sb[pb[g]:pb[g + 1]].T.copy())
        if integers:
            assert np.array_equal(got[g], ref), f"group {g}"
        else:
            err = float(np.abs(got[g] - ref).max() / np.abs(ref).max())
            worst = max(worst, err)
    print(f"wgrad GEMM ({'integers' if integers else 'random'}): worst max-abs / max|ref| {worst:.3e}")
    assert worst <= 1e-5


# ------------------------------------------------------------ the layer
def _run(cfg, seed=6):
    from fine_grained_fp8_bias_b300.layer import MoELayer
    layer = MoELayer.from_config(cfg, "cuda")
    u = wl.tokens(cfg, "cuda")
    out = layer.forward(u)
    dh = wl.normal(wl.stream_key(seed, 89), (cfg.T, cfg.d), 1.0, "cuda").to(torch.bfloat16)
    layer.backward_dgrad(u, dh, out)
    dW = layer.backward_wgrad(cfg.T)
    torch.cuda.synchronize()
    assert layer.status() == 0 and layer.backward_status() == 0
    return layer, u, out, dh, dW


def _check_groups(orc, cfg, pick):
    """pick(counts) -> the groups to compare (counts: rows of each routed expert)."""
    layer, u, out, dh, dW = _run(cfg)
    gidx, ggate = out["idx"].cpu().numpy(), out["gate"].cpu().numpy()
    groups = pick(np.bincount(gidx.ravel(), minlength=cfg.E))
    W = oracle_weights(orc, cfg, groups)
    u_bits, dh_bits = bits(u.cpu()), bits(dh.cpu())
    for g in groups:
        # the oracle differentiates the forward the GPU ran (its routing and gates)
        ref = orc.layer_backward_wgrad(u_bits, gidx, ggate, (W.gate[g], W.up[g], W.down[g]), dh_bits,
                                       cfg.d, cfg.E, cfg.K, cfg.I, g)
        got = [t[g].cpu().numpy() for t in dW]
        rows = cfg.T if g >= cfg.E else int((gidx == g).sum())
        if rows == 0:
            assert all(not np.any(x) for x in got)
            print(f"{cfg.name} group {g}: no rows, zeros")
            continue
        errs = [rel_fro(a, b) for a, b in zip(got, ref)]
        print(f"{cfg.name} group {g} ({rows} rows): rel_fro gate {errs[0]:.3e} up {errs[1]:.3e} "
              f"down {errs[2]:.3e}")
        assert max(errs) <= DW_REL


def test_wgrad_tiny(orc):
    cfg = wl.TINY
    _check_groups(orc, cfg, lambda counts: list(range(cfg.E + cfg.S)))


def test_wgrad_ragged(orc):
    cfg = wl.LayerConfig("ragged", T=301, d=640, E=24, K=3, S=2, I=384, seed=23)
    # the fullest routed expert (more than one 128-row block), the emptiest, the shared ones
    _check_groups(orc, cfg, lambda c: sorted({int(np.argmax(c)), int(np.argmin(c)), 24, 25}))


def test_wgrad_v3_smallest_group(orc):
    # the routed expert with the fewest (non-zero) rows keeps the oracle's work small
    _check_groups(orc, wl.V3_PREFILL,
                  lambda c: [int(np.argmin(np.where(c > 0, c, 1 << 30)))])
