"""GPU parity of the tcgen05 grouped FP8 GEMM against the oracle's block-scaled GEMM."""
import numpy as np
import pytest
import torch

from fine_grained_fp8_bias_b300 import workloads as wl
from tests.helpers import rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    from fine_grained_fp8_bias_b300 import lib
    return lib


def bf16_round(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).float().numpy()


def groups(sizes, extra_rows=0):
    go = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    return go, int(go[-1]) + extra_rows


def int_operands(orc, M, G, N, Kdim, seed, vmax=4):
    """Small-integer E4M3 codes with power-of-two scales: every slab partial and
    every promotion step is exact, so any correct datapath gives identical bits."""
    rng = np.random.default_rng(seed)
    qa = orc.e4m3_encode(rng.integers(-vmax, vmax + 1, (M, Kdim)).astype(np.float32))
    sa = np.exp2(rng.integers(-4, 3, (M, Kdim // 128))).astype(np.float32)
    qw = orc.e4m3_encode(rng.integers(-vmax, vmax + 1, (G, N, Kdim)).astype(np.float32))
    sw = np.exp2(rng.integers(-6, 1, (G, N // 128, Kdim // 128))).astype(np.float32)
    return qa, sa, qw, sw


def random_operands(orc, M, G, N, Kdim, seed):
    a = wl.normal(wl.stream_key(seed, 1), (M, Kdim), 1.0).to(torch.bfloat16)
    qa, sa = orc.quant_1x128(a.view(torch.int16).numpy().view(np.uint16))
    qw = np.empty((G, N, Kdim), np.uint8)
    sw = np.empty((G, N // 128, Kdim // 128), np.float32)
    for g in range(G):
        w = wl.normal(wl.stream_key(seed, 2, g), (N, Kdim), 1.0 / np.sqrt(Kdim)).numpy()
        qw[g], sw[g] = orc.quant_128x128(w)
    return qa, sa, qw, sw


def run_down(L, qa, sa, go, qw, sw, M_total, small=False, f32=False):
    dev = "cuda"
    out = torch.full((M_total, qw.shape[1]), 7.0, dtype=torch.float32 if f32 else torch.bfloat16,
                     device=dev)
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    fn = L.moe_grouped_gemm_fp8_small if small else L.moe_grouped_gemm_fp8
    fn(L.MOE_GEMM_DOWN_F32 if f32 else L.MOE_GEMM_DOWN, torch.from_numpy(qa).to(dev),
                           torch.from_numpy(np.ascontiguousarray(sa.T)).to(dev),
                           torch.from_numpy(go).to(dev), torch.from_numpy(qw).to(dev), None,
                           torch.from_numpy(sw).to(dev), None, out=out, status=status)
    assert L.moe_check_device_status(status) == 0
    return out.float().cpu().numpy()


def oracle_grouped(orc, qa, sa, go, qw, sw):
    ref = np.zeros((int(go[-1]), qw.shape[1]), np.float32)
    for g in range(len(go) - 1):
        r0, r1 = int(go[g]), int(go[g + 1])
        if r1 > r0:
            ref[r0:r1] = orc.gemm_fp8(qa[r0:r1], sa[r0:r1], qw[g], sw[g])
    return ref


@pytest.mark.parametrize("sizes,N,Kdim", [
    ([0, 5, 128, 129, 300, 0, 1], 512, 384),
    ([1], 256, 128),
    ([64, 200], 384, 256),          # N = 384: the second 256-wide tile is half empty
    ([260, 3, 0, 0, 77], 768, 1024),
])
@pytest.mark.parametrize("small", [False, True], ids=["large", "small"])
def test_down_exact_integer_bit_exact(L, orc, sizes, N, Kdim, small):
    go, M = groups(sizes, extra_rows=9)
    qa, sa, qw, sw = int_operands(orc, M, len(sizes), N, Kdim, seed=sum(sizes) + N)
    got = run_down(L, qa, sa, go, qw, sw, M, small)
    ref = oracle_grouped(orc, qa, sa, go, qw, sw)
    assert np.array_equal(got[: go[-1]], bf16_round(ref))
    assert np.all(got[go[-1]:] == 7.0)              # rows outside every group untouched


@pytest.mark.parametrize("sizes,N,Kdim", [([3, 190, 0, 64], 512, 512), ([400], 256, 2048),
                                          ([17, 1, 129], 384, 256)])
@pytest.mark.parametrize("small", [False, True], ids=["large", "small"])
def test_down_random(L, orc, sizes, N, Kdim, small):
    go, M = groups(sizes)
    qa, sa, qw, sw = random_operands(orc, M, len(sizes), N, Kdim, seed=N + Kdim)
    got = run_down(L, qa, sa, go, qw, sw, M, small)
    ref = oracle_grouped(orc, qa, sa, go, qw, sw)
    # float32 promotion agrees to a few ulps; the bf16 output rounding then
    # differs by at most one bf16 ulp where the float32 values straddle a tie
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
    assert np.all(np.abs(got - bf16_round(ref)) <= ulp + 1e-30)
    assert rel_fro(got, ref) < 4e-3


def run_gate_up(L, qa, sa, go, wg, sg, wu, su, M_total, small=False):
    dev = "cuda"
    N = wg.shape[1]
    out = torch.full((M_total, N), 0x55, dtype=torch.uint8, device=dev)
    scales = torch.full((N // 128, M_total), -1.0, dtype=torch.float32, device=dev)
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    fn = L.moe_grouped_gemm_fp8_small if small else L.moe_grouped_gemm_fp8
    fn(L.MOE_GEMM_GATE_UP_SILU_QUANT, T(qa), T(sa.T), T(go), T(wg), T(wu), T(sg), T(su), out=out,
       out_scales=scales, status=status)
    assert L.moe_check_device_status(status) == 0
    return out.cpu().numpy(), scales.cpu().numpy().T


@pytest.mark.parametrize("sizes,I,d", [([0, 5, 128, 129, 0, 1], 256, 384), ([300], 128, 1024),
                                       ([40, 90], 1408 // 128 * 128, 256)])
@pytest.mark.parametrize("small", [False, True], ids=["large", "small"])
def test_gate_up_against_oracle(L, orc, sizes, I, d, small):
    go, M = groups(sizes, extra_rows=5)
    G = len(sizes)
    qa, sa, wg, sg = random_operands(orc, M, G, I, d, seed=I + d)
    _, _, wu, su = random_operands(orc, M, G, I, d, seed=I + d + 1)
    qh, sh = run_gate_up(L, qa, sa, go, wg, sg, wu, su, M, small)
    dec = orc.e4m3_decode(np.arange(256, dtype=np.uint8))
    n = int(go[-1])
    ref_q = np.zeros((n, I), np.uint8)
    ref_s = np.zeros((n, I // 128), np.float32)
    for g in range(G):
        r0, r1 = int(go[g]), int(go[g + 1])
        if r1 > r0:
            ref_q[r0:r1], ref_s[r0:r1] = orc.gate_up(qa[r0:r1], sa[r0:r1], wg[g], sg[g], wu[g], su[g])
    # scales agree to float32 rounding of h; codes agree except where h sits on
    # an E4M3 rounding boundary, and then by one code step
    assert np.all(np.abs(sh[:n] - ref_s) <= 4e-7 * np.abs(ref_s))
    same = qh[:n] == ref_q
    assert same.mean() > 0.999
    assert np.all(np.abs(dec[qh[:n]][~same] - dec[ref_q][~same]) <=
                  np.abs(dec[ref_q][~same]) / 8 + 2.0 ** -9)
    hv = dec[qh[:n]] * np.repeat(sh[:n], 128, 1)
    hr = dec[ref_q] * np.repeat(ref_s, 128, 1)
    assert rel_fro(hv, hr) < 1e-3
    assert np.all(qh[n:] == 0x55) and np.all(sh[n:] == -1.0)


@pytest.mark.parametrize("small", [False, True], ids=["large", "small"])
def test_gate_up_exact_integer(L, orc, small):
    # exact G and U; only the SiLU evaluation (expf) may differ by float32 ulps
    sizes = [130, 7]
    go, M = groups(sizes)
    G, I, d = 2, 256, 256
    qa, sa, wg, sg = int_operands(orc, M, G, I, d, seed=5, vmax=2)
    _, _, wu, su = int_operands(orc, M, G, I, d, seed=6, vmax=2)
    qh, sh = run_gate_up(L, qa, sa, go, wg, sg, wu, su, M, small)
    for g in range(G):
        r0, r1 = int(go[g]), int(go[g + 1])
        rq, rs = orc.gate_up(qa[r0:r1], sa[r0:r1], wg[g], sg[g], wu[g], su[g])
        assert (qh[r0:r1] == rq).mean() > 0.999
        assert np.all(np.abs(sh[r0:r1] - rs) <= 4e-7 * np.abs(rs))


@pytest.mark.parametrize("small", [False, True], ids=["large", "small"])
def test_empty_groups_and_no_rows(L, orc, small):
    go = np.zeros(5, np.int32)
    qa, sa, qw, sw = int_operands(orc, 8, 4, 256, 128, seed=9)
    got = run_down(L, qa, sa, go, qw, sw, 8, small)
    assert np.all(got == 7.0)


@pytest.mark.parametrize("small", [False, True], ids=["large", "small"])
def test_many_groups_v3_shape(L, orc, small):
    # 257 groups (256 routed + 1 shared), d = 7168, I = 2048 down projection on
    # a few rows per group: exercises the tile schedule at full group count
    rng = np.random.default_rng(11)
    sizes = rng.integers(0, 3, 257)
    sizes[256] = 5
    go, M = groups(sizes)
    G, N, Kdim = 257, 256, 2048
    qa, sa, qw, sw = int_operands(orc, M, G, N, Kdim, seed=12, vmax=2)
    got = run_down(L, qa, sa, go, qw, sw, M, small)
    ref = oracle_grouped(orc, qa, sa, go, qw, sw)
    assert np.array_equal(got, bf16_round(ref))


# The small-group tiles cut a group's rows into chunks of 32 (MMA N = 16 or 32
# from boxes of 16 rows): ragged sizes around every chunk and box boundary.
SMALL_SIZES = [0, 1, 15, 16, 17, 31, 32, 33, 47, 64, 65, 100, 0, 2]


def test_small_down_chunk_edges_bit_exact(L, orc):
    go, M = groups(SMALL_SIZES, extra_rows=3)
    G, N, Kdim = len(SMALL_SIZES), 384, 512
    qa, sa, qw, sw = int_operands(orc, M, G, N, Kdim, seed=31)
    got = run_down(L, qa, sa, go, qw, sw, M, small=True)
    ref = oracle_grouped(orc, qa, sa, go, qw, sw)
    assert np.array_equal(got[: go[-1]], bf16_round(ref))
    assert np.all(got[go[-1]:] == 7.0)


def test_small_gate_up_chunk_edges(L, orc):
    go, M = groups(SMALL_SIZES, extra_rows=3)
    G, I, d = len(SMALL_SIZES), 256, 384
    qa, sa, wg, sg = random_operands(orc, M, G, I, d, seed=41)
    _, _, wu, su = random_operands(orc, M, G, I, d, seed=42)
    qh, sh = run_gate_up(L, qa, sa, go, wg, sg, wu, su, M, small=True)
    n = int(go[-1])
    dec = orc.e4m3_decode(np.arange(256, dtype=np.uint8))
    for g in range(G):
        r0, r1 = int(go[g]), int(go[g + 1])
        if r1 == r0:
            continue
        rq, rs = orc.gate_up(qa[r0:r1], sa[r0:r1], wg[g], sg[g], wu[g], su[g])
        assert np.all(np.abs(sh[r0:r1] - rs) <= 4e-7 * np.abs(rs)), g
        same = qh[r0:r1] == rq
        assert same.mean() > 0.99, g
        assert np.all(np.abs(dec[qh[r0:r1]][~same] - dec[rq][~same]) <= np.abs(dec[rq][~same]) / 8
                      + 2.0 ** -9)
    assert np.all(qh[n:] == 0x55) and np.all(sh[n:] == -1.0)


def test_small_and_large_tiles_agree_on_v3_decode_shapes(L, orc):
    # 9 groups of one row (a T = 1 decode step) and a T = 16 mix at d = 7168,
    # I = 2048: the two tile shapes run the same arithmetic
    for sizes in ([1] * 9, [16, 3, 1, 1, 2, 0, 5, 1, 16]):
        go, M = groups(sizes)
        G, N, Kdim = len(sizes), 256, 2048
        qa, sa, qw, sw = random_operands(orc, M, G, N, Kdim, seed=51 + M)
        a = run_down(L, qa, sa, go, qw, sw, M, small=False)
        b = run_down(L, qa, sa, go, qw, sw, M, small=True)
        ref = oracle_grouped(orc, qa, sa, go, qw, sw)
        assert rel_fro(b, ref) < 4e-3
        print(f"sizes {sizes}: small vs large tiles identical: {np.array_equal(a, b)}")


@pytest.mark.parametrize("small", [False, True], ids=["large", "small"])
@pytest.mark.parametrize("sizes,N,Kdim", [([0, 5, 128, 129, 300, 0, 1], 512, 384),
                                          ([1] * 9, 256, 2048), ([33, 0, 17], 384, 256)])
def test_down_f32_exact_integer_bit_exact(L, orc, sizes, N, Kdim, small):
    # the layer forward keeps y in float32: with exact operands it equals the
    # oracle's float32 result bit for bit
    go, M = groups(sizes, extra_rows=4)
    qa, sa, qw, sw = int_operands(orc, M, len(sizes), N, Kdim, seed=sum(sizes) + Kdim)
    got = run_down(L, qa, sa, go, qw, sw, M, small, f32=True)
    ref = oracle_grouped(orc, qa, sa, go, qw, sw)
    assert np.array_equal(got[: go[-1]], ref)
    assert np.all(got[go[-1]:] == 7.0)


@pytest.mark.parametrize("small", [False, True], ids=["large", "small"])
def test_down_f32_random(L, orc, small):
    sizes = [3, 190, 0, 64, 1]
    go, M = groups(sizes)
    qa, sa, qw, sw = random_operands(orc, M, len(sizes), 512, 1024, seed=77)
    got = run_down(L, qa, sa, go, qw, sw, M, small, f32=True)
    ref = oracle_grouped(orc, qa, sa, go, qw, sw)
    # promotion agrees to float32 rounding of the tensor core's in-slab sums
    scale = np.abs(ref).max()
    assert np.abs(got - ref).max() <= 1e-5 * scale
    assert rel_fro(got, ref) < 1e-5


@pytest.mark.parametrize("small", [False, True], ids=["large", "small"])
def test_down_split_precision_bit_exact(L, orc, small):
    # the layer's down projection: routed groups' rows in bf16, the last
    # (shared) groups' rows in float32 at row - f32_row0
    sizes = [5, 0, 130, 17, 1, 40, 40]          # 5 routed groups, then 2 shared groups of 40
    go, M = groups(sizes)
    G, N, Kdim = len(sizes), 384, 512
    qa, sa, qw, sw = int_operands(orc, M, G, N, Kdim, seed=91)
    ref = oracle_grouped(orc, qa, sa, go, qw, sw)
    r0 = int(go[5])
    dev = "cuda"
    y = torch.full((r0, N), 7.0, dtype=torch.bfloat16, device=dev)
    y32 = torch.full((M - r0, N), 7.0, dtype=torch.float32, device=dev)
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    L.moe_grouped_gemm_fp8_down(T(qa), T(sa.T), T(go), T(qw), T(sw), 5, r0, y, y32,
                                small_tiles=small, status=status)
    assert L.moe_check_device_status(status) == 0
    assert np.array_equal(y.float().cpu().numpy(), bf16_round(ref[:r0]))
    assert np.array_equal(y32.cpu().numpy(), ref[r0:])
