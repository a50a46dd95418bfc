"""Shared helpers of the GPU parity tests: build the same layer for the CUDA
library and for the oracle from the seeded generator, and compare results."""
from __future__ import annotations

import numpy as np
import torch

from fine_grained_fp8_bias_b300 import workloads as wl

# Layer-output tolerance (the one the layer's FP8 specification states):
# relative Frobenius error <= 2e-3 and max abs error <= 2e-2 against the
# oracle's emulation of the same quantisation with FP32 promotion.
REL_FRO = 2e-3
MAX_ABS = 2e-2


def bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bfloat16 tensor."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def master(cfg, which, g, gen_device="cuda") -> np.ndarray:
    """Float32 master weight from the generator (its CUDA path when available: the
    generator gives bit-identical values on both devices, see test_gpu_generator)."""
    dev = gen_device if torch.cuda.is_available() else "cpu"
    return wl.master_weight(cfg, which, g, dev).cpu().numpy()


def oracle_weights(orc, cfg, groups):
    return orc.quantised_weights(cfg, sorted(set(int(g) for g in groups)),
                                 lambda which, g: master(cfg, which, g))


def rel_fro(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def routing_agreement(gpu_idx, gpu_gate, orc_r, gate_rtol=4e-6, bias=None):
    """The selected SET of experts must be identical on every token the oracle
    does not flag as a near tie at the K/K+1 boundary, with gates that agree to
    float32 rounding (matched by expert).  Within a selection the order is by
    descending biased score z = s + b; two selected experts whose oracle z
    differ by less than 1e-6 may come in either order (their z are equal to
    within the computation's rounding), every other pair must keep the
    oracle's order (checked when `bias` is given; without it the order must be
    identical).  Returns the flagged tokens whose selected set differs."""
    gi = np.asarray(gpu_idx)
    oi = orc_r["idx"]
    flagged = orc_r["tie"].astype(bool)
    set_diff = np.any(np.sort(gi, axis=1) != np.sort(oi, axis=1), axis=1)
    bad_unflagged = np.flatnonzero(set_diff & ~flagged)
    if len(bad_unflagged):
        t = int(bad_unflagged[0])
        msg = f"unflagged routing mismatch at {bad_unflagged[:10]}: token {t} gpu {gi[t]} oracle {oi[t]}"
        if bias is not None and "scores" in orc_r:
            z = (orc_r["scores"][t] + np.asarray(bias, np.float32)).astype(np.float32)
            order = np.argsort(-z, kind="stable")
            K = oi.shape[1]
            msg += f"; oracle z of the best {K + 2}: {[(int(e), float(z[e])) for e in order[:K + 2]]}"
        raise AssertionError(msg)
    same = ~set_diff
    # gates matched by expert
    gs = np.take_along_axis(np.asarray(gpu_gate), np.argsort(gi, axis=1), axis=1)[same]
    os_ = np.take_along_axis(orc_r["gate"], np.argsort(oi, axis=1), axis=1)[same]
    assert np.all(np.abs(gs - os_) <= gate_rtol * np.abs(os_) + 1e-7)
    # order within the selection
    order_diff = np.any(gi != oi, axis=1) & same
    if order_diff.any():
        if bias is None or "scores" not in orc_r:
            raise AssertionError(f"selection order differs at {np.flatnonzero(order_diff)[:10]}")
        for t in np.flatnonzero(order_diff):
            z = (orc_r["scores"][t] + np.asarray(bias, np.float32)).astype(np.float32)
            zg = z[gi[t]]
            assert np.all(zg[:-1] - zg[1:] > -1e-6), (t, gi[t], oi[t], zg)
        print(f"routing: {int(order_diff.sum())} tokens order two selected experts whose "
              f"biased scores differ by < 1e-6 the other way")
    return np.flatnonzero(set_diff)


# ------------------------------------------------------------ threaded oracle
# The oracle is single-threaded C; ctypes releases the GIL while it runs, so
# independent tokens (routing, layer outputs) and independent weight matrices
# (quantisation) are spread over a thread pool.  Nothing here changes what the
# oracle computes: each call is one of its functions on a slice of the input.
import os
from concurrent.futures import ThreadPoolExecutor

THREADS = max(1, min(os.cpu_count() or 1, 64))


def _pool():
    return ThreadPoolExecutor(max_workers=THREADS)


def route_threaded(orc, u_bits, cent, bias, K, chunk=512):
    """orc.route over token chunks; counts are the sum of the chunks' counts."""
    u_bits = np.ascontiguousarray(u_bits)
    T = u_bits.shape[0]
    starts = list(range(0, T, chunk))
    with _pool() as ex:
        parts = list(ex.map(lambda s: orc.route(u_bits[s:s + chunk], cent, bias, K), starts))
    out = {k: np.concatenate([p[k] for p in parts]) for k in ("idx", "gate", "tie", "scores")}
    out["counts"] = np.sum([p["counts"] for p in parts], axis=0).astype(np.int32)
    return out


def layer_forward_threaded(orc, u_bits, idx, gate, W, cfg, toks):
    toks = [int(t) for t in toks]
    n = max(1, (len(toks) + THREADS - 1) // THREADS)
    chunks = [toks[i:i + n] for i in range(0, len(toks), n)]
    with _pool() as ex:
        parts = list(ex.map(lambda c: orc.layer_forward(u_bits, idx, gate, W, cfg.d, cfg.E, cfg.K,
                                                        cfg.S, cfg.I, c), chunks))
    return np.concatenate(parts) if parts else np.zeros((0, cfg.d), np.float32)


_W_CACHE: dict = {}


def oracle_weights_threaded(orc, cfg, groups):
    """Oracle-quantised weights of the listed groups, quantised in parallel.
    The master weights come from the seeded generator (on the GPU when there
    is one: it gives the same bits as on the CPU).  The quantised weights of
    the most recent weight seed are kept, so workloads that share a seed
    (V3 prefill and its skewed form) quantise each matrix once; a V3-sized
    set replaces the sets cached before it."""
    key = (cfg.seed, cfg.d, cfg.I, cfg.E, cfg.S)
    if key not in _W_CACHE:
        # keep small weight sets; a large one (V3: 11 GB of codes) evicts the others
        big = lambda k: k[1] * k[2] * (k[3] + k[4]) * 3 > (1 << 30)
        for k in [k for k in _W_CACHE if big(k) or big(key)]:
            del _W_CACHE[k]
        _W_CACHE[key] = orc.Weights(cfg.E + cfg.S)
    W = _W_CACHE[key]
    todo = [int(g) for g in sorted(set(int(g) for g in groups)) if W.gate[int(g)] is None]

    def one(job):
        which, g, w = job
        return which, g, orc.quant_128x128(w)

    # generate a batch of masters on the device, quantise them on the host threads
    batch = max(THREADS, 8)
    for i in range(0, len(todo), batch):
        jobs = [(which, g, master(cfg, which, g)) for g in todo[i:i + batch]
                for which in ("gate", "up", "down")]
        with _pool() as ex:
            res = list(ex.map(one, jobs))
        mats = {(which, g): qs for which, g, qs in res}
        for g in todo[i:i + batch]:
            W.set(g, mats[("gate", g)], mats[("up", g)], mats[("down", g)])
    return W


def tile_covering_tokens(r_idx, cfg, n_groups=64, total=256, seed=0):
    """Tokens whose dispatch rows cover the grouped GEMMs' tiles: one token in
    every 128-row M tile of the shared groups (they hold every token in order),
    and for n_groups routed experts spread over [0, E) plus the largest and the
    smallest non-empty one, the expert's first row, its last row and the first
    row of its last (ragged) M tile; then random tokens up to `total`."""
    T, E = cfg.T, cfg.E
    toks = {0, T - 1}
    for j in range((T + 127) // 128):
        toks.add(min(T - 1, 128 * j + (37 * j) % 128))
    members = [[] for _ in range(E)]
    for t in range(T):
        for e in r_idx[t]:
            members[int(e)].append(t)
    counts = np.array([len(m) for m in members])
    nonempty = np.flatnonzero(counts > 0)
    pick = set(int(e) for e in np.linspace(0, E - 1, n_groups).round().astype(int) if counts[e] > 0)
    pick.add(int(nonempty[np.argmax(counts[nonempty])]))
    pick.add(int(nonempty[np.argmin(counts[nonempty])]))
    for e in pick:
        m = members[e]                       # ascending token order = row order
        toks.update((m[0], m[-1], m[128 * ((len(m) - 1) // 128)]))
    rng = np.random.default_rng(seed)
    rest = [t for t in range(T) if t not in toks]
    need = max(0, total - len(toks))
    toks.update(int(t) for t in rng.choice(rest, size=min(need, len(rest)), replace=False))
    return np.array(sorted(toks), np.int64), sorted(pick)
