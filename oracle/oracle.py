"""numpy interface to the plain C oracle (oracle/moe_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg call this module.  The CUDA library and its
Python binding never import it.

Arrays are numpy; bfloat16 tensors travel as their uint16 bit patterns.
The oracle keeps its own natural layouts: activation scales are [rows, d/128]
(row-major), weight scales [N/128, K/128].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
CFLAGS = ["-O2", "-fno-fast-math", "-ffp-contract=off", "-Wall", "-shared", "-fPIC"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no GPU involved)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32 = ctypes.c_int
        _lib.orc_e4m3_decode.restype = ctypes.c_double
        _lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        _lib.orc_e4m3_encode.restype = ctypes.c_uint8
        _lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
        _lib.orc_e4m3_encode_array.argtypes = [P, ctypes.c_int64, P]
        _lib.orc_quant_1x128_f32.argtypes = [P, i32, i32, P, P]
        _lib.orc_quant_1x128_bf16.argtypes = [P, i32, i32, P, P]
        _lib.orc_quant_128x128.argtypes = [P, i32, i32, P, P]
        _lib.orc_gemm_fp8.argtypes = [P, P, i32, i32, P, P, i32, P]
        _lib.orc_expert_ffn.argtypes = [P, P, i32, i32, i32, P, P, P, P, P, P, P]
        _lib.orc_gate_up.argtypes = [P, P, i32, i32, i32, P, P, P, P, P, P]
        _lib.orc_route.argtypes = [P, P, P, i32, i32, i32, i32, P, P, P, P, P]
        _lib.orc_route_grouped.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, i32, P, P, P, P, P]
        _lib.orc_dispatch.restype = i32
        _lib.orc_dispatch.argtypes = [P, i32, i32, i32, P, P, P, P]
        _lib.orc_layer_forward.argtypes = [P, i32, i32, i32, i32, i32, i32, P, P,
                                           P, P, P, P, P, P, P, i32, P]
        _lib.orc_update_bias.argtypes = [P, i32, i32, i32, ctypes.c_float, P]
        _lib.orc_layer_backward_dgrad.argtypes = [P, i32, i32, i32, i32, i32, i32, P, P, P,
                                                  P, P, P, P, P, P, P, P, i32, P]
        _lib.orc_requant_128x1.argtypes = [P, P, i32, i32, P, P]
        _lib.orc_gemm_fp8_rowscaled.argtypes = [P, P, i32, i32, P, P, i32, P]
        _lib.orc_layer_backward_wgrad.argtypes = [P, i32, i32, i32, i32, i32, P, P, P, P, P, P,
                                                  P, P, P, i32, P, P, P]
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


# ---------------------------------------------------------------- codec
def e4m3_decode(codes) -> np.ndarray:
    codes = _c(codes, np.uint8)
    return np.array([lib().orc_e4m3_decode(int(c)) for c in codes.ravel()]).reshape(codes.shape)


def e4m3_encode(x) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().orc_e4m3_encode_array(_p(x), x.size, _p(out))
    return out


# ---------------------------------------------------------- quantisation
def quant_1x128(x) -> tuple[np.ndarray, np.ndarray]:
    """x: float32 [M, D] or bfloat16 bits (uint16) [M, D] -> (codes [M, D], scales [M, D/128])."""
    x = np.asarray(x)
    M, D = x.shape
    q = np.empty((M, D), np.uint8)
    s = np.empty((M, D // 128), np.float32)
    if x.dtype == np.uint16:
        x = _c(x, np.uint16)
        lib().orc_quant_1x128_bf16(_p(x), M, D, _p(q), _p(s))
    else:
        x = _c(x, np.float32)
        lib().orc_quant_1x128_f32(_p(x), M, D, _p(q), _p(s))
    return q, s


def quant_128x128(w) -> tuple[np.ndarray, np.ndarray]:
    """w float32 [R, C] -> (codes [R, C], scales [R/128, C/128])."""
    w = _c(w, np.float32)
    R, C = w.shape
    q = np.empty((R, C), np.uint8)
    s = np.empty((R // 128, C // 128), np.float32)
    lib().orc_quant_128x128(_p(w), R, C, _p(q), _p(s))
    return q, s


# ---------------------------------------------------------------- GEMM
def gemm_fp8(qa, sa, qw, sw) -> np.ndarray:
    """Block-scaled FP8 GEMM: qa [M, K] codes, sa [M, K/128]; qw [N, K], sw [N/128, K/128]."""
    qa, sa, qw, sw = _c(qa, np.uint8), _c(sa, np.float32), _c(qw, np.uint8), _c(sw, np.float32)
    M, K = qa.shape
    N = qw.shape[0]
    out = np.empty((M, N), np.float32)
    lib().orc_gemm_fp8(_p(qa), _p(sa), M, K, _p(qw), _p(sw), N, _p(out))
    return out


def gate_up(qa, sa, wg, sg, wu, su) -> tuple[np.ndarray, np.ndarray]:
    """h = SiLU(A Wg^T) * (A Wu^T) quantised 1x128 -> (codes [M, I], scales [M, I/128])."""
    qa, sa = _c(qa, np.uint8), _c(sa, np.float32)
    wg, wu, sg, su = _c(wg, np.uint8), _c(wu, np.uint8), _c(sg, np.float32), _c(su, np.float32)
    M, d = qa.shape
    I = wg.shape[0]
    qh = np.empty((M, I), np.uint8)
    sh = np.empty((M, I // 128), np.float32)
    lib().orc_gate_up(_p(qa), _p(sa), M, d, I, _p(wg), _p(sg), _p(wu), _p(su), _p(qh), _p(sh))
    return qh, sh


def expert_ffn(qa, sa, wg, sg, wu, su, wd, sd) -> np.ndarray:
    qa, sa = _c(qa, np.uint8), _c(sa, np.float32)
    wg, wu, wd = _c(wg, np.uint8), _c(wu, np.uint8), _c(wd, np.uint8)
    sg, su, sd = _c(sg, np.float32), _c(su, np.float32), _c(sd, np.float32)
    M, d = qa.shape
    I = wg.shape[0]
    y = np.empty((M, d), np.float32)
    lib().orc_expert_ffn(_p(qa), _p(sa), M, d, I, _p(wg), _p(sg), _p(wu), _p(su),
                         _p(wd), _p(sd), _p(y))
    return y


# -------------------------------------------------------------- routing
def route(u_bits, cent, bias, K: int) -> dict:
    """u_bits: bfloat16 bit patterns [T, d]; cent float32 [E, d]; bias float32 [E]."""
    u_bits, cent, bias = _c(u_bits, np.uint16), _c(cent, np.float32), _c(bias, np.float32)
    T, d = u_bits.shape
    E = cent.shape[0]
    idx = np.empty((T, K), np.int32)
    gate = np.empty((T, K), np.float32)
    tie = np.empty((T,), np.uint8)
    counts = np.empty((E,), np.int32)
    scores = np.empty((T, E), np.float32)
    lib().orc_route(_p(u_bits), _p(cent), _p(bias), T, d, E, K, _p(idx), _p(gate), _p(tie),
                    _p(counts), _p(scores))
    return {"idx": idx, "gate": gate, "tie": tie, "counts": counts, "scores": scores}


def dispatch(idx, E: int) -> dict:
    idx = _c(idx, np.int32)
    T, K = idx.shape
    counts = np.empty((E,), np.int32)
    offsets = np.empty((E + 1,), np.int32)
    perm = np.empty((T * K,), np.int32)
    inv = np.empty((T, K), np.int32)
    rc = lib().orc_dispatch(_p(idx), T, K, E, _p(counts), _p(offsets), _p(perm), _p(inv))
    if rc != 0:
        raise ValueError("expert index out of range")
    return {"counts": counts, "offsets": offsets, "perm_token": perm, "inv_row": inv}


# ---------------------------------------------------------------- layer
class Weights:
    """Quantised expert weights per group (routed 0..E-1, shared E..E+S-1).

    Each entry is (codes, scales) for gate, up and down, or None for a routed
    expert that the evaluated tokens never select.
    """

    def __init__(self, G: int):
        self.G = G
        self.gate: list = [None] * G
        self.up: list = [None] * G
        self.down: list = [None] * G

    def set(self, g: int, gate, up, down):
        self.gate[g] = tuple(_c(a, t) for a, t in zip(gate, (np.uint8, np.float32)))
        self.up[g] = tuple(_c(a, t) for a, t in zip(up, (np.uint8, np.float32)))
        self.down[g] = tuple(_c(a, t) for a, t in zip(down, (np.uint8, np.float32)))


def layer_forward(u_bits, idx, gate, W: Weights, d: int, E: int, K: int, S: int, I: int,
                  tokens: Sequence[int]) -> np.ndarray:
    """h'_t for the listed tokens -> float32 [len(tokens), d]."""
    u_bits = _c(u_bits, np.uint16)
    idx, gate = _c(idx, np.int32), _c(gate, np.float32)
    T = u_bits.shape[0]
    tok = _c(tokens, np.int32)
    G = E + S
    for t in tok:
        for g in list(idx[t]) + list(range(E, G)):
            if W.gate[g] is None:
                raise ValueError(f"weights of group {g} are needed for token {t}")

    def ptrs(lst, j):
        arr = (ctypes.c_void_p * G)()
        for g in range(G):
            arr[g] = lst[g][j].ctypes.data if lst[g] is not None else None
        return arr

    out = np.empty((len(tok), d), np.float32)
    lib().orc_layer_forward(_p(u_bits), T, d, E, K, S, I, _p(idx), _p(gate),
                            ptrs(W.gate, 0), ptrs(W.gate, 1), ptrs(W.up, 0), ptrs(W.up, 1),
                            ptrs(W.down, 0), ptrs(W.down, 1), _p(tok), len(tok), _p(out))
    return out


def route_grouped(u_bits, cent, bias, K: int, n_groups: int, topk_groups: int,
                  group_topk: int) -> dict:
    """Group-limited routing (reading R14): keep the topk_groups groups of
    E / n_groups experts with the largest sums of their group_topk best biased
    scores, then top-K among the kept groups' experts."""
    u_bits, cent, bias = _c(u_bits, np.uint16), _c(cent, np.float32), _c(bias, np.float32)
    T, d = u_bits.shape
    E = cent.shape[0]
    if E % n_groups or not (1 <= topk_groups <= n_groups) or not (1 <= group_topk <= E // n_groups) \
            or K > topk_groups * (E // n_groups):
        raise ValueError("bad group configuration")
    idx = np.empty((T, K), np.int32)
    gate = np.empty((T, K), np.float32)
    tie = np.empty((T,), np.uint8)
    counts = np.empty((E,), np.int32)
    scores = np.empty((T, E), np.float32)
    lib().orc_route_grouped(_p(u_bits), _p(cent), _p(bias), T, d, E, K, n_groups, topk_groups,
                            group_topk, _p(idx), _p(gate), _p(tie), _p(counts), _p(scores))
    return {"idx": idx, "gate": gate, "tie": tie, "counts": counts, "scores": scores}


def layer_backward_dgrad(u_bits, idx, gate, W: Weights, cent, dh_bits, d: int, E: int, K: int,
                         S: int, I: int, tokens: Sequence[int]) -> np.ndarray:
    """du for the listed tokens (reading R15) -> float32 [len(tokens), d].
    dh_bits: bfloat16 bit patterns [T, d] of the upstream gradient of h'."""
    u_bits, dh_bits = _c(u_bits, np.uint16), _c(dh_bits, np.uint16)
    idx, gate, cent = _c(idx, np.int32), _c(gate, np.float32), _c(cent, np.float32)
    T = u_bits.shape[0]
    tok = _c(tokens, np.int32)
    G = E + S
    for t in tok:
        for g in list(idx[t]) + list(range(E, G)):
            if W.gate[g] is None:
                raise ValueError(f"weights of group {g} are needed for token {t}")

    def ptrs(lst, j):
        arr = (ctypes.c_void_p * G)()
        for g in range(G):
            arr[g] = lst[g][j].ctypes.data if lst[g] is not None else None
        return arr
    out = np.empty((len(tok), d), np.float32)
    lib().orc_layer_backward_dgrad(_p(u_bits), T, d, E, K, S, I, _p(cent), _p(idx), _p(gate),
                                   ptrs(W.gate, 0), ptrs(W.gate, 1), ptrs(W.up, 0), ptrs(W.up, 1),
                                   ptrs(W.down, 0), ptrs(W.down, 1), _p(dh_bits), _p(tok),
                                   len(tok), _p(out))
    return out


def requant_128x1(q, s) -> tuple[np.ndarray, np.ndarray]:
    """Reading R16: codes q [M, C] with 1x128 scales s [M, C/128] ->
    (codes [C, Mp], scales [C, Mp/128]) in 128x1 tiles, Mp = M rounded up to 128."""
    q, s = _c(q, np.uint8), _c(s, np.float32)
    M, C = q.shape
    nb = (M + 127) // 128
    qt = np.empty((C, nb * 128), np.uint8)
    st = np.empty((C, nb), np.float32)
    lib().orc_requant_128x1(_p(q), _p(s), M, C, _p(qt), _p(st))
    return qt, st


def gemm_fp8_rowscaled(qa, sa, qb, sb) -> np.ndarray:
    """Token-contracted FP8 GEMM of reading R16: qa [Na, K], sa [Na, K/128];
    qb [Nb, K], sb [Nb, K/128] -> float32 [Na, Nb]."""
    qa, sa, qb, sb = _c(qa, np.uint8), _c(sa, np.float32), _c(qb, np.uint8), _c(sb, np.float32)
    Na, K = qa.shape
    Nb = qb.shape[0]
    assert qb.shape[1] == K and sa.shape == (Na, K // 128) and sb.shape == (Nb, K // 128)
    out = np.empty((Na, Nb), np.float32)
    lib().orc_gemm_fp8_rowscaled(_p(qa), _p(sa), Na, K, _p(qb), _p(sb), Nb, _p(out))
    return out


def layer_backward_wgrad(u_bits, idx, gate, w_group, dh_bits, d: int, E: int, K: int, I: int,
                         g: int) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Reading R16: (dW_gate [I, d], dW_up [I, d], dW_down [d, I]) float32 of
    group g.  w_group = ((wg, sg), (wu, su), (wd, sd)) of that group."""
    u_bits, dh_bits = _c(u_bits, np.uint16), _c(dh_bits, np.uint16)
    idx, gate = _c(idx, np.int32), _c(gate, np.float32)
    (wg, sg), (wu, su), (wd, sd) = w_group
    wg, wu, wd = _c(wg, np.uint8), _c(wu, np.uint8), _c(wd, np.uint8)
    sg, su, sd = _c(sg, np.float32), _c(su, np.float32), _c(sd, np.float32)
    T = u_bits.shape[0]
    dWg = np.empty((I, d), np.float32)
    dWu = np.empty((I, d), np.float32)
    dWd = np.empty((d, I), np.float32)
    lib().orc_layer_backward_wgrad(_p(u_bits), T, d, E, K, I, _p(idx), _p(gate), _p(wg), _p(sg),
                                   _p(wu), _p(su), _p(wd), _p(sd), _p(dh_bits), g, _p(dWg),
                                   _p(dWu), _p(dWd))
    return dWg, dWu, dWd


def update_bias(counts, bias, T: int, K: int, gamma: float) -> np.ndarray:
    counts = _c(counts, np.int32)
    b = _c(bias, np.float32).copy()
    lib().orc_update_bias(_p(counts), counts.shape[0], T, K, gamma, _p(b))
    return b


# ------------------------------------------------------------ helpers
def bf16_bits(t) -> np.ndarray:
    """uint16 bit patterns of a torch bfloat16 tensor (no arithmetic)."""
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def quantised_weights(cfg, groups, weight_fn) -> Weights:
    """Oracle-quantised weights for the listed groups.

    weight_fn(which, g) returns the float32 master weight (numpy or torch, CPU).
    """
    W = Weights(cfg.E + cfg.S)
    for g in groups:
        mats = []
        for which in ("gate", "up", "down"):
            w = weight_fn(which, g)
            w = w.numpy() if hasattr(w, "numpy") else w
            mats.append(quant_128x128(w))
        W.set(g, *mats)
    return W
