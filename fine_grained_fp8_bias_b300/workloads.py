"""Seeded synthetic workloads for the DeepSeekMoE FP8 layer.

This module only draws numbers. It holds none of the layer's arithmetic (no
routing, no quantisation, no GEMM): the tests hand its tensors to both the
CUDA library and the CPU oracle, and the benchmark uses it to fill device
memory.

Every tensor is produced by one counter-based generator written with exact
integer tensor operations, so the same call gives bit-identical values on
the CPU and on a CUDA device:

* ``lowbias32`` (Chris Wellons' 32-bit integer hash: xor-shift 16, multiply
  by 0x7feb352d, xor-shift 15, multiply by 0x846ca68b, xor-shift 16) mixes a
  per-tensor key with the element counter.  Multiplications are split into
  16-bit halves so that no intermediate leaves the int64 range.
* A "normal" draw is the Irwin-Hall sum of four 16-bit uniforms, centred and
  scaled to the requested standard deviation (the sum is an exact integer, so
  the only rounding is one IEEE float32 multiply, identical on both devices).
  It matches the mean and variance of N(0, std^2) and is bounded at about
  3.46 standard deviations.
* A uniform draw on (lo, hi) uses the top 24 bits of one hash word.

The shapes follow the five layer configurations of the DeepSeekMoE FP8
workload (tiny, mid, V3 prefill, V3 decode, V3 long prefill).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

_M32 = 0xFFFFFFFF
_IH_STD = math.sqrt((65536.0 * 65536.0 - 1.0) / 3.0)  # std of a sum of four U{0..65535}


def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2^32 for int64 tensors holding values in [0, 2^32)."""
    hi = ((x >> 16) * c) & 0xFFFF
    lo = (x & 0xFFFF) * c
    return ((hi << 16) + lo) & _M32


def _lowbias32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def _lowbias32_int(x: int) -> int:
    x &= _M32
    x ^= x >> 16
    x = (x * 0x7FEB352D) & _M32
    x ^= x >> 15
    x = (x * 0x846CA68B) & _M32
    x ^= x >> 16
    return x


def stream_key(seed: int, *ids: int) -> tuple[int, int]:
    """Two 32-bit keys that name one tensor: (seed, id0, id1, ...)."""
    k = _lowbias32_int(seed * 0x9E3779B9 + 0x1234567)
    for i in ids:
        k = _lowbias32_int(k ^ (i * 0x85EBCA6B + 0x27D4EB2F))
    k2 = _lowbias32_int(k ^ 0x68E31DA4)
    return k, k2


def _lowbias32_np(x: np.ndarray) -> np.ndarray:
    """lowbias32 on uint32 arrays (numpy wraps uint32 products mod 2^32)."""
    x = x ^ (x >> np.uint32(16))
    x = x * np.uint32(0x7FEB352D)
    x = x ^ (x >> np.uint32(15))
    x = x * np.uint32(0x846CA68B)
    x = x ^ (x >> np.uint32(16))
    return x


def _words(key: tuple[int, int], start: int, n: int, per: int, device) -> torch.Tensor:
    """Hash words for elements [start, start+n), `per` words each -> int64 [n, per].

    The CPU path uses numpy uint32 arithmetic, the CUDA path torch int64
    arithmetic reduced mod 2^32; both compute the same function."""
    if torch.device(device).type == "cpu":
        lo = start * per
        if lo + n * per > 1 << 32:
            raise ValueError("counter range beyond 2^32 elements")
        idx = np.arange(lo, lo + n * per, dtype=np.uint32)   # high counter word is 0
        x = _lowbias32_np(idx ^ np.uint32(key[0]))
        x = _lowbias32_np(x ^ np.uint32(key[1]))
        return torch.from_numpy(x.astype(np.int64)).view(n, per)
    idx = torch.arange(start * per, (start + n) * per, dtype=torch.int64, device=device)
    x = _lowbias32((idx & _M32) ^ key[0])
    x = _lowbias32(x ^ ((idx >> 32) * 0x9E3779B9 & _M32) ^ key[1])
    return x.view(n, per)


def normal(key, shape, std: float, device="cpu", start: int = 0) -> torch.Tensor:
    """Irwin-Hall(4) approximation of N(0, std^2), float32, bit-identical on any device."""
    n = math.prod(shape)
    w = _words(key, start, n, 2, device)
    s = (w[:, 0] & 0xFFFF) + (w[:, 0] >> 16) + (w[:, 1] & 0xFFFF) + (w[:, 1] >> 16)
    c = torch.tensor(std / _IH_STD, dtype=torch.float32)
    return ((s - 131070).to(torch.float32) * c.to(device)).view(shape)


def uniform(key, shape, lo: float, hi: float, device="cpu") -> torch.Tensor:
    """Uniform on [lo, hi) with 24-bit resolution, float32."""
    n = math.prod(shape)
    w = _words(key, 0, n, 1, device)[:, 0]
    c = torch.tensor((hi - lo) / 16777216.0, dtype=torch.float32, device=device)
    return ((w >> 8).to(torch.float32) * c + torch.tensor(lo, dtype=torch.float32, device=device)).view(shape)


def randint(key, shape, lo: int, hi: int, device="cpu") -> torch.Tensor:
    """Integers in [lo, hi) (slightly non-uniform for ranges far from powers of two)."""
    n = math.prod(shape)
    w = _words(key, 0, n, 1, device)[:, 0]
    return (lo + (w % (hi - lo))).view(shape)


# Tensor ids inside one configuration's key space.
ID_U, ID_CENT, ID_BIAS, ID_WGATE, ID_WUP, ID_WDOWN, ID_MIX, ID_HOT = range(8)


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    """One DeepSeekMoE layer workload.

    T tokens of hidden size d; E routed experts of which each token uses K;
    S shared experts; expert FFN intermediate size I (SiLU-gated: W_gate and
    W_up are [I, d], W_down is [d, I]).
    """
    name: str
    T: int
    d: int
    E: int
    K: int
    S: int
    I: int
    seed: int
    bias: str = "uniform"       # "uniform" (U(-0.05, 0.05)) or "zeros"
    tokens: str = "normal"      # "normal" (N(0,1)) or "mixture4" (4-component mixture)
    gamma: float = 1e-3
    hot_experts: int = 0        # decode skew: number of hot experts (0 = none)
    hot_alpha: float = 0.0      # decode skew: centroid shift along the calibration mean direction
    n_groups: int = 0           # group-limited routing: expert groups (0 = plain top-K)
    topk_groups: int = 0        # groups kept per token
    group_topk: int = 0         # best scores summed into a group's score

    @property
    def G(self) -> int:
        return self.E + self.S

    def with_(self, **kw) -> "LayerConfig":
        return dataclasses.replace(self, **kw)


TINY = LayerConfig("tiny", T=256, d=256, E=16, K=2, S=1, I=128, seed=0)
MID = LayerConfig("mid", T=4096, d=2048, E=64, K=6, S=2, I=1408, seed=1, bias="zeros")
V3_PREFILL = LayerConfig("v3_prefill", T=4096, d=7168, E=256, K=8, S=1, I=2048, seed=2)
# hot_alpha: the shift that gives the 16 hot experts 40% of the selections of
# the T = 256 batch under the oracle's routing (bisection by
# tests/golden/calibrate_decode_skew.py, recorded in tests/golden/decode_skew.json).
DECODE_HOT_ALPHA = 5.25
V3_DECODE = LayerConfig("v3_decode", T=256, d=7168, E=256, K=8, S=1, I=2048, seed=3,
                        hot_experts=16, hot_alpha=DECODE_HOT_ALPHA)
V3_LONG = LayerConfig("v3_long", T=32768, d=7168, E=256, K=8, S=1, I=2048, seed=4,
                      tokens="mixture4")

# The V3 prefill batch with node-limited routing: 8 groups of 32 experts (one
# per node), at most 4 groups per token, group score from its 2 best experts.
V3_GROUPED = V3_PREFILL.with_(name="v3_grouped", n_groups=8, topk_groups=4, group_topk=2)

# The V3 prefill batch with skewed expert popularity: 16 hot experts whose
# centroids lean towards the tokens' mean direction (as the decode workload).
V3_SKEW = V3_PREFILL.with_(name="v3_skew", hot_experts=16, hot_alpha=DECODE_HOT_ALPHA)

# Profiling-size slice of the V3 prefill batch: the same expert shapes and the
# same rows per expert (T*K/E = 128), 32 routed experts (1.45 GB of weights).
V3_SLICE = LayerConfig("v3_slice", T=512, d=7168, E=32, K=8, S=1, I=2048, seed=5)

CONFIGS = {c.name: c for c in (TINY, MID, V3_PREFILL, V3_DECODE, V3_LONG, V3_SLICE, V3_GROUPED,
                                V3_SKEW)}


def tokens(cfg: LayerConfig, device="cpu", step: int = 0) -> torch.Tensor:
    """Layer input u [T, d] in bfloat16 (round-to-nearest-even from the float32 draw)."""
    if cfg.tokens == "normal":
        x = normal(stream_key(cfg.seed, ID_U, step), (cfg.T, cfg.d), 1.0, device)
    elif cfg.tokens == "mixture4":
        mu = normal(stream_key(cfg.seed, ID_MIX), (4, cfg.d), 1.0, device)
        comp = randint(stream_key(cfg.seed, ID_MIX, 1, step), (cfg.T,), 0, 4, device)
        z = normal(stream_key(cfg.seed, ID_U, step), (cfg.T, cfg.d), 0.5, device)
        x = mu[comp] + z
    else:
        raise ValueError(cfg.tokens)
    return x.to(torch.bfloat16)


def centroids(cfg: LayerConfig, device="cpu") -> torch.Tensor:
    """Expert centroids e_i [E, d] float32, N(0, 1/d).

    For the skewed decode workload the first `hot_experts` centroids are
    shifted by hot_alpha along the unit mean direction of a 4096-token
    calibration draw of the same token distribution.
    """
    c = normal(stream_key(cfg.seed, ID_CENT), (cfg.E, cfg.d), 1.0 / math.sqrt(cfg.d), device)
    if cfg.hot_experts:
        # The direction is always computed on the CPU so that both devices agree bit for bit.
        cal = normal(stream_key(cfg.seed, ID_HOT), (4096, cfg.d), 1.0, "cpu")
        v = cal.to(torch.float64).mean(0)
        v = (v / v.norm()).to(torch.float32)
        shift = torch.tensor(cfg.hot_alpha, dtype=torch.float32) * v
        c[: cfg.hot_experts] += shift.to(device)
    return c


def bias(cfg: LayerConfig, device="cpu") -> torch.Tensor:
    if cfg.bias == "zeros":
        return torch.zeros(cfg.E, dtype=torch.float32, device=device)
    return uniform(stream_key(cfg.seed, ID_BIAS), (cfg.E,), -0.05, 0.05, device)


def master_weight(cfg: LayerConfig, which: str, g: int, device="cpu") -> torch.Tensor:
    """Float32 master weight of group g (routed 0..E-1, shared E..E+S-1), N(0, 1/d).

    which: "gate" / "up" ([I, d]) or "down" ([d, I]).
    """
    tid = {"gate": ID_WGATE, "up": ID_WUP, "down": ID_WDOWN}[which]
    shape = (cfg.I, cfg.d) if which in ("gate", "up") else (cfg.d, cfg.I)
    return normal(stream_key(cfg.seed, tid, g), shape, 1.0 / math.sqrt(cfg.d), device)


def small_inputs(cfg: LayerConfig, device="cpu", step: int = 0) -> dict:
    return {"u": tokens(cfg, device, step), "centroids": centroids(cfg, device),
            "bias": bias(cfg, device)}


def pinned_like(t: torch.Tensor) -> torch.Tensor:
    out = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    out.copy_(t)
    return out


def describe(cfg: LayerConfig) -> dict:
    return {"workload": cfg.name, "T": cfg.T, "d": cfg.d, "experts_routed": cfg.E,
            "top_k": cfg.K, "experts_shared": cfg.S, "intermediate": cfg.I, "seed": cfg.seed}


def check_config(cfg: LayerConfig, T: Optional[int] = None) -> None:
    T = cfg.T if T is None else T
    if cfg.d % 128 or cfg.I % 128:
        raise ValueError("d and I must be multiples of 128")
    if not (1 <= cfg.K <= cfg.E):
        raise ValueError("need 1 <= K <= E")
