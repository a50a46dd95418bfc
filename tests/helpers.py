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


def routing_agreement(gpu_idx, gpu_gate, orc_r, gate_rtol=4e-6):
    """Selections must be identical on every token the oracle does not flag
    as a near tie; gates agree to float32 rounding there.  Returns the list of
    flagged tokens whose selection differs."""
    gi = np.asarray(gpu_idx)
    oi = orc_r["idx"]
    flagged = orc_r["tie"].astype(bool)
    diff = np.any(gi != oi, axis=1)
    assert not np.any(diff & ~flagged), f"unflagged routing mismatch at {np.flatnonzero(diff & ~flagged)[:10]}"
    same = ~diff
    g = np.asarray(gpu_gate)[same]
    o = orc_r["gate"][same]
    assert np.all(np.abs(g - o) <= gate_rtol * np.abs(o) + 1e-7)
    return np.flatnonzero(diff)
