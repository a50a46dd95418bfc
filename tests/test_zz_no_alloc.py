"""moe_route_noalloc: the router for callers that cannot allocate device memory.

It must give what moe_route gives (same selections on every token that is
not a near tie, gates within float32 rounding), call after call, although
its logits live in one fixed array of the library that every call reuses.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from fine_grained_fp8_bias_b300 import workloads as wl

pytestmark = pytest.mark.gpu


def call_noalloc(L, u, c, b, K):
    T, d = u.shape
    E = c.shape[0]
    fn = L.lib().moe_route_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 4 + [ctypes.c_void_p] * 5
    out = {"idx": torch.full((T, K), -1, dtype=torch.int32, device="cuda"),
           "gate": torch.zeros((T, K), dtype=torch.float32, device="cuda"),
           "tie": torch.zeros((T,), dtype=torch.uint8, device="cuda"),
           "counts": torch.zeros((E,), dtype=torch.int32, device="cuda")}
    rc = fn(u.data_ptr(), c.data_ptr(), b.data_ptr(), T, d, E, K, out["idx"].data_ptr(),
            out["gate"].data_ptr(), out["tie"].data_ptr(), out["counts"].data_ptr(),
            torch.cuda.current_stream().cuda_stream)
    assert rc == 0, L.lib().moe_status_string(rc)
    return out


def agree(a, b):
    ia, ib = a["idx"].cpu().numpy(), b["idx"].cpu().numpy()
    tie = (a["tie"].cpu().numpy() | b["tie"].cpu().numpy()).astype(bool)
    diff = np.any(ia != ib, axis=1)
    assert not np.any(diff & ~tie)
    ga, gb = a["gate"].cpu().numpy()[~diff], b["gate"].cpu().numpy()[~diff]
    assert np.all(np.abs(ga - gb) <= 4e-6 * np.abs(gb) + 1e-7)
    if not diff.any():
        assert torch.equal(a["counts"], b["counts"])


@pytest.mark.parametrize("cfg", [wl.V3_PREFILL, wl.V3_DECODE.with_(T=16), wl.TINY],
                         ids=["v3_prefill_T4096", "v3_decode_T16", "tiny"])
def test_noalloc_router_matches_router_twice(cfg):
    from fine_grained_fp8_bias_b300 import lib as L
    inp = wl.small_inputs(cfg, "cuda")
    ref = L.moe_route(inp["u"], inp["centroids"], inp["bias"], cfg.K)
    for _ in range(2):
        got = call_noalloc(L, inp["u"], inp["centroids"], inp["bias"], cfg.K)
        torch.cuda.synchronize()
        agree(got, ref)


def test_noalloc_router_rejects_too_large():
    from fine_grained_fp8_bias_b300 import lib as L
    cfg = wl.V3_PREFILL.with_(T=4097)                 # T * E = 1048832 > 1048576
    u = torch.zeros((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    c = torch.zeros((cfg.E, cfg.d), dtype=torch.float32, device="cuda")
    b = torch.zeros((cfg.E,), dtype=torch.float32, device="cuda")
    with pytest.raises(L.MoeError):
        L.moe_route_noalloc(u, c, b, cfg.K)
