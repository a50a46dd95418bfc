"""moe_route_noalloc: the router for callers that cannot allocate device memory.

It must route as the oracle does (same selections on every token the oracle
does not flag as a near tie, gates within float32 rounding), agree with
moe_route, and give identical results call after call, although its logits
and partial sums live in one fixed array of the library that every call
reuses.  The sizes cover each of its summation paths: one block per expert
(T <= 8), split-K partials added in a fixed order (T = 16, 256) and a single
split when the logits fill the array (T * E = 1048576).  This file is
collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from fine_grained_fp8_bias_b300 import workloads as wl
from tests.helpers import bits, routing_agreement

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
           "counts": torch.full((E,), 7, dtype=torch.int32, device="cuda")}
    rc = fn(u.data_ptr() if T else None, c.data_ptr(), b.data_ptr(), T, d, E, K,
            out["idx"].data_ptr() if T else None, out["gate"].data_ptr() if T else None,
            out["tie"].data_ptr() if T else None, out["counts"].data_ptr(),
            torch.cuda.current_stream().cuda_stream)
    assert rc == 0, L.lib().moe_status_string(rc)
    return out


def agree(a, b):
    # same selected set wherever neither call flags a near tie, gates matched by
    # expert (the order of two selected experts with equal scores to within
    # rounding may differ; the oracle comparison checks the order)
    ia, ib = a["idx"].cpu().numpy(), b["idx"].cpu().numpy()
    tie = (a["tie"].cpu().numpy() | b["tie"].cpu().numpy()).astype(bool)
    diff = np.any(np.sort(ia, 1) != np.sort(ib, 1), axis=1)
    assert not np.any(diff & ~tie)
    ga = np.take_along_axis(a["gate"].cpu().numpy(), np.argsort(ia, 1), 1)[~diff]
    gb = np.take_along_axis(b["gate"].cpu().numpy(), np.argsort(ib, 1), 1)[~diff]
    assert np.all(np.abs(ga - gb) <= 4e-6 * np.abs(gb) + 1e-7)
    if not diff.any():
        assert torch.equal(a["counts"], b["counts"])


CASES = [wl.V3_PREFILL, wl.V3_DECODE.with_(T=1), wl.V3_DECODE.with_(T=8),
         wl.V3_DECODE.with_(T=16), wl.V3_DECODE.with_(T=256), wl.TINY]
IDS = ["v3_prefill_T4096", "v3_decode_T1", "v3_decode_T8", "v3_decode_T16", "v3_decode_T256",
       "tiny"]


@pytest.mark.parametrize("cfg", CASES, ids=IDS)
def test_noalloc_router_matches_oracle_and_router_twice(cfg, orc):
    from fine_grained_fp8_bias_b300 import lib as L
    inp = wl.small_inputs(cfg, "cuda")
    ref = L.moe_route(inp["u"], inp["centroids"], inp["bias"], cfg.K)
    first = call_noalloc(L, inp["u"], inp["centroids"], inp["bias"], cfg.K)
    second = call_noalloc(L, inp["u"], inp["centroids"], inp["bias"], cfg.K)
    torch.cuda.synchronize()
    # the oracle routes the same bits
    r = orc.route(bits(inp["u"]), inp["centroids"].cpu().numpy(), inp["bias"].cpu().numpy(), cfg.K)
    gidx = first["idx"].cpu().numpy()
    bad = routing_agreement(gidx, first["gate"].cpu().numpy(), r, bias=inp["bias"].cpu().numpy())
    counts_o = r["counts"].copy()
    if len(bad):                   # flagged near ties: the oracle adopts the GPU's choice
        idx_o = r["idx"].copy()
        idx_o[bad] = gidx[bad]
        counts_o = np.bincount(idx_o.ravel(), minlength=cfg.E).astype(np.int32)
    assert np.array_equal(first["counts"].cpu().numpy(), counts_o)
    # and agrees with the workspace router
    agree(first, ref)
    # two calls in a row give identical results, although they share the array
    for k in ("idx", "gate", "tie", "counts"):
        assert torch.equal(first[k], second[k]), k


def test_noalloc_router_empty_batch_clears_counts():
    from fine_grained_fp8_bias_b300 import lib as L
    cfg = wl.TINY
    inp = wl.small_inputs(cfg, "cuda")
    u0 = inp["u"][:0]
    out = call_noalloc(L, u0, inp["centroids"], inp["bias"], cfg.K)
    torch.cuda.synchronize()
    assert torch.equal(out["counts"], torch.zeros(cfg.E, dtype=torch.int32, device="cuda"))


def test_noalloc_router_rejects_too_large():
    from fine_grained_fp8_bias_b300 import lib as L
    cfg = wl.V3_PREFILL.with_(T=4097)                 # T * E = 1048832 > 1048576
    u = torch.zeros((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    c = torch.zeros((cfg.E, cfg.d), dtype=torch.float32, device="cuda")
    b = torch.zeros((cfg.E,), dtype=torch.float32, device="cuda")
    with pytest.raises(L.MoeError):
        L.moe_route_noalloc(u, c, b, cfg.K)
