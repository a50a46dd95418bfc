"""ctypes binding of libmoefp8.so (include/moe_fp8.h).

Argument marshalling only: every function passes device pointers of torch
tensors to the C entry point of the same name and raises MoeError on a
non-zero status.  Every step of the layer runs in the library's CUDA
kernels; there is no CPU fallback, and importing this module on a machine
without the built library raises ImportError.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoefp8.so")

MOE_OK = 0
MOE_GEMM_GATE_UP_SILU_QUANT = 1
MOE_GEMM_DOWN = 2
MOE_GEMM_DOWN_F32 = 4

P = ctypes.c_void_p
I32 = ctypes.c_int


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = _lib.moe_status_string(code).decode() if _lib else str(code)
        if code == -4 and _lib:
            msg += f" (cudaError {_lib.moe_last_cuda_error()})"
        super().__init__(f"{where}: {msg} [{code}]")


class moe_layer_t(ctypes.Structure):
    _fields_ = [("d", I32), ("E", I32), ("K", I32), ("S", I32), ("I", I32),
                ("centroids", P), ("bias", P), ("w_gate", P), ("w_up", P), ("w_down", P),
                ("s_gate", P), ("s_up", P), ("s_down", P),
                ("n_groups", I32), ("topk_groups", I32), ("group_topk", I32)]


class moe_layer_bwd_t(ctypes.Structure):
    _fields_ = [("w_down_t", P), ("s_down_t", P), ("w_gu_t", P), ("s_gu_t", P)]


class moe_batch_buffers_t(ctypes.Structure):
    _fields_ = [("u", P), ("h", P), ("topk_idx", P), ("topk_gate", P), ("tie_flag", P),
                ("counts", P)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmoefp8.so is not built ({LIB_PATH}); run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_status_string.argtypes = [I32]
    lib.moe_last_cuda_error.restype = I32
    lib.moe_kernel_launches.restype = ctypes.c_uint64
    lib.moe_kernel_launches.argtypes = []
    lib.moe_set_pipeline_wait_limit.restype = ctypes.c_longlong
    lib.moe_set_pipeline_wait_limit.argtypes = [ctypes.c_longlong]
    lib.moe_set_pipeline_stall.restype = I32
    lib.moe_set_pipeline_stall.argtypes = [I32]
    lib.moe_last_cuda_error.argtypes = []
    lib.moe_workspace_size.restype = ctypes.c_size_t
    lib.moe_workspace_size.argtypes = [ctypes.POINTER(moe_layer_t), I32]
    lib.moe_route_workspace_size.restype = ctypes.c_size_t
    lib.moe_route_workspace_size.argtypes = [I32, I32, I32]
    lib.moe_backward_workspace_size.restype = ctypes.c_size_t
    lib.moe_backward_workspace_size.argtypes = [ctypes.POINTER(moe_layer_t), I32]
    lib.moe_wgrad_workspace_size.restype = ctypes.c_size_t
    lib.moe_wgrad_workspace_size.argtypes = [ctypes.POINTER(moe_layer_t), I32]
    # Every other entry point returns an int status.  Each one is called only
    # with these argument types: ctypes would otherwise pass Python ints as C
    # int and cut 64-bit pointers to 32 bits.
    sigs = {
        "moe_quant_1x128": [P, I32, P, I32, I32, P, P, I32, P, P],
        "moe_quant_128x128": [P, I32, I32, P, P, P],
        "moe_quant_1x128_dispatch": [P, I32, I32, P, I32, I32, P, P, I32, P, P],
        "moe_route": [P, P, P, I32, I32, I32, I32, P, P, P, P, P, ctypes.c_size_t, P],
        "moe_route_noalloc": [P, P, P, I32, I32, I32, I32, P, P, P, P, P],
        "moe_route_grouped": [P, P, P, I32, I32, I32, I32, I32, I32, I32, P, P, P, P, P,
                              ctypes.c_size_t, P],
        "moe_route_estimate_logits": [P, P, I32, I32, I32, P, P, P, ctypes.c_size_t, P],
        "moe_permute": [P, I32, I32, I32, I32, P, P, P, P, P, P, ctypes.c_size_t, P],
        "moe_grouped_gemm_fp8": [I32, P, P, I32, P, I32, P, P, P, P, I32, I32, P, P, P, P],
        "moe_grouped_gemm_fp8_small": [I32, P, P, I32, P, I32, P, P, P, P, I32, I32, P, P, P, P],
        "moe_grouped_gemm_fp8_down": [P, P, I32, P, I32, I32, I32, P, P, I32, I32, P, P, I32, P, P],
        "moe_combine": [P, P, P, P, P, I32, I32, I32, I32, P, P],
        "moe_forward": [ctypes.POINTER(moe_layer_t), P, I32, P, P, P, P, P, P, ctypes.c_size_t, P],
        "moe_update_bias": [P, I32, I32, I32, ctypes.c_float, P, P],
        "moe_prepare_backward_weights": [ctypes.POINTER(moe_layer_t), P, P, P, P, P],
        "moe_backward_dgrad": [ctypes.POINTER(moe_layer_t), ctypes.POINTER(moe_layer_bwd_t), P, P,
                               I32, P, P, P, P, ctypes.c_size_t, P, ctypes.c_size_t, P],
        "moe_forward_host": [ctypes.POINTER(moe_layer_t), I32, I32, P, P, ctypes.c_float,
                             ctypes.POINTER(moe_batch_buffers_t), P, ctypes.c_size_t, P, P, P],
        "moe_check_device_status": [P, P],
        "moe_forward_pipelined": [ctypes.POINTER(moe_layer_t), I32, I32,
                                  ctypes.POINTER(moe_batch_buffers_t), ctypes.c_float, P, P,
                                  ctypes.c_size_t, I32, P, P],
        "moe_wgrad_ld": [I32, I32],
        "moe_requant_128x1": [P, P, I32, I32, P, I32, P, P, I32, P, P],
        "moe_wgrad_gemm_fp8": [P, P, I32, P, P, I32, I32, P, I32, P, P, I32, P, P],
        "moe_backward_wgrad": [ctypes.POINTER(moe_layer_t), I32, P, P, P, P, ctypes.c_size_t, P,
                               ctypes.c_size_t, P, ctypes.c_size_t, P],
    }
    for name, args in sigs.items():
        fn = getattr(lib, name)
        fn.restype = I32
        fn.argtypes = args
    return lib


_lib: Optional[ctypes.CDLL] = None
_lib = _load()


def lib() -> ctypes.CDLL:
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return t.data_ptr()


def _dev(t: torch.Tensor, name: str):
    if t is not None and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(rc: int, where: str):
    if rc != MOE_OK:
        raise MoeError(rc, where)


def _bits(t: torch.Tensor, dtype) -> torch.Tensor:
    if t.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {t.dtype}")
    return t


def _router_inputs(u: torch.Tensor, centroids: torch.Tensor, bias: torch.Tensor):
    """Checks the router's inputs before their pointers reach a kernel:
    u bf16 [T, d], centroids float32 [E, d] and bias float32 [E], all
    contiguous on the same CUDA device.  Returns (T, d, E)."""
    _bits(u, torch.bfloat16)
    _bits(centroids, torch.float32)
    _bits(bias, torch.float32)
    for t, n in ((u, "u"), (centroids, "centroids"), (bias, "bias")):
        _dev(t, n)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
        if t.device != u.device:
            raise ValueError(f"{n} must be on {u.device}")
    if u.dim() != 2 or centroids.dim() != 2 or bias.dim() != 1:
        raise ValueError("need u [T, d], centroids [E, d], bias [E]")
    T, d = u.shape
    E = centroids.shape[0]
    if centroids.shape[1] != d or bias.shape[0] != E:
        raise ValueError(f"centroids {tuple(centroids.shape)} and bias {tuple(bias.shape)} "
                         f"do not match u {tuple(u.shape)}")
    return T, d, E


def set_pipeline_wait_limit(cycles: int) -> int:
    """Limit of the grouped GEMMs' pipeline waits in SM clock cycles for later
    launches (<= 0: the default, about 2 s); returns the previous limit."""
    return int(_lib.moe_set_pipeline_wait_limit(cycles))


def set_pipeline_stall(on: bool) -> int:
    """Test switch: grouped GEMMs launched afterwards issue no loads, so their
    pipeline waits run out (MOE_ERR_TIMEOUT); returns the previous setting."""
    return int(_lib.moe_set_pipeline_stall(1 if on else 0))


def kernel_launches() -> int:
    return int(_lib.moe_kernel_launches())


# ------------------------------------------------------------ entry points
def moe_quant_1x128(x: torch.Tensor, gather_rows: Optional[torch.Tensor] = None,
                    M: Optional[int] = None, q: Optional[torch.Tensor] = None,
                    scales: Optional[torch.Tensor] = None, scale_ld: Optional[int] = None,
                    status: Optional[torch.Tensor] = None, stream=None):
    """x bf16 [n_src, d] -> (q uint8 [M, d], scales float32 [d/128, scale_ld])."""
    _bits(x, torch.bfloat16)
    _dev(x, "x")
    n_src, d = x.shape
    M = (gather_rows.numel() if gather_rows is not None else n_src) if M is None else M
    scale_ld = M if scale_ld is None else scale_ld
    if q is None:
        q = torch.empty((M, d), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((d // 128, scale_ld), dtype=torch.float32, device=x.device)
    _check(_lib.moe_quant_1x128(_ptr(x), n_src, _ptr(gather_rows), M, d, _ptr(q), _ptr(scales),
                                scale_ld, _ptr(status), _stream(stream)), "moe_quant_1x128")
    return q, scales


def moe_quant_1x128_dispatch(x: torch.Tensor, inv_row: Optional[torch.Tensor], K: int, S: int,
                             q: Optional[torch.Tensor] = None,
                             scales: Optional[torch.Tensor] = None,
                             status: Optional[torch.Tensor] = None, stream=None):
    """x bf16 [T, d] -> (q uint8 [T*(K+S), d], scales float32 [d/128, T*(K+S)]), each token
    quantised once and written to its routed rows inv_row[t] and its shared rows."""
    _bits(x, torch.bfloat16)
    _dev(x, "x")
    T, d = x.shape
    M = T * (K + S)
    if q is None:
        q = torch.empty((M, d), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((d // 128, M), dtype=torch.float32, device=x.device)
    _check(_lib.moe_quant_1x128_dispatch(_ptr(x), T, d, _ptr(inv_row), K, S, _ptr(q),
                                         _ptr(scales), scales.shape[1], _ptr(status),
                                         _stream(stream)), "moe_quant_1x128_dispatch")
    return q, scales


def moe_quant_128x128(w: torch.Tensor, q: Optional[torch.Tensor] = None,
                      scales: Optional[torch.Tensor] = None, stream=None):
    """w float32 [R, C] -> (q uint8 [R, C], scales float32 [R/128, C/128])."""
    _bits(w, torch.float32)
    _dev(w, "w")
    R, C = w.shape
    if q is None:
        q = torch.empty((R, C), dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty((R // 128, C // 128), dtype=torch.float32, device=w.device)
    _check(_lib.moe_quant_128x128(_ptr(w), R, C, _ptr(q), _ptr(scales), _stream(stream)),
           "moe_quant_128x128")
    return q, scales


def route_workspace_bytes(T: int, E: int, d: int) -> int:
    """moe_route's workspace bytes (moe_route_workspace_size)."""
    return max(int(_lib.moe_route_workspace_size(T, d, E)), 256)


def moe_route(u: torch.Tensor, centroids: torch.Tensor, bias: torch.Tensor, K: int,
              ws: Optional[torch.Tensor] = None, out: Optional[dict] = None, stream=None) -> dict:
    T, d, E = _router_inputs(u, centroids, bias)
    dev = u.device
    if out is None:
        out = {"idx": torch.empty((T, K), dtype=torch.int32, device=dev),
               "gate": torch.empty((T, K), dtype=torch.float32, device=dev),
               "tie": torch.empty((T,), dtype=torch.uint8, device=dev),
               "counts": torch.empty((E,), dtype=torch.int32, device=dev)}
    if ws is None:
        ws = torch.empty(route_workspace_bytes(T, E, d), dtype=torch.uint8, device=dev)
    _check(_lib.moe_route(_ptr(u), _ptr(centroids), _ptr(bias), T, d, E, K, _ptr(out["idx"]),
                          _ptr(out["gate"]), _ptr(out["tie"]), _ptr(out["counts"]), _ptr(ws),
                          ws.numel() * ws.element_size(), _stream(stream)), "moe_route")
    return out


def moe_route_grouped(u: torch.Tensor, centroids: torch.Tensor, bias: torch.Tensor, K: int,
                      n_groups: int, topk_groups: int, group_topk: int,
                      ws: Optional[torch.Tensor] = None, out: Optional[dict] = None,
                      stream=None) -> dict:
    """Group-limited routing: keep the topk_groups best of n_groups expert
    groups (score: sum of a group's group_topk best biased scores), then top-K
    inside them."""
    T, d, E = _router_inputs(u, centroids, bias)
    dev = u.device
    if out is None:
        out = {"idx": torch.empty((T, K), dtype=torch.int32, device=dev),
               "gate": torch.empty((T, K), dtype=torch.float32, device=dev),
               "tie": torch.empty((T,), dtype=torch.uint8, device=dev),
               "counts": torch.empty((E,), dtype=torch.int32, device=dev)}
    if ws is None:
        ws = torch.empty(route_workspace_bytes(T, E, d), dtype=torch.uint8, device=dev)
    _check(_lib.moe_route_grouped(_ptr(u), _ptr(centroids), _ptr(bias), T, d, E, K, n_groups,
                                  topk_groups, group_topk, _ptr(out["idx"]), _ptr(out["gate"]),
                                  _ptr(out["tie"]), _ptr(out["counts"]), _ptr(ws),
                                  ws.numel() * ws.element_size(), _stream(stream)),
           "moe_route_grouped")
    return out


def moe_route_estimate_logits(u: torch.Tensor, centroids: torch.Tensor, stream=None):
    """The router's tensor-core logit estimates [T, E] and the per-expert
    centroid norms of its error bound (check hook of moe_route's screening step)."""
    _bits(u, torch.bfloat16)
    _dev(u, "u")
    T, d = u.shape
    E = centroids.shape[0]
    out = torch.empty((T, E), dtype=torch.float32, device=u.device)
    norms = torch.empty((E,), dtype=torch.float32, device=u.device)
    ws = torch.empty(route_workspace_bytes(T, E, d), dtype=torch.uint8, device=u.device)
    _check(_lib.moe_route_estimate_logits(_ptr(u), _ptr(centroids), T, d, E, _ptr(out), _ptr(norms),
                                          _ptr(ws), ws.numel(), _stream(stream)),
           "moe_route_estimate_logits")
    return out, norms


def moe_route_noalloc(u: torch.Tensor, centroids: torch.Tensor, bias: torch.Tensor, K: int,
                      out: Optional[dict] = None, stream=None) -> dict:
    """moe_route without a workspace (the logits use the library's fixed
    device array; T * E <= 1048576; concurrent calls on one device race)."""
    fn = _lib.moe_route_noalloc
    T, d, E = _router_inputs(u, centroids, bias)
    dev = u.device
    if out is None:
        out = {"idx": torch.empty((T, K), dtype=torch.int32, device=dev),
               "gate": torch.empty((T, K), dtype=torch.float32, device=dev),
               "tie": torch.empty((T,), dtype=torch.uint8, device=dev),
               "counts": torch.empty((E,), dtype=torch.int32, device=dev)}
    _check(fn(_ptr(u), _ptr(centroids), _ptr(bias), T, d, E, K, _ptr(out["idx"]),
              _ptr(out["gate"]), _ptr(out["tie"]), _ptr(out["counts"]), _stream(stream)),
           "moe_route_noalloc")
    return out


def moe_permute(topk_idx: torch.Tensor, E: int, S: int = 0, ws: Optional[torch.Tensor] = None,
                status: Optional[torch.Tensor] = None, out: Optional[dict] = None,
                stream=None) -> dict:
    _dev(topk_idx, "topk_idx")
    T, K = topk_idx.shape
    dev = topk_idx.device
    if out is None:
        out = {"offsets": torch.empty((E + 1,), dtype=torch.int32, device=dev),
               "group_offsets": torch.empty((E + S + 1,), dtype=torch.int32, device=dev),
               "perm_token": torch.empty((T * (K + S),), dtype=torch.int32, device=dev),
               "inv_row": torch.empty((T, K), dtype=torch.int32, device=dev)}
    if ws is None:
        nchunks = (T + 63) // 64
        ws = torch.empty(2 * ((4 * nchunks * E + 255) // 256 * 256) + 256, dtype=torch.uint8,
                         device=dev)
    _check(_lib.moe_permute(_ptr(topk_idx), T, K, E, S, _ptr(out["offsets"]),
                            _ptr(out.get("group_offsets")), _ptr(out["perm_token"]),
                            _ptr(out["inv_row"]), _ptr(status), _ptr(ws),
                            ws.numel() * ws.element_size(), _stream(stream)), "moe_permute")
    return out


def _out_dtype(mode: int):
    return {MOE_GEMM_GATE_UP_SILU_QUANT: torch.uint8, MOE_GEMM_DOWN_F32: torch.float32}.get(
        mode, torch.bfloat16)


def moe_grouped_gemm_fp8(mode: int, A: torch.Tensor, sa: torch.Tensor,
                         group_offsets: torch.Tensor, W0: torch.Tensor,
                         W1: Optional[torch.Tensor], sw0: torch.Tensor,
                         sw1: Optional[torch.Tensor], out: Optional[torch.Tensor] = None,
                         out_scales: Optional[torch.Tensor] = None,
                         status: Optional[torch.Tensor] = None, stream=None):
    """A uint8 [M_total, Kdim]; W0/W1 uint8 [G, N, Kdim] -> out (fp8 codes or bf16) [, scales]."""
    _dev(A, "A")
    M_total, Kdim = A.shape
    G, N, _ = W0.shape
    dev = A.device
    if out is None:
        out = torch.empty((M_total, N), dtype=_out_dtype(mode), device=dev)
    if mode == MOE_GEMM_GATE_UP_SILU_QUANT and out_scales is None:
        out_scales = torch.empty((N // 128, M_total), dtype=torch.float32, device=dev)
    _check(_lib.moe_grouped_gemm_fp8(mode, _ptr(A), _ptr(sa), M_total, _ptr(group_offsets), G,
                                     _ptr(W0), _ptr(W1), _ptr(sw0), _ptr(sw1), N, Kdim, _ptr(out),
                                     _ptr(out_scales), _ptr(status), _stream(stream)),
           "moe_grouped_gemm_fp8")
    return (out, out_scales) if mode == MOE_GEMM_GATE_UP_SILU_QUANT else out


def moe_grouped_gemm_fp8_small(mode: int, A: torch.Tensor, sa: torch.Tensor,
                               group_offsets: torch.Tensor, W0: torch.Tensor,
                               W1: Optional[torch.Tensor], sw0: torch.Tensor,
                               sw1: Optional[torch.Tensor], out: Optional[torch.Tensor] = None,
                               out_scales: Optional[torch.Tensor] = None,
                               status: Optional[torch.Tensor] = None, stream=None):
    """moe_grouped_gemm_fp8 with the small-group tiles (same arguments and results)."""
    _dev(A, "A")
    M_total, Kdim = A.shape
    G, N, _ = W0.shape
    dev = A.device
    if out is None:
        out = torch.empty((M_total, N), dtype=_out_dtype(mode), device=dev)
    if mode == MOE_GEMM_GATE_UP_SILU_QUANT and out_scales is None:
        out_scales = torch.empty((N // 128, M_total), dtype=torch.float32, device=dev)
    _check(_lib.moe_grouped_gemm_fp8_small(mode, _ptr(A), _ptr(sa), M_total, _ptr(group_offsets),
                                           G, _ptr(W0), _ptr(W1), _ptr(sw0), _ptr(sw1), N, Kdim,
                                           _ptr(out), _ptr(out_scales), _ptr(status),
                                           _stream(stream)), "moe_grouped_gemm_fp8_small")
    return (out, out_scales) if mode == MOE_GEMM_GATE_UP_SILU_QUANT else out


def moe_grouped_gemm_fp8_down(H: torch.Tensor, sh: torch.Tensor, group_offsets: torch.Tensor,
                              W: torch.Tensor, sw: torch.Tensor, f32_group0: int, f32_row0: int,
                              y: Optional[torch.Tensor], y_f32: Optional[torch.Tensor],
                              small_tiles: bool = False, status: Optional[torch.Tensor] = None,
                              stream=None):
    """The layer's down projection: rows of groups < f32_group0 to y (bf16),
    rows of the later groups to y_f32 (float32, row - f32_row0)."""
    _dev(H, "H")
    M_total, Kdim = H.shape
    G, N, _ = W.shape
    if y is not None:
        _bits(y, torch.bfloat16)
    if y_f32 is not None:
        _bits(y_f32, torch.float32)
    _check(_lib.moe_grouped_gemm_fp8_down(_ptr(H), _ptr(sh), M_total, _ptr(group_offsets), G,
                                          f32_group0, f32_row0, _ptr(W), _ptr(sw), N, Kdim, _ptr(y),
                                          _ptr(y_f32), 1 if small_tiles else 0, _ptr(status),
                                          _stream(stream)), "moe_grouped_gemm_fp8_down")
    return y, y_f32


def moe_combine(u: torch.Tensor, Y: torch.Tensor, topk_gate: torch.Tensor, inv_row: torch.Tensor,
                Y_shared: Optional[torch.Tensor], S: int, h: Optional[torch.Tensor] = None,
                stream=None) -> torch.Tensor:
    """h' = u + shared rows + gate-weighted routed rows; Y bf16 (routed rows),
    Y_shared float32 (the outputs of moe_grouped_gemm_fp8_down)."""
    _bits(u, torch.bfloat16)
    _bits(Y, torch.bfloat16)
    if Y_shared is not None:
        _bits(Y_shared, torch.float32)
    T, d = u.shape
    K = topk_gate.shape[1]
    if h is None:
        h = torch.empty((T, d), dtype=torch.float32, device=u.device)
    _check(_lib.moe_combine(_ptr(u), _ptr(Y), _ptr(topk_gate), _ptr(inv_row), _ptr(Y_shared), T, d,
                            K, S, _ptr(h), _stream(stream)), "moe_combine")
    return h


def moe_update_bias(counts: torch.Tensor, bias: torch.Tensor, T: int, K: int, gamma: float,
                    stream=None) -> torch.Tensor:
    _check(_lib.moe_update_bias(_ptr(counts), counts.numel(), T, K, gamma, _ptr(bias),
                                _stream(stream)), "moe_update_bias")
    return bias


def moe_check_device_status(status: torch.Tensor, stream=None) -> int:
    return int(_lib.moe_check_device_status(_ptr(status), _stream(stream)))


def moe_workspace_size(layer: moe_layer_t, T: int) -> int:
    return int(_lib.moe_workspace_size(ctypes.byref(layer), T))


def moe_forward(layer: moe_layer_t, u: torch.Tensor, ws: torch.Tensor, out: dict,
                stream=None) -> dict:
    """One layer forward into the preallocated tensors of `out` (h, idx, gate, counts, tie)."""
    T = u.shape[0]
    _check(_lib.moe_forward(ctypes.byref(layer), _ptr(u), T, _ptr(out["h"]), _ptr(out["idx"]),
                            _ptr(out["gate"]), _ptr(out["counts"]), _ptr(out["tie"]), _ptr(ws),
                            ws.numel() * ws.element_size(), _stream(stream)), "moe_forward")
    return out


def moe_forward_host(L: moe_layer_t, T: int, u_host: list, h_host: list, gamma: float,
                     bufs: list, ws: torch.Tensor, compute_stream=None, h2d_stream=None,
                     d2h_stream=None) -> None:
    """moe_forward_host: the layer over the batches u_host[k] (pinned [T, d]
    bf16 host tensors), outputs to h_host[k] (pinned [T, d] float32), with
    uploads, compute and downloads on three streams.  bufs: two dicts of
    device tensors with keys u, h, idx, gate, tie, counts.  Asynchronous:
    synchronise d2h_stream before reading h_host."""
    n = len(u_host)
    if len(h_host) != n or len(bufs) != 2:
        raise ValueError("need one output per batch and two buffer sets")
    for t in u_host:
        _bits(t, torch.bfloat16)
        if t.is_cuda:
            raise ValueError("u_host must be host tensors")
    for t in h_host:
        if t.is_cuda or t.dtype != torch.float32:
            raise ValueError("h_host must be float32 host tensors")
    u_arr = (ctypes.c_void_p * max(n, 1))(*[_ptr(t) for t in u_host])
    h_arr = (ctypes.c_void_p * max(n, 1))(*[_ptr(t) for t in h_host])
    b_arr = (moe_batch_buffers_t * 2)(*[moe_batch_buffers_t(_ptr(b["u"]), _ptr(b["h"]), _ptr(b["idx"]),
                                                            _ptr(b["gate"]), _ptr(b["tie"]),
                                                            _ptr(b["counts"])) for b in bufs])
    _check(_lib.moe_forward_host(ctypes.byref(L), T, n, ctypes.cast(u_arr, P),
                                 ctypes.cast(h_arr, P), gamma, b_arr, _ptr(ws),
                                 ws.numel() * ws.element_size(), _stream(compute_stream),
                                 _stream(h2d_stream), _stream(d2h_stream)), "moe_forward_host")


def moe_forward_pipelined(L: moe_layer_t, batches: list, gamma: float, ws0: torch.Tensor,
                          ws1: torch.Tensor, reserve_sms: int = 0, gemm_stream=None,
                          side_stream=None) -> None:
    """moe_forward_pipelined: batches is a list of dicts of device tensors
    (u, h, idx, gate, tie, counts), all with the same T; two micro-batches are
    in flight (one in its expert GEMMs, the other in routing/dispatch or
    combine).  Asynchronous: synchronise side_stream before reading outputs."""
    n = len(batches)
    if n == 0:
        return
    T = batches[0]["u"].shape[0]
    for b in batches:
        _bits(b["u"], torch.bfloat16)
        _dev(b["u"], "u")
        if b["u"].shape[0] != T:
            raise ValueError("every batch needs the same number of tokens")
    arr = (moe_batch_buffers_t * n)(*[moe_batch_buffers_t(_ptr(b["u"]), _ptr(b["h"]), _ptr(b["idx"]),
                                                          _ptr(b["gate"]), _ptr(b["tie"]),
                                                          _ptr(b["counts"])) for b in batches])
    nbytes = min(ws0.numel() * ws0.element_size(), ws1.numel() * ws1.element_size())
    _check(_lib.moe_forward_pipelined(ctypes.byref(L), T, n, arr, gamma, _ptr(ws0), _ptr(ws1), nbytes,
                                      reserve_sms, _stream(gemm_stream), _stream(side_stream)),
           "moe_forward_pipelined")


def moe_prepare_backward_weights(L: moe_layer_t, w_down_t: torch.Tensor, s_down_t: torch.Tensor,
                                 w_gu_t: torch.Tensor, s_gu_t: torch.Tensor, stream=None) -> None:
    """The transposed weight blocks the input gradient uses (exact in FP8)."""
    _check(_lib.moe_prepare_backward_weights(ctypes.byref(L), _ptr(w_down_t), _ptr(s_down_t),
                                             _ptr(w_gu_t), _ptr(s_gu_t), _stream(stream)),
           "moe_prepare_backward_weights")


def moe_backward_workspace_size(L: moe_layer_t, T: int) -> int:
    return int(_lib.moe_backward_workspace_size(ctypes.byref(L), T))


def moe_backward_dgrad(L: moe_layer_t, B: moe_layer_bwd_t, u: torch.Tensor, dh: torch.Tensor,
                       fwd: dict, fwd_ws: torch.Tensor, bwd_ws: torch.Tensor,
                       du: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """du for the forward whose outputs (idx, gate) and workspace are given."""
    _bits(u, torch.bfloat16)
    _bits(dh, torch.bfloat16)
    _dev(u, "u")
    T, d = u.shape
    if du is None:
        du = torch.empty((T, d), dtype=torch.float32, device=u.device)
    _check(_lib.moe_backward_dgrad(ctypes.byref(L), ctypes.byref(B), _ptr(u), _ptr(dh), T,
                                   _ptr(fwd["idx"]), _ptr(fwd["gate"]), _ptr(du), _ptr(fwd_ws),
                                   fwd_ws.numel() * fwd_ws.element_size(), _ptr(bwd_ws),
                                   bwd_ws.numel() * bwd_ws.element_size(), _stream(stream)),
           "moe_backward_dgrad")
    return du


def moe_wgrad_ld(M: int, G: int) -> int:
    """Columns of a 128x1 re-quantised operand with M rows in G groups."""
    return int(_lib.moe_wgrad_ld(M, G))


def moe_requant_128x1(q: torch.Tensor, scales: torch.Tensor, group_offsets: torch.Tensor,
                      ld: Optional[int] = None, status: Optional[torch.Tensor] = None,
                      stream=None):
    """q uint8 [M, C] with scales [C/128, M] -> (qt uint8 [C, ld], st float32 [ld/128, C])."""
    _dev(q, "q")
    M, C = q.shape
    G = group_offsets.numel() - 1
    if ld is None:
        ld = moe_wgrad_ld(M, G)
    qt = torch.zeros((C, ld), dtype=torch.uint8, device=q.device)
    st = torch.zeros((ld // 128, C), dtype=torch.float32, device=q.device)
    _check(_lib.moe_requant_128x1(_ptr(q), _ptr(scales), M, C, _ptr(group_offsets), G, _ptr(qt),
                                  _ptr(st), ld, _ptr(status), _stream(stream)), "moe_requant_128x1")
    return qt, st


def moe_wgrad_gemm_fp8(At: torch.Tensor, sAt: torch.Tensor, Bt: torch.Tensor, sBt: torch.Tensor,
                       group_offsets: torch.Tensor, split: Optional[int] = None,
                       status: Optional[torch.Tensor] = None, stream=None):
    """At uint8 [Na, ld], Bt uint8 [Nb, ld] (128x1 layout) -> float32 [G, Na, Nb]
    (or the two row blocks [G, split, Nb], [G, Na - split, Nb] when split < Na)."""
    _dev(At, "At")
    Na, ld = At.shape
    Nb = Bt.shape[0]
    G = group_offsets.numel() - 1
    split = Na if split is None else split
    out0 = torch.empty((G, split, Nb), dtype=torch.float32, device=At.device)
    out1 = (torch.empty((G, Na - split, Nb), dtype=torch.float32, device=At.device)
            if split < Na else None)
    _check(_lib.moe_wgrad_gemm_fp8(_ptr(At), _ptr(sAt), Na, _ptr(Bt), _ptr(sBt), Nb, ld,
                                   _ptr(group_offsets), G, _ptr(out0), _ptr(out1), split,
                                   _ptr(status), _stream(stream)), "moe_wgrad_gemm_fp8")
    return out0 if out1 is None else (out0, out1)


def moe_wgrad_workspace_size(L: moe_layer_t, T: int) -> int:
    return int(_lib.moe_wgrad_workspace_size(ctypes.byref(L), T))


def moe_backward_wgrad(L: moe_layer_t, T: int, fwd_ws: torch.Tensor, bwd_ws: torch.Tensor,
                       wgrad_ws: torch.Tensor, dW_gate: torch.Tensor, dW_up: torch.Tensor,
                       dW_down: torch.Tensor, stream=None) -> None:
    """Weight gradients of every expert for the batch of the last forward and
    input-gradient calls that used fwd_ws and bwd_ws."""
    for t, n in ((dW_gate, "dW_gate"), (dW_up, "dW_up"), (dW_down, "dW_down")):
        _dev(t, n)
        if t.dtype != torch.float32:
            raise TypeError(f"{n} must be float32")
    _check(_lib.moe_backward_wgrad(ctypes.byref(L), T, _ptr(dW_gate), _ptr(dW_up), _ptr(dW_down),
                                   _ptr(fwd_ws), fwd_ws.numel() * fwd_ws.element_size(),
                                   _ptr(bwd_ws), bwd_ws.numel() * bwd_ws.element_size(),
                                   _ptr(wgrad_ws), wgrad_ws.numel() * wgrad_ws.element_size(),
                                   _stream(stream)), "moe_backward_wgrad")
