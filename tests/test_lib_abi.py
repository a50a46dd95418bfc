"""The C ABI library loads without a GPU, exports every declared entry point,
and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(moe_\w+)\s*\(", src, flags=re.M)
    return names


@pytest.fixture(scope="module")
def lib():
    from fine_grained_fp8_bias_b300 import build
    build.build()
    from fine_grained_fp8_bias_b300 import lib as L
    return L


def test_every_declared_symbol_is_exported(lib):
    names = declared()
    assert len(names) >= 13
    for n in ("moe_route", "moe_permute", "moe_quant_1x128", "moe_grouped_gemm_fp8",
              "moe_combine", "moe_forward", "moe_update_bias", "moe_workspace_size",
              "moe_status_string"):
        assert n in names
    for n in names:
        assert hasattr(lib.lib(), n), n


def declared_params():
    """name -> number of parameters, from the declarations in include/*.h."""
    out = {}
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            for m in re.finditer(r"\b(moe_\w+)\s*\(([^;{]*?)\)\s*;", src, flags=re.S):
                params = m.group(2).strip()
                out[m.group(1)] = 0 if params in ("", "void") else len(params.split(","))
    return out


def test_every_entry_point_has_its_ctypes_signature(lib):
    # ctypes passes Python ints as C int unless argtypes say otherwise, which
    # cuts device pointers to 32 bits: every declared call must be typed, with
    # as many argument types as the declaration has parameters
    params = declared_params()
    assert set(params) == set(declared())
    for name, n in params.items():
        fn = getattr(lib.lib(), name)
        assert fn.argtypes is not None, name
        assert len(fn.argtypes) == n, (name, len(fn.argtypes), n)
        assert fn.restype is not None, name


def test_status_strings(lib):
    L = lib.lib()
    assert L.moe_status_string(0) == b"ok"
    for code in range(-7, 0):
        assert L.moe_status_string(code) not in (b"", b"unknown status")


def test_host_side_validation_needs_no_device(lib):
    L = lib.lib()
    fake = 1 << 20                     # never dereferenced: every call below fails validation
    # d not a multiple of 128
    assert L.moe_quant_1x128(fake, 4, None, 4, 100, fake, fake, 4, None, None) == -2
    assert L.moe_quant_128x128(fake, 100, 128, fake, fake, None) == -2
    # K > E, K > 32, E > 1024
    assert L.moe_route(fake, fake, fake, 4, 128, 4, 5, fake, fake, fake, fake, fake, 1 << 20, None) == -1
    assert L.moe_route(fake, fake, fake, 4, 128, 64, 33, fake, fake, fake, fake, fake, 1 << 20, None) == -1
    assert L.moe_route(fake, fake, fake, 4, 128, 2048, 8, fake, fake, fake, fake, fake, 1 << 20, None) == -1
    # workspace too small, misaligned pointer
    assert L.moe_route(fake, fake, fake, 4, 128, 8, 2, fake, fake, fake, fake, fake, 16, None) == -6
    assert L.moe_route(fake + 8, fake, fake, 4, 128, 8, 2, fake, fake, fake, fake, fake, 1 << 20, None) == -3
    assert L.moe_permute(fake, 4, 2, 8, 1, fake, None, fake, fake, None, fake, 0, None) == -6
    # GEMM: bad mode, N not a multiple of 128, too many groups, null pointers
    assert L.moe_grouped_gemm_fp8(3, fake, fake, 8, fake, 1, fake, None, fake, None, 128, 128,
                                  fake, None, None, None) == -1
    assert L.moe_grouped_gemm_fp8(2, fake, fake, 8, fake, 1, fake, None, fake, None, 100, 128,
                                  fake, None, None, None) == -2
    assert L.moe_grouped_gemm_fp8(2, fake, fake, 8, fake, 5000, fake, None, fake, None, 128, 128,
                                  fake, None, None, None) == -2
    assert L.moe_grouped_gemm_fp8(1, fake, fake, 8, fake, 1, fake, None, fake, None, 128, 128,
                                  fake, None, None, None) == -1
    assert L.moe_combine(fake, fake, fake, fake, fake, 4, 100, 2, 1, fake, None) == -2
    assert L.moe_update_bias(None, 8, 4, 2, ctypes.c_float(1e-3), fake, None) == -1
    assert L.moe_forward(None, fake, 4, fake, fake, fake, fake, fake, fake, 1 << 30, None) == -1


def test_workspace_size_and_layer_checks(lib):
    L = lib.lib()
    layer = lib.moe_layer_t(7168, 256, 8, 1, 2048, *([1 << 20] * 8))
    n = L.moe_workspace_size(ctypes.byref(layer), 4096)
    M = 4096 * 9
    # the routed + shared activation copies, h and y dominate
    assert n >= M * 7168 + M * 2048 + 2 * M * 7168
    assert L.moe_workspace_size(ctypes.byref(layer), 0) > 0
    bad = lib.moe_layer_t(7000, 256, 8, 1, 2048, *([1 << 20] * 8))
    assert L.moe_forward(ctypes.byref(bad), 1 << 20, 4, 1 << 20, 1 << 20, 1 << 20, 1 << 20,
                         1 << 20, 1 << 20, 1 << 40, None) == -2
    k_too_big = lib.moe_layer_t(7168, 4, 8, 1, 2048, *([1 << 20] * 8))
    assert L.moe_forward(ctypes.byref(k_too_big), 1 << 20, 4, 1 << 20, 1 << 20, 1 << 20,
                         1 << 20, 1 << 20, 1 << 20, 1 << 40, None) == -1
    # workspace smaller than required
    assert L.moe_forward(ctypes.byref(layer), 1 << 20, 4096, 1 << 20, 1 << 20, 1 << 20, 1 << 20,
                         1 << 20, 1 << 20, 1024, None) == -6


def test_backward_entry_points_validate_on_the_host(lib):
    L = lib.lib()
    fake = 1 << 20                     # never dereferenced: every call below fails validation
    # padded column count of the 128x1 form: M + 127 G rounded up to 128
    assert L.moe_wgrad_ld(36864, 257) == (36864 + 127 * 257 + 127) // 128 * 128
    assert L.moe_wgrad_ld(1, 1) == 128 and L.moe_wgrad_ld(0, 5) == 640 and L.moe_wgrad_ld(-1, 1) == 0
    # re-quantisation: C not a multiple of 128, ld not a multiple of 16, null or misaligned buffers
    assert L.moe_requant_128x1(fake, fake, 300, 100, fake, 4, fake, fake, 1024, None, None) == -2
    assert L.moe_requant_128x1(fake, fake, 300, 128, fake, 4, fake, fake, 1000, None, None) == -2
    assert L.moe_requant_128x1(fake, None, 300, 128, fake, 4, fake, fake, 1024, None, None) == -1
    assert L.moe_requant_128x1(fake + 8, fake, 300, 128, fake, 4, fake, fake, 1024, None, None) == -3
    assert L.moe_requant_128x1(fake, fake, 0, 128, fake, 4, fake, fake, 1024, None, None) == 0
    # token-contracted GEMM: sizes, split, the second output, alignment
    assert L.moe_wgrad_gemm_fp8(fake, fake, 100, fake, fake, 128, 1024, fake, 4, fake, None, 100,
                                None, None) == -2
    assert L.moe_wgrad_gemm_fp8(fake, fake, 256, fake, fake, 128, 1024, fake, 4, fake, None, 384,
                                None, None) == -1
    assert L.moe_wgrad_gemm_fp8(fake, fake, 256, fake, fake, 128, 1024, fake, 4, fake, None, 128,
                                None, None) == -1
    assert L.moe_wgrad_gemm_fp8(fake, fake, 256, fake, fake, 128, 1024, fake, 4, fake + 8, fake, 128,
                                None, None) == -3
    assert L.moe_wgrad_gemm_fp8(fake, fake, 256, fake, fake, 128, 1024, fake, 0, fake, fake, 128,
                                None, None) == 0
    # layer-level backward: workspace sizes, a missing transposed-weight set, short or misaligned workspaces
    layer = lib.moe_layer_t(7168, 256, 8, 1, 2048, *([1 << 20] * 8))
    T = 4096
    nb = L.moe_backward_workspace_size(ctypes.byref(layer), T)
    nw = L.moe_wgrad_workspace_size(ctypes.byref(layer), T)
    M, ld = T * 9, L.moe_wgrad_ld(T * 9, 257)
    assert nb >= M * 7168 + 2 * M * 2048 + M * 2 * 2048 + 2 * M * 7168
    assert nw >= ld * (2 * 7168 + 2048 + 2 * 2048)
    nf = L.moe_workspace_size(ctypes.byref(layer), T)
    assert L.moe_backward_dgrad(ctypes.byref(layer), None, fake, fake, T, fake, fake, fake, fake, nf,
                                fake, nb, None) == -1
    assert L.moe_backward_wgrad(ctypes.byref(layer), T, fake, fake, fake, fake, nf, fake, nb, fake,
                                nw - 256, None) == -6
    assert L.moe_backward_wgrad(ctypes.byref(layer), T, fake, fake, fake, fake, nf, fake, nb,
                                fake + 16, nw, None) == -3
    assert L.moe_backward_wgrad(ctypes.byref(layer), -1, fake, fake, fake, fake, nf, fake, nb, fake,
                                nw, None) == -1


def test_layer_with_more_than_32_rows_per_token_is_rejected(lib):
    # K + S > 32: a token would need more dispatch rows than the quantiser's lanes
    L = lib.lib()
    fake = 1 << 20
    layer = lib.moe_layer_t(256, 64, 32, 1, 128, *([fake] * 8))
    assert L.moe_forward(ctypes.byref(layer), fake, 4, fake, fake, fake, fake, fake, fake,
                         1 << 40, None) == -1
    ok = lib.moe_layer_t(256, 64, 31, 1, 128, *([fake] * 8))
    # K + S = 32 passes the layer checks (and then fails on the short workspace)
    assert L.moe_forward(ctypes.byref(ok), fake, 4, fake, fake, fake, fake, fake, fake, 16,
                         None) == -6


def test_router_wrappers_check_their_inputs_on_the_host(lib):
    # CPU tensors, wrong dtypes and mismatched shapes never reach a kernel
    import torch
    u = torch.zeros((4, 128), dtype=torch.bfloat16)
    c = torch.zeros((8, 128), dtype=torch.float32)
    b = torch.zeros((8,), dtype=torch.float32)
    for fn in (lib.moe_route, lib.moe_route_noalloc):
        with pytest.raises(ValueError):
            fn(u, c, b, 2)                                   # host tensors
        with pytest.raises(TypeError):
            fn(u, c.half(), b, 2)                            # centroids not float32
        with pytest.raises(TypeError):
            fn(u.float(), c, b, 2)                           # u not bf16
    with pytest.raises(ValueError):
        lib._router_inputs(u, c, b)
