"""The C-ABI library builds, loads without a GPU and exports every entry point
include/moe_ffn.h declares; host-side argument checks answer before any CUDA
call.  (No compute calls here: this module runs on machines without a GPU.)"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_ffn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*(moe_[a-z0-9_]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_ffn_top_gb300 import build

    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_pipeline_calls():
    names = declared_functions()
    for n in ["moe_router_topk", "moe_bucket", "moe_grouped_ffn", "moe_combine", "moe_ffn_prefill",
              "moe_weights_create", "moe_ffn_workspace_size", "moe_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"


def test_binding_covers_every_declared_symbol():
    from mixture_experts_ffn_top_gb300 import ops

    missing = [n for n in declared_functions() if n not in ops._SIGS]
    assert not missing


def test_status_strings_and_version(lib):
    lib.moe_status_string.restype = ctypes.c_char_p
    for code in range(0, -9, -1):
        assert lib.moe_status_string(code)
    assert lib.moe_abi_version() == 1
    assert lib.moe_status_from_word(0) == 0
    assert lib.moe_status_from_word(1) == -7 and lib.moe_status_from_word(2) == -8 and lib.moe_status_from_word(4) == -5


def test_workspace_size_rules(lib):
    f = lib.moe_ffn_workspace_size
    f.restype = ctypes.c_size_t
    assert f(2048, 2048, 64, 1024, 8, 0) > 0
    assert f(2048, 2048, 64, 1024, 8, 0) >= f(1024, 2048, 64, 1024, 8, 0)
    assert f(512, 2048, 256, 512, 8, 512) > f(512, 2048, 256, 512, 8, 0)
    # invalid shapes give 0
    assert f(0, 2048, 64, 1024, 8, 0) == 0          # N < 1
    assert f(16, 2000, 64, 1024, 8, 0) == 0         # D not a multiple of 32
    assert f(16, 2048, 64, 1000, 8, 0) == 0         # F not a multiple of 32
    assert f(16, 2048, 4, 1024, 8, 0) == 0          # top_k > E
    assert f(16, 2048, 2048, 1024, 8, 0) == 0       # E > 1024
    assert f(16, 2048, 64, 1024, 33, 0) == 0        # top_k > 32


def test_bucket_workspace_size(lib):
    f = lib.moe_bucket_workspace_size
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
    assert f(2048, 8, 64) > 256                     # status block + count table
    assert f(2048, 8, 1024) >= f(2048, 8, 64)
    assert f(0, 8, 64) == 0 and f(16, 33, 64) == 0 and f(16, 8, 4) == 0
    full = lib.moe_ffn_workspace_size
    full.restype = ctypes.c_size_t
    for N, E, k in [(2048, 64, 8), (512, 256, 8), (40000, 64, 8), (20000, 1024, 2)]:
        assert full(N, 2048, E, 1024, k, 0) >= f(N, k, E)


def test_null_arguments_rejected_before_any_cuda_call(lib):
    V = ctypes.c_void_p
    lib.moe_combine.argtypes = [V, V, V, ctypes.c_int, ctypes.c_int, ctypes.c_int, V, V]
    assert lib.moe_combine(None, None, None, 4, 2, 64, None, None) == -1
    lib.moe_router_topk.argtypes = [V, V, V] + [ctypes.c_int] * 5 + [V] * 7 + [ctypes.c_size_t, V]
    assert lib.moe_router_topk(*([None] * 3 + [4, 64, 8, 2, 0] + [None] * 7 + [0, None])) == -1
    lib.moe_weights_create.argtypes = [ctypes.POINTER(V), ctypes.c_int, ctypes.c_int, ctypes.c_int, V, V, V,
                                       ctypes.c_int, V, V, V, V]
    h = V()
    assert lib.moe_weights_create(ctypes.byref(h), 8, 256, 128, None, None, None, 0, None, None, None, None) == -1
    lib.moe_ffn_prefill.argtypes = [V, V, V, V] + [ctypes.c_int] * 3 + [V, V, ctypes.c_size_t, V]
    assert lib.moe_ffn_prefill(None, None, None, None, 4, 2, 0, None, None, 0, None) == -1
    lib.moe_device_host_numa_node.argtypes = [V]
    assert lib.moe_device_host_numa_node(None) == -1


def test_norm_entry_points_reject_bad_arguments_before_any_cuda_call(lib):
    """Null pointers, a non-positive or non-finite eps and a normed buffer that is the output are
    refused (MOE_ERR_INVALID_ARG) by the host-side checks; the pointers below are never dereferenced."""
    V, F, I = ctypes.c_void_p, ctypes.c_float, ctypes.c_int
    a, b, c, d = V(0x1000), V(0x2000), V(0x3000), V(0x4000)
    lib.moe_rmsnorm.argtypes = [V, V, F, I, I, V, V]
    assert lib.moe_rmsnorm(None, b, 1e-6, 4, 64, c, None) == -1
    for eps in (0.0, -1.0, float("inf"), float("nan")):
        assert lib.moe_rmsnorm(a, b, eps, 4, 64, c, None) == -1
    assert lib.moe_rmsnorm(a, b, 1e-6, 4, 64, a, None) == -1          # normed is x
    lib.moe_combine_residual_rmsnorm.argtypes = [V, V, V, V, V, F, I, I, I, V, V, V]
    assert lib.moe_combine_residual_rmsnorm(a, b, None, None, c, 1e-6, 4, 2, 64, d, V(0x5000), None) == -1
    assert lib.moe_combine_residual_rmsnorm(a, b, None, c, d, 1e-6, 4, 2, 64, V(0x5000), V(0x5000), None) == -1
    assert lib.moe_combine_residual_rmsnorm(a, b, None, c, d, 0.0, 4, 2, 64, V(0x5000), V(0x6000), None) == -1
    lib.moe_ffn_prefill_residual_rmsnorm.argtypes = [V, V, V, V, V, V, F, I, I, I, V, V, I, V, ctypes.c_size_t, V]
    assert lib.moe_ffn_prefill_residual_rmsnorm(None, a, b, None, c, d, 1e-6, 4, 2, 0, V(0x5000), V(0x5000), 0,
                                                None, 0, None) == -1
    lib.moe_ffn_prefill_stack_rmsnorm.argtypes = [V, V, V, V, F, I, V, V, I, I, I, I, V, ctypes.c_size_t, V]
    assert lib.moe_ffn_prefill_stack_rmsnorm(None, None, None, None, 1e-6, 1, a, b, 4, 2, 0, 0, None, 0, None) == -1
