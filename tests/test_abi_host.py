"""C-ABI checks on the host: the library builds and loads, exports every
function that include/k3moe.h declares, and rejects bad arguments before any
launch (no GPU needed).  One GPU-marked test checks the AUTO mode's resolution,
which needs the driver's tensor-map encoder that the GEMM modes depend on."""
import ctypes
import os
import re

import pytest

import mxfp4_expert_ffn_router_gb300 as k3
from mxfp4_expert_ffn_router_gb300 import build as k3build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    k3build.build()
    return k3.lib()


def _declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        txt = open(os.path.join(ROOT, "include", h)).read()
        txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
        names += re.findall(r"\b(k3moe_[a-z0-9_]+)\s*\(", txt)
    return sorted(set(names))


def test_exports_every_declared_function(L):
    names = _declared_functions()
    assert {"k3moe_route", "k3moe_bucket", "k3moe_expert_ffn", "k3moe_combine"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def _shape(T=4, H=128, I=64, E=8, k=2):
    return k3.Shape(T, H, I, E, k)


@pytest.mark.parametrize("bad", [
    dict(T=-1), dict(E=0), dict(E=4097), dict(k=0), dict(k=33, E=64), dict(k=9, E=8),
    dict(H=48), dict(H=16416), dict(I=0), dict(I=40), dict(T=1 << 27, k=16),
])
def test_shape_rejected(L, bad):
    s = _shape(**bad)
    dummy = ctypes.c_void_p(256)
    assert L.k3moe_route(s, dummy, dummy, dummy, None, None) == k3.K3MOE_ERR_SHAPE
    assert L.k3moe_combine(s, dummy, dummy, dummy, dummy, None, None) == k3.K3MOE_ERR_SHAPE
    assert L.k3moe_workspace_bytes(s, k3.K3MOE_OP_EXPERT_FFN, 0) == 0


def test_null_pointers_rejected(L):
    s = _shape()
    d = ctypes.c_void_p(256)
    assert L.k3moe_route(s, None, d, d, None, None) == k3.K3MOE_ERR_ARG
    assert L.k3moe_route(s, d, None, d, None, None) == k3.K3MOE_ERR_ARG
    assert L.k3moe_bucket(s, d, None, d, d, d, None, 0, None, None) == k3.K3MOE_ERR_ARG
    assert L.k3moe_bucket(s, None, d, d, d, d, None, 0, None, None) == k3.K3MOE_ERR_ARG
    assert L.k3moe_combine(s, d, d, d, None, None, None) == k3.K3MOE_ERR_ARG
    ws = ctypes.c_void_p(4096)
    assert L.k3moe_expert_ffn(s, d, None, d, d, d, 0, ws, 1 << 30, None, None) == k3.K3MOE_ERR_ARG
    wz = k3._WeightsC(0, 256, 256, 256)
    assert L.k3moe_expert_ffn(s, d, ctypes.byref(wz), d, d, d, 0, ws, 1 << 30, None, None) == k3.K3MOE_ERR_ARG


def test_bad_mode_and_alignment_and_workspace(L):
    s = _shape()
    d = ctypes.c_void_p(256)
    wz = k3._WeightsC(256, 256, 256, 256)
    ws = ctypes.c_void_p(4096)
    need = L.k3moe_workspace_bytes(s, k3.K3MOE_OP_EXPERT_FFN, 0)
    assert need > 0
    assert L.k3moe_expert_ffn(s, d, ctypes.byref(wz), d, d, d, 99, ws, need, None, None) == k3.K3MOE_ERR_ARG
    assert L.k3moe_expert_ffn(s, ctypes.c_void_p(258), ctypes.byref(wz), d, d, d, 0, ws, need, None,
                              None) == k3.K3MOE_ERR_ALIGN
    assert L.k3moe_expert_ffn(s, d, ctypes.byref(wz), d, d, d, 0, ws, need - 1, None, None) == k3.K3MOE_ERR_WORKSPACE
    assert L.k3moe_expert_ffn(s, d, ctypes.byref(wz), d, d, d, 0, ctypes.c_void_p(4096 + 16), need,
                              None, None) == k3.K3MOE_ERR_WORKSPACE
    assert L.k3moe_combine(s, ctypes.c_void_p(260), d, d, d, None, None) == k3.K3MOE_ERR_ALIGN
    big = _shape(T=4096, k=16, E=896)
    nb = L.k3moe_workspace_bytes(big, k3.K3MOE_OP_BUCKET, 0)
    assert nb > 0
    assert L.k3moe_bucket(big, d, d, d, d, d, None, 0, None, None) == k3.K3MOE_ERR_WORKSPACE
    assert L.k3moe_bucket(big, d, d, d, d, d, ws, nb - 4, None, None) == k3.K3MOE_ERR_WORKSPACE


def test_empty_input_is_a_no_op(L):
    s = _shape(T=0)
    assert L.k3moe_route(s, None, None, None, None, None) == k3.K3MOE_OK
    assert L.k3moe_expert_ffn(s, None, None, None, None, None, 0, None, 0, None, None) == k3.K3MOE_OK
    assert L.k3moe_combine(s, None, None, None, None, None, None) == k3.K3MOE_OK


def test_no_gpu_means_arch_error_not_a_launch(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    s = _shape()
    d = ctypes.c_void_p(256)
    assert L.k3moe_route(s, d, d, d, None, None) == k3.K3MOE_ERR_ARCH


def test_status_strings(L):
    for code in range(-8, 1):
        assert k3.status_string(code) and "unknown" not in k3.status_string(code)
    assert "unknown" in k3.status_string(-99)


def test_binding_refuses_cpu_tensors(L):
    import torch
    s = _shape()
    with pytest.raises(ValueError):
        k3.k3moe_route(s, torch.zeros(4, 8), torch.zeros(4, 2, dtype=torch.int32),
                       torch.zeros(4, 2))


def test_quantize_host_validation(L):
    d = ctypes.c_void_p(256)
    assert L.k3moe_quantize_mxfp4(ctypes.c_int64(0), None, None, None, None) == k3.K3MOE_OK
    assert L.k3moe_quantize_mxfp4(ctypes.c_int64(48), d, d, d, None) == k3.K3MOE_ERR_SHAPE
    assert L.k3moe_quantize_mxfp4(ctypes.c_int64(-32), d, d, d, None) == k3.K3MOE_ERR_SHAPE
    assert L.k3moe_quantize_mxfp4(ctypes.c_int64(64), None, d, d, None) == k3.K3MOE_ERR_ARG
    assert L.k3moe_quantize_mxfp4(ctypes.c_int64(64), d, d, None, None) == k3.K3MOE_ERR_ARG
    assert L.k3moe_quantize_mxfp4(ctypes.c_int64(64), ctypes.c_void_p(258), d, d, None) == k3.K3MOE_ERR_ALIGN
    assert L.k3moe_quantize_mxfp4(ctypes.c_int64(64), d, ctypes.c_void_p(264), d, None) == k3.K3MOE_ERR_ALIGN


def test_w4a4_mode_is_a_valid_mode(L):
    s = _shape(T=8, H=256, I=128, E=4, k=2)
    assert L.k3moe_workspace_bytes(s, k3.K3MOE_OP_EXPERT_FFN, k3.K3MOE_FFN_W4A4) == \
        L.k3moe_workspace_bytes(s, k3.K3MOE_OP_EXPERT_FFN, k3.K3MOE_FFN_GEMM)
    d = ctypes.c_void_p(256)
    wz = k3._WeightsC(256, 256, 256, 256)
    assert L.k3moe_expert_ffn(s, d, ctypes.byref(wz), d, d, d, 5, d, 1 << 30, None, None) == k3.K3MOE_ERR_ARG


def _bench_module():
    import importlib.util
    spec = importlib.util.spec_from_file_location("k3moe_bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.gpu
@pytest.mark.parametrize("T,E,k,gemm", [
    (1, 896, 16, False), (8, 896, 16, False), (44, 896, 16, False),   # < 0.8 assignments per expert
    (45, 896, 16, True), (128, 896, 16, True), (300, 5, 1, True),     # >= 0.8: the tensor-core GEMM
])
def test_auto_mode_resolution(L, T, E, k, gemm):
    """AUTO resolves to the GEMM exactly when 5 A >= 4 E (the measured
    crossover at H = 7168, I = 2048), seen through the workspace it asks for, and
    bench.py's mirror of the rule (which labels and counts the kernels) agrees."""
    import gen
    s = gen.Shape(T, 7168, 2048, E, k)
    ws = {m: k3.k3moe_workspace_bytes(s, k3.K3MOE_OP_EXPERT_FFN, m)
          for m in (k3.K3MOE_FFN_AUTO, k3.K3MOE_FFN_GEMV, k3.K3MOE_FFN_GEMM)}
    assert ws[k3.K3MOE_FFN_GEMM] != ws[k3.K3MOE_FFN_GEMV]
    assert ws[k3.K3MOE_FFN_AUTO] == ws[k3.K3MOE_FFN_GEMM if gemm else k3.K3MOE_FFN_GEMV]
    assert _bench_module().resolved_mode(s, k3.K3MOE_FFN_AUTO) == (3 if gemm else 1)


def test_noalloc_modes_on_the_host(L):
    """The allocation-free entry point serves the CUDA-core modes only: GEMM and
    W4A4 are refused as unsupported and an unknown mode as a bad argument, before
    any device call (so on a machine without a GPU too)."""
    s = _shape()
    d = ctypes.c_void_p(256)
    wz = k3._WeightsC(256, 256, 256, 256)
    for mode in (k3.K3MOE_FFN_GEMM, k3.K3MOE_FFN_W4A4):
        assert L.k3moe_expert_ffn_noalloc(s, d, ctypes.byref(wz), d, d, d, mode, None, None) == \
            k3.K3MOE_ERR_UNSUPPORTED
    for mode in (-1, 5, 99):
        assert L.k3moe_expert_ffn_noalloc(s, d, ctypes.byref(wz), d, d, d, mode, None, None) == k3.K3MOE_ERR_ARG
    big = _shape(T=4096, H=7168, I=2048, E=896, k=16)
    assert L.k3moe_expert_ffn_noalloc(big, d, ctypes.byref(wz), d, d, d, k3.K3MOE_FFN_GEMV, None, None) == \
        k3.K3MOE_ERR_NOALLOC_LIMIT
    # the limit is checked against the GEMV workspace whatever AUTO resolves to elsewhere
    mid = _shape(T=8, H=7168, I=2048, E=48, k=16)
    assert L.k3moe_workspace_bytes(mid, k3.K3MOE_OP_EXPERT_FFN, k3.K3MOE_FFN_GEMV) <= k3.K3MOE_NOALLOC_SCRATCH_BYTES
    assert L.k3moe_expert_ffn_noalloc(_shape(T=0), None, None, None, None, None, 0, None, None) == k3.K3MOE_OK
