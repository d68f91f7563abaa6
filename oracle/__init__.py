"""ORACLE for the routed MoE expert FFN -- test infrastructure only.

A plain, slow, single-threaded C99 implementation (``k3moe_ref.c``) of what the
hot path computes, accumulating in float64, plus this ctypes wrapper.  Only the
tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may use
it; the CUDA library never does.  It shares no code with the CUDA sources.

Pins: every function here is checked by ``tests/test_oracle_*.py`` against
closed forms, brute force, library routines and hand-worked examples.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libk3ref.so")
_lock = threading.Lock()
_lib = None


class Shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32)]


def build(force: bool = False) -> str:
    """Compile libk3ref.so (gcc, C99, -ffp-contract=off so no fused multiply-add)."""
    src = os.path.join(_HERE, "k3moe_ref.c")
    hdr = os.path.join(_HERE, "k3moe_ref.h")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < max(
            os.path.getmtime(src), os.path.getmtime(hdr)):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-Wall", "-Wextra",
                               "-Werror", "-ffp-contract=off", "-o", tmp, src, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            vp, i32 = ctypes.c_void_p, ctypes.c_int
            L.k3ref_e2m1.restype = ctypes.c_double
            L.k3ref_e2m1.argtypes = [ctypes.c_uint]
            L.k3ref_e8m0.restype = ctypes.c_double
            L.k3ref_e8m0.argtypes = [ctypes.c_uint]
            L.k3ref_bf16_value.restype = ctypes.c_double
            L.k3ref_bf16_value.argtypes = [ctypes.c_uint16]
            L.k3ref_bf16_rne.restype = ctypes.c_uint16
            L.k3ref_bf16_rne.argtypes = [ctypes.c_double]
            L.k3ref_silu.restype = ctypes.c_double
            L.k3ref_silu.argtypes = [ctypes.c_double]
            L.k3ref_quant_mxfp4.argtypes = [vp, i32, vp, vp]
            L.k3ref_route.restype = i32
            L.k3ref_route.argtypes = [Shape, vp, vp, vp, vp]
            L.k3ref_bucket.restype = i32
            L.k3ref_bucket.argtypes = [Shape, vp, vp, vp, vp, vp]
            L.k3ref_expert_ffn.restype = i32
            L.k3ref_expert_ffn.argtypes = [Shape, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp]
            L.k3ref_expert_gateup.restype = i32
            L.k3ref_expert_gateup.argtypes = [Shape, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp]
            L.k3ref_expert_down.restype = i32
            L.k3ref_expert_down.argtypes = [Shape, vp, vp, vp, vp, vp, vp, i32, vp]
            L.k3ref_combine.restype = i32
            L.k3ref_combine.argtypes = [Shape, vp, vp, vp, vp, vp]
            L.k3ref_moe_token.restype = i32
            L.k3ref_moe_token.argtypes = [Shape, vp, vp, vp, vp, vp, vp, vp, i32, vp]
            L.k3ref_router_logits.restype = i32
            L.k3ref_router_logits.argtypes = [Shape, vp, vp, vp]
            L.k3ref_router.restype = i32
            L.k3ref_router.argtypes = [Shape, vp, vp, vp, vp, vp, vp, vp]
            L.k3ref_moe_layer.restype = i32
            L.k3ref_moe_layer.argtypes = [Shape, vp, vp, vp, vp, vp, vp, i32, vp, vp]
            _lib = L
    return _lib


def _shape(s) -> Shape:
    return Shape(s.T, s.H, s.I, s.E, s.k)


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


class Weights:
    """Host MXFP4 expert weights as four E-long arrays of pointers (0 = absent).

    ``experts`` maps an expert id to its (w13 codes, w13 scales, w2 codes,
    w2 scales) numpy arrays; the arrays are kept alive by this object."""

    def __init__(self, E: int, experts: dict):
        self._keep = []
        self.ptrs = [np.zeros(E, dtype=np.uintp) for _ in range(4)]
        for e, tensors in experts.items():
            for q in range(4):
                if tensors[q] is None:
                    continue
                a = np.ascontiguousarray(tensors[q], dtype=np.uint8)
                self._keep.append(a)
                self.ptrs[q][e] = a.ctypes.data

    def args(self):
        return [p.ctypes.data for p in self.ptrs]


def e2m1(code: int) -> float:
    return lib().k3ref_e2m1(code)


def e8m0(byte: int) -> float:
    return lib().k3ref_e8m0(byte)


def bf16_value(bits: int) -> float:
    return lib().k3ref_bf16_value(bits)


def bf16_rne(v: float) -> int:
    return lib().k3ref_bf16_rne(v)


def silu(z: float) -> float:
    return lib().k3ref_silu(z)


def quant_mxfp4(v_bits: np.ndarray):
    v = _c(v_bits, np.uint16).ravel()
    assert v.size % 32 == 0
    codes = np.zeros(v.size // 2, np.uint8)
    scales = np.zeros(v.size // 32, np.uint8)
    lib().k3ref_quant_mxfp4(v.ctypes.data, v.size, codes.ctypes.data, scales.ctypes.data)
    return codes, scales


def route(s, logits: np.ndarray):
    l = _c(logits, np.float32)
    idx = np.zeros((s.T, s.k), np.int32)
    w = np.zeros((s.T, s.k), np.float64)
    bad = np.zeros(s.T, np.int32)
    n = lib().k3ref_route(_shape(s), l.ctypes.data, idx.ctypes.data, w.ctypes.data, bad.ctypes.data)
    if n < 0:
        raise ValueError("k3ref_route: bad shape")
    return idx, w, bad


def router_logits(s, x_bits: np.ndarray, wr_bits: np.ndarray) -> np.ndarray:
    """float64 [T, E]: x [T, H] (bf16 bits) times the router rows wr [E, H] (bf16 bits)."""
    x = _c(x_bits, np.uint16)
    wr = _c(wr_bits, np.uint16)
    out = np.zeros((s.T, s.E), np.float64)
    if lib().k3ref_router_logits(_shape(s), x.ctypes.data, wr.ctypes.data, out.ctypes.data) != 0:
        raise ValueError("k3ref_router_logits: bad shape")
    return out


def router(s, x_bits: np.ndarray, wr_bits: np.ndarray):
    """Router then route: (logits float64, logits float32, idx, w, row_bad)."""
    x = _c(x_bits, np.uint16)
    wr = _c(wr_bits, np.uint16)
    l64 = np.zeros((s.T, s.E), np.float64)
    l32 = np.zeros((s.T, s.E), np.float32)
    idx = np.zeros((s.T, s.k), np.int32)
    w = np.zeros((s.T, s.k), np.float64)
    bad = np.zeros(s.T, np.int32)
    n = lib().k3ref_router(_shape(s), x.ctypes.data, wr.ctypes.data, l64.ctypes.data, l32.ctypes.data,
                           idx.ctypes.data, w.ctypes.data, bad.ctypes.data)
    if n < 0:
        raise ValueError("k3ref_router: bad shape")
    return l64, l32, idx, w, bad


def bucket(s, idx: np.ndarray):
    i = _c(idx, np.int32)
    counts = np.zeros(s.E, np.int32)
    offsets = np.zeros(s.E + 1, np.int32)
    perm = np.zeros(s.T * s.k, np.int32)
    inv = np.zeros(s.T * s.k, np.int32)
    if lib().k3ref_bucket(_shape(s), i.ctypes.data, counts.ctypes.data, offsets.ctypes.data,
                          perm.ctypes.data, inv.ctypes.data) != 0:
        raise ValueError("k3ref_bucket: bad arguments")
    return counts, offsets, perm, inv


def expert_ffn(s, x_bits: np.ndarray, weights: Weights, offsets: np.ndarray, perm: np.ndarray,
               a4: bool = False, want_h: bool = False):
    x = _c(x_bits, np.uint16)
    o = _c(offsets, np.int32)
    p = _c(perm, np.int32)
    A = s.T * s.k
    Y = np.zeros((A, s.H), np.float64)
    h = np.zeros((A, s.I), np.uint16) if want_h else None
    rc = lib().k3ref_expert_ffn(_shape(s), x.ctypes.data, *weights.args(), o.ctypes.data,
                                p.ctypes.data, int(a4), Y.ctypes.data,
                                h.ctypes.data if want_h else None)
    if rc != 0:
        raise ValueError("k3ref_expert_ffn: bad arguments")
    return (Y, h) if want_h else Y


def expert_gateup(s, x_bits: np.ndarray, weights: Weights, offsets: np.ndarray, perm: np.ndarray,
                  a4: bool = False, sums: bool = False):
    """(hpre float64 [A, I], h bf16 bits uint16 [A, I]) in bucket order; with sums
    also a dict of g, u, gabs = sum |Wg x|, uabs = sum |Wu x| (float64 [A, I])."""
    x = _c(x_bits, np.uint16)
    o = _c(offsets, np.int32)
    p = _c(perm, np.int32)
    A = s.T * s.k
    hpre = np.zeros((A, s.I), np.float64)
    h = np.zeros((A, s.I), np.uint16)
    extra = {k: np.zeros((A, s.I), np.float64) for k in ("g", "u", "gabs", "uabs")} if sums else None
    ptr = [extra[k].ctypes.data for k in ("g", "u", "gabs", "uabs")] if sums else [None] * 4
    if lib().k3ref_expert_gateup(_shape(s), x.ctypes.data, *weights.args(), o.ctypes.data, p.ctypes.data,
                                 int(a4), hpre.ctypes.data, h.ctypes.data, *ptr) != 0:
        raise ValueError("k3ref_expert_gateup: bad arguments")
    return (hpre, h, extra) if sums else (hpre, h)


def expert_down(s, h_bits: np.ndarray, weights: Weights, offsets: np.ndarray, a4: bool = False):
    """Y float64 [A, H] = W2 h for the given bf16 h rows [A, I] in bucket order."""
    h = _c(h_bits, np.uint16)
    o = _c(offsets, np.int32)
    Y = np.zeros((s.T * s.k, s.H), np.float64)
    if lib().k3ref_expert_down(_shape(s), h.ctypes.data, *weights.args(), o.ctypes.data, int(a4),
                               Y.ctypes.data) != 0:
        raise ValueError("k3ref_expert_down: bad arguments")
    return Y


def combine(s, Y: np.ndarray, w: np.ndarray, inv: np.ndarray):
    Yc = _c(Y, np.float64)
    wc = _c(w, np.float64)
    ic = _c(inv, np.int32)
    out = np.zeros((s.T, s.H), np.float64)
    ob = np.zeros((s.T, s.H), np.uint16)
    if lib().k3ref_combine(_shape(s), Yc.ctypes.data, wc.ctypes.data, ic.ctypes.data,
                           out.ctypes.data, ob.ctypes.data) != 0:
        raise ValueError("k3ref_combine: bad arguments")
    return out, ob


def moe_token(s, x_row: np.ndarray, idx_row: np.ndarray, w_row: np.ndarray, weights: Weights,
              a4: bool = False) -> np.ndarray:
    x = _c(x_row, np.uint16)
    i = _c(idx_row, np.int32)
    w = _c(w_row, np.float64)
    out = np.zeros(s.H, np.float64)
    if lib().k3ref_moe_token(_shape(s), x.ctypes.data, i.ctypes.data, w.ctypes.data,
                             *weights.args(), int(a4), out.ctypes.data) != 0:
        raise ValueError("k3ref_moe_token: bad arguments")
    return out


def moe_layer(s, logits: np.ndarray, x_bits: np.ndarray, weights: Weights, a4: bool = False):
    l = _c(logits, np.float32)
    x = _c(x_bits, np.uint16)
    out = np.zeros((s.T, s.H), np.float64)
    ob = np.zeros((s.T, s.H), np.uint16)
    if lib().k3ref_moe_layer(_shape(s), l.ctypes.data, x.ctypes.data, *weights.args(), int(a4),
                             out.ctypes.data, ob.ctypes.data) != 0:
        raise ValueError("k3ref_moe_layer: bad arguments")
    return out, ob
