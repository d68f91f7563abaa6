"""Seeded synthetic inputs for the routed MoE expert FFN (shared by both sides).

This package is the only code that the oracle side and the GPU side have in
common.  It draws bytes, integers and normal variates from the counter-based
SplitMix64 generator defined in ``k3gen.h`` and arranges them into the
workloads below.  It contains none of the MoE method's arithmetic (no routing,
no decoding of MXFP4, no matmul).

Workloads (shapes T tokens, H hidden, I expert intermediate, E experts, k top-k):

* ``tiny``      T=4,    H=128,  I=64,   E=8,   k=2,  logits N(0,1)
* ``decode``    T=1,    H=7168, I=2048, E=896, k=16, logits N(0, sigma=2)
* ``batch8``    T=8,    as decode; tokens 0-3 put their 8 largest logits on one
                seeded set S of 8 experts (in S order), tokens 4-7 are plain
* ``specN``     N in {2, 4, 12, 16}: the batch8 recipe at T=N (speculative-verify
                batches); tokens 0..N/2-1 share S, the rest are plain
* ``prefill``   T=4096, as decode, logits iid N(0,1) (uniform expected load)
* ``skewed``    T=2048, logits z + 0.5 * ln p_e with p_e proportional to
                rank(e)^-1.2 over a seeded permutation of the experts
* ``decode_i1536`` the decode layer with I=1536
* ``probe``     E=16, k=1, T=32768, each expert receives exactly 2048 tokens

Router matrix (for the router entry point): bf16 [E, H], N(0, 2/sqrt(H)).

MXFP4 weights: code bytes uniform (both nibbles uniform over 0..15), e8m0 scale
bytes uniform over {119..123}, i.e. block scales 2^-8 .. 2^-4.  Activations x
are N(0,1) rounded to bf16.  Seeds: 0 for weights, 1 for activations and logits.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libk3gen.so")
_lock = threading.Lock()
_lib = None

KIND_W13_CODES, KIND_W13_SCALES, KIND_W2_CODES, KIND_W2_SCALES = 1, 2, 3, 4
KIND_X, KIND_LOGITS, KIND_AUX, KIND_ROUTER = 5, 6, 7, 8
WEIGHT_SEED, INPUT_SEED = 0, 1
SCALE_LO, SCALE_HI = 119, 123


def build(force: bool = False) -> str:
    """Compile libk3gen.so next to this file (plain C99 + pthreads)."""
    src = os.path.join(_HERE, "k3gen.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < max(
        os.path.getmtime(src), os.path.getmtime(os.path.join(_HERE, "k3gen.h"))
    ):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-Wall", "-Wextra", "-Werror",
             "-ffp-contract=off", "-o", tmp, src, "-lm", "-lpthread"]
        )
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            u64, sz, vp, i32 = ctypes.c_uint64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int
            L.k3gen_draw.restype = u64
            L.k3gen_draw.argtypes = [u64, u64, u64]
            L.k3gen_u53.restype = ctypes.c_double
            L.k3gen_u53.argtypes = [u64, u64, u64]
            L.k3gen_bytes.argtypes = [u64, u64, u64, vp, sz]
            L.k3gen_uint8_range.argtypes = [u64, u64, u64, vp, sz, i32, i32]
            L.k3gen_normal_f64.argtypes = [u64, u64, u64, vp, sz]
            L.k3gen_normal_f32.argtypes = [u64, u64, u64, vp, sz, ctypes.c_double]
            L.k3gen_normal_bf16.argtypes = [u64, u64, u64, vp, sz, ctypes.c_double]
            L.k3gen_uniform_f64.argtypes = [u64, u64, u64, vp, sz]
            L.k3gen_experts.restype = i32
            L.k3gen_experts.argtypes = [u64, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, i32]
            _lib = L
    return _lib


def stream(kind: int, sub: int = 0) -> int:
    return (int(kind) << 32) | (int(sub) & 0xFFFFFFFF)


def draws(seed: int, strm: int, first: int, n: int) -> np.ndarray:
    L = lib()
    return np.array([L.k3gen_draw(seed, strm, first + i) for i in range(n)], dtype=np.uint64)


def uniform_f64(seed: int, strm: int, n: int, first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    lib().k3gen_uniform_f64(seed, strm, first, out.ctypes.data, n)
    return out


def normal_f64(seed: int, strm: int, n: int, first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    lib().k3gen_normal_f64(seed, strm, first, out.ctypes.data, n)
    return out


def normal_f32(seed: int, strm: int, n: int, sigma: float = 1.0, first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    lib().k3gen_normal_f32(seed, strm, first, out.ctypes.data, n, float(sigma))
    return out


def normal_bf16_bits(seed: int, strm: int, n: int, sigma: float = 1.0, first: int = 0) -> np.ndarray:
    """bf16 values as their uint16 bit patterns."""
    out = np.empty(n, dtype=np.uint16)
    lib().k3gen_normal_bf16(seed, strm, first, out.ctypes.data, n, float(sigma))
    return out


def random_bytes(seed: int, strm: int, n: int, first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint8)
    lib().k3gen_bytes(seed, strm, first, out.ctypes.data, n)
    return out


@dataclass(frozen=True)
class Shape:
    T: int
    H: int
    I: int
    E: int
    k: int

    @property
    def A(self) -> int:
        return self.T * self.k

    def expert_bytes(self) -> int:
        """Packed codes + e8m0 scales of one expert: 3*H*I*(1/2 + 1/32) bytes."""
        return 3 * self.H * self.I * 17 // 32


def expert_sizes(H: int, I: int) -> tuple[int, int, int, int]:
    """Byte sizes of one expert's (w13 codes, w13 scales, w2 codes, w2 scales)."""
    return 2 * I * (H // 2), 2 * I * (H // 32), H * (I // 2), H * (I // 32)


def fill_experts(H: int, I: int, e0: int, e1: int, w13c: int, w13s: int, w2c: int, w2s: int,
                 seed: int = WEIGHT_SEED, nthreads: int | None = None,
                 slo: int = SCALE_LO, shi: int = SCALE_HI) -> None:
    """Write experts [e0, e1) back to back at the given host addresses (0 = skip)."""
    nt = nthreads if nthreads else max(1, min(32, os.cpu_count() or 1))
    rc = lib().k3gen_experts(seed, H, I, e0, e1, slo, shi, w13c or None, w13s or None,
                             w2c or None, w2s or None, nt)
    if rc != 0:
        raise ValueError("k3gen_experts: bad arguments")


def expert_arrays(H: int, I: int, e0: int, e1: int, seed: int = WEIGHT_SEED,
                  nthreads: int | None = None, slo: int = SCALE_LO, shi: int = SCALE_HI):
    """Numpy arrays (n, 2I, H/2), (n, 2I, H/32), (n, H, I/2), (n, H, I/32) for experts [e0, e1)."""
    n = e1 - e0
    a = np.empty((n, 2 * I, H // 2), np.uint8)
    b = np.empty((n, 2 * I, H // 32), np.uint8)
    c = np.empty((n, H, I // 2), np.uint8)
    d = np.empty((n, H, I // 32), np.uint8)
    fill_experts(H, I, e0, e1, a.ctypes.data, b.ctypes.data, c.ctypes.data, d.ctypes.data,
                 seed, nthreads, slo, shi)
    return a, b, c, d


def _fisher_yates(n: int, strm: int, seed: int = INPUT_SEED, m: int | None = None) -> np.ndarray:
    """First m entries of a seeded Fisher-Yates shuffle of range(n)."""
    m = n if m is None else m
    u = uniform_f64(seed, strm, m)
    p = np.arange(n, dtype=np.int64)
    for i in range(m):
        j = i + int(np.floor(u[i] * (n - i)))
        p[i], p[j] = p[j], p[i]
    return p[:m].copy()


CONFIGS = {
    "tiny": Shape(4, 128, 64, 8, 2),
    "decode": Shape(1, 7168, 2048, 896, 16),
    "batch8": Shape(8, 7168, 2048, 896, 16),
    "prefill": Shape(4096, 7168, 2048, 896, 16),
    "skewed": Shape(2048, 7168, 2048, 896, 16),
    "decode_i1536": Shape(1, 7168, 1536, 896, 16),
    "spec2": Shape(2, 7168, 2048, 896, 16),
    "spec4": Shape(4, 7168, 2048, 896, 16),
    "spec12": Shape(12, 7168, 2048, 896, 16),
    "spec16": Shape(16, 7168, 2048, 896, 16),
    "probe": Shape(32768, 7168, 2048, 16, 1),
}


def make_logits(name: str, s: Shape | None = None, seed: int = INPUT_SEED) -> np.ndarray:
    """Router logits f32 [T, E] for a workload (its recipe is in the module docstring)."""
    s = s or CONFIGS[name]
    T, E = s.T, s.E
    ls = stream(KIND_LOGITS)
    if name in ("decode", "decode_i1536"):
        return normal_f32(seed, ls, T * E, 2.0).reshape(T, E)
    if name == "batch8" or name.startswith("spec"):
        l = normal_f32(seed, ls, T * E, 2.0).reshape(T, E)
        S = _fisher_yates(E, stream(KIND_AUX, 1), seed, 8)
        rest_pos = np.setdiff1d(np.arange(E), S)  # ascending
        for t in range(T // 2):
            row = l[t]
            order = np.argsort(-row.astype(np.float64), kind="stable")
            top, rest = order[:8], np.sort(order[8:])
            new = np.empty_like(row)
            new[S] = row[top]
            new[rest_pos] = row[rest]
            l[t] = new
        return l
    if name == "skewed":
        z = normal_f32(seed, ls, T * E, 1.0).reshape(T, E).astype(np.float64)
        perm = _fisher_yates(E, stream(KIND_AUX, 2), seed)
        rank = np.empty(E, np.float64)
        rank[perm] = np.arange(1, E + 1)
        p = rank ** -1.2
        p /= p.sum()
        return (z + 0.5 * np.log(p)[None, :]).astype(np.float32)
    if name == "probe":
        z = normal_f32(seed, ls, T * E, 1.0).reshape(T, E)
        t = np.arange(T)
        z[t, t % E] = 8.0 + np.abs(z[t, t % E])
        return z
    return normal_f32(seed, ls, T * E, 1.0).reshape(T, E)


def make_router(s: Shape, seed: int = WEIGHT_SEED) -> np.ndarray:
    """Router matrix as bf16 bit patterns, uint16 [E, H] (row e scores expert e),
    N(0, sigma = 2 / sqrt(H)): with x ~ N(0, 1) the scores have standard
    deviation 2, the decode workload's logit distribution."""
    return normal_bf16_bits(seed, stream(KIND_ROUTER), s.E * s.H, 2.0 / np.sqrt(s.H)).reshape(s.E, s.H)


def make_x(s: Shape, seed: int = INPUT_SEED) -> np.ndarray:
    """Activations x as bf16 bit patterns, uint16 [T, H], N(0,1)."""
    return normal_bf16_bits(seed, stream(KIND_X), s.T * s.H, 1.0).reshape(s.T, s.H)
