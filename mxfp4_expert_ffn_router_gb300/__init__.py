"""GB300 (sm_103a) routed MoE expert FFN with MXFP4 experts -- Python binding.

Thin ctypes marshalling over the C ABI in ``include/k3moe.h`` (``libk3moe.so``):
the functions below take torch CUDA tensors, check dtype/device/contiguity,
and pass raw pointers and the current CUDA stream.  Every step of the path runs
in the library's CUDA kernels; there is no CPU or PyTorch fallback -- if the
library is missing or the device is not sm_103 the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libk3moe.so")
_lock = threading.Lock()
_lib = None

K3MOE_OK, K3MOE_ERR_ARG, K3MOE_ERR_SHAPE, K3MOE_ERR_ALIGN = 0, -1, -2, -3
K3MOE_ERR_WORKSPACE, K3MOE_ERR_ARCH, K3MOE_ERR_LAUNCH, K3MOE_ERR_UNSUPPORTED = -4, -5, -6, -7
K3MOE_ERR_NOALLOC_LIMIT = -8
K3MOE_NOALLOC_SCRATCH_BYTES = 8 << 20
K3MOE_DEV_NONFINITE, K3MOE_DEV_BOUNDS, K3MOE_DEV_TIMEOUT = 1, 2, 4
K3MOE_FFN_AUTO, K3MOE_FFN_GEMV, K3MOE_FFN_STREAM, K3MOE_FFN_GEMM, K3MOE_FFN_W4A4 = 0, 1, 2, 3, 4
K3MOE_OP_BUCKET, K3MOE_OP_EXPERT_FFN, K3MOE_OP_LAYER = 1, 2, 3


class K3moeError(RuntimeError):
    def __init__(self, fn: str, code: int):
        msg = f"{fn}: {status_string(code)} ({code})"
        if code == K3MOE_ERR_LAUNCH:
            msg += f": {lib().k3moe_last_cuda_error().decode()}"
        super().__init__(msg)
        self.code = code


class Shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32)]

    @classmethod
    def of(cls, s) -> "Shape":
        return s if isinstance(s, Shape) else cls(s.T, s.H, s.I, s.E, s.k)


class _WeightsC(ctypes.Structure):
    _fields_ = [("w13_codes", ctypes.c_void_p), ("w13_scales", ctypes.c_void_p),
                ("w2_codes", ctypes.c_void_p), ("w2_scales", ctypes.c_void_p)]


def library_path() -> str:
    return _SO


def lib():
    """Load libk3moe.so (built by ``build.build()``); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_SO):
                raise ImportError(f"libk3moe.so not built ({_SO}); run "
                                  "python -m mxfp4_expert_ffn_router_gb300.build")
            L = ctypes.CDLL(_SO)
            vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            L.k3moe_workspace_bytes.restype = sz
            L.k3moe_workspace_bytes.argtypes = [Shape, i32, i32]
            L.k3moe_workspace_h_offset.restype = sz
            L.k3moe_workspace_h_offset.argtypes = [Shape, i32]
            L.k3moe_route.restype = i32
            L.k3moe_route.argtypes = [Shape, vp, vp, vp, vp, vp]
            L.k3moe_router.restype = i32
            L.k3moe_router.argtypes = [Shape, vp, vp, vp, vp, vp, vp, vp]
            L.k3moe_bucket.restype = i32
            L.k3moe_bucket.argtypes = [Shape, vp, vp, vp, vp, vp, vp, sz, vp, vp]
            L.k3moe_expert_ffn.restype = i32
            L.k3moe_expert_ffn.argtypes = [Shape, vp, ctypes.POINTER(_WeightsC), vp, vp, vp, i32, vp,
                                           sz, vp, vp]
            L.k3moe_expert_ffn_noalloc.restype = i32
            L.k3moe_expert_ffn_noalloc.argtypes = [Shape, vp, ctypes.POINTER(_WeightsC), vp, vp, vp, i32,
                                                   vp, vp]
            L.k3moe_cache_bytes.restype = sz
            L.k3moe_cache_bytes.argtypes = [Shape, i32]
            L.k3moe_cache_weights.restype = i32
            L.k3moe_cache_weights.argtypes = [Shape, i32, vp, ctypes.POINTER(_WeightsC)]
            L.k3moe_cache_init.restype = i32
            L.k3moe_cache_init.argtypes = [Shape, i32, vp, sz, vp]
            L.k3moe_cache_fetch.restype = i32
            L.k3moe_cache_fetch.argtypes = [Shape, i32, vp, sz, ctypes.POINTER(_WeightsC), vp, i32, i32, vp, vp,
                                             vp]
            L.k3moe_quantize_mxfp4.restype = i32
            L.k3moe_quantize_mxfp4.argtypes = [ctypes.c_int64, vp, vp, vp, vp]
            L.k3moe_combine.restype = i32
            L.k3moe_combine.argtypes = [Shape, vp, vp, vp, vp, vp, vp]
            L.k3moe_combine_residual.restype = i32
            L.k3moe_combine_residual.argtypes = [Shape, vp, vp, vp, vp, vp, vp, vp]
            L.k3moe_layer.restype = i32
            L.k3moe_layer.argtypes = [Shape, vp, vp, ctypes.POINTER(_WeightsC), vp, vp, vp, vp, vp, vp, vp, vp, vp, i32,
                                      vp, sz, vp, vp]
            L.k3moe_selftest_bounded_wait.restype = i32
            L.k3moe_selftest_bounded_wait.argtypes = [vp, vp, vp]
            L.k3moe_status_string.restype = ctypes.c_char_p
            L.k3moe_status_string.argtypes = [i32]
            L.k3moe_last_cuda_error.restype = ctypes.c_char_p
            L.k3moe_last_cuda_error.argtypes = []
            _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().k3moe_status_string(code).decode()


_BF16 = (torch.bfloat16, torch.int16)  # bf16 values, or their bit patterns


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    ok = dtype is None or (t.dtype in dtype if isinstance(dtype, tuple) else t.dtype == dtype)
    if not ok:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return t.data_ptr() if t.numel() else None


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(fn, rc):
    if rc != K3MOE_OK:
        raise K3moeError(fn, rc)


class Weights:
    """MXFP4 expert weights as the four device-resident arrays of E pointers.

    ``ptrs`` is a list of four int64 CUDA tensors [E] (0 = absent expert) in the
    order (w13 codes, w13 scales, w2 codes, w2 scales).  ``keep`` holds the
    tensors the pointers refer to."""

    def __init__(self, ptrs, keep=()):
        self.ptrs = [p.to(torch.int64).contiguous() for p in ptrs]
        self.keep = list(keep)
        self._c = _WeightsC(*[p.data_ptr() for p in self.ptrs])

    @classmethod
    def from_stacked(cls, w13c, w13s, w2c, w2s, present=None):
        """Build from four uint8 CUDA tensors [E, ...]; ``present`` (bool [E]) marks absent experts."""
        E = w13c.shape[0]
        ptrs = []
        for t in (w13c, w13s, w2c, w2s):
            assert t.is_cuda and t.dtype == torch.uint8 and t.is_contiguous() and t.shape[0] == E
            stride = t[0].numel()
            p = t.data_ptr() + stride * torch.arange(E, dtype=torch.int64)
            if present is not None:
                p = torch.where(torch.as_tensor(present, dtype=torch.bool), p, torch.zeros_like(p))
            ptrs.append(p.to(t.device))
        return cls(ptrs, keep=(w13c, w13s, w2c, w2s))

    def cstruct(self):
        return ctypes.byref(self._c)


def k3moe_workspace_bytes(shape, op: int, mode: int = 0) -> int:
    return int(lib().k3moe_workspace_bytes(Shape.of(shape), op, mode))


def k3moe_workspace_h_offset(shape, mode: int = 0) -> int:
    """Byte offset of h (bf16 [A, I], bucket order) in the expert FFN workspace."""
    v = int(lib().k3moe_workspace_h_offset(Shape.of(shape), mode))
    return -1 if v == (1 << 64) - 1 else v


def k3moe_route(shape, logits, idx, w, dev_status=None, stream=None):
    rc = lib().k3moe_route(Shape.of(shape), _ptr(logits, torch.float32, "logits"),
                           _ptr(idx, torch.int32, "idx"), _ptr(w, torch.float32, "w"),
                           _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check("k3moe_route", rc)


def k3moe_router(shape, x, wr, logits, idx, w, dev_status=None, stream=None):
    """Router scores logits [T, E] = x [T, H] . wr [E, H]^T (bf16 in, fp32 out),
    then the top-k route on them (idx, w)."""
    rc = lib().k3moe_router(Shape.of(shape), _ptr(x, _BF16, "x"), _ptr(wr, _BF16, "wr"),
                            _ptr(logits, torch.float32, "logits"), _ptr(idx, torch.int32, "idx"),
                            _ptr(w, torch.float32, "w"), _ptr(dev_status, torch.int32, "dev_status"),
                            _stream(stream))
    _check("k3moe_router", rc)


def k3moe_bucket(shape, idx, counts, offsets, perm, inv, ws=None, dev_status=None, stream=None):
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    rc = lib().k3moe_bucket(Shape.of(shape), _ptr(idx, torch.int32, "idx"),
                            _ptr(counts, torch.int32, "counts"), _ptr(offsets, torch.int32, "offsets"),
                            _ptr(perm, torch.int32, "perm"), _ptr(inv, torch.int32, "inv"),
                            _ptr(ws, None, "ws"), ws_bytes, _ptr(dev_status, torch.int32, "dev_status"),
                            _stream(stream))
    _check("k3moe_bucket", rc)


def k3moe_expert_ffn(shape, x, weights: Weights, offsets, perm, Y, mode=K3MOE_FFN_AUTO, ws=None,
                     dev_status=None, stream=None):
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    rc = lib().k3moe_expert_ffn(Shape.of(shape), _ptr(x, _BF16, "x"), weights.cstruct(),
                                _ptr(offsets, torch.int32, "offsets"), _ptr(perm, torch.int32, "perm"),
                                _ptr(Y, torch.float32, "Y"), mode, _ptr(ws, None, "ws"), ws_bytes,
                                _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check("k3moe_expert_ffn", rc)


def k3moe_expert_ffn_noalloc(shape, x, weights: Weights, offsets, perm, Y, mode=K3MOE_FFN_AUTO,
                             dev_status=None, stream=None):
    """k3moe_expert_ffn with its scratch in the library's fixed device array (no
    workspace argument), for callers that cannot allocate device memory."""
    rc = lib().k3moe_expert_ffn_noalloc(Shape.of(shape), _ptr(x, _BF16, "x"), weights.cstruct(),
                                        _ptr(offsets, torch.int32, "offsets"),
                                        _ptr(perm, torch.int32, "perm"), _ptr(Y, torch.float32, "Y"),
                                        mode, _ptr(dev_status, torch.int32, "dev_status"),
                                        _stream(stream))
    _check("k3moe_expert_ffn_noalloc", rc)


class ExpertCache:
    """Host-resident experts with a least-recently-used arena of expert slots in
    device memory (k3moe_cache_*).  ``host`` is a Weights whose pointer tables
    (device tensors) point at page-locked host arrays; ``arena`` is a uint8 CUDA
    tensor of at least k3moe_cache_bytes(shape, slots) bytes."""

    def __init__(self, shape, slots: int, host: "Weights", arena, stream=None):
        self.shape, self.slots, self.host, self.arena = Shape.of(shape), int(slots), host, arena
        self.nbytes = arena.numel() * arena.element_size()
        _check("k3moe_cache_init", lib().k3moe_cache_init(self.shape, self.slots, _ptr(arena, torch.uint8, "arena"),
                                                           self.nbytes, _stream(stream)))
        wc = _WeightsC()
        _check("k3moe_cache_weights", lib().k3moe_cache_weights(self.shape, self.slots, arena.data_ptr(),
                                                                ctypes.byref(wc)))
        self.weights = Weights.__new__(Weights)
        self.weights.ptrs, self.weights.keep, self.weights._c = [], [arena], wc

    @staticmethod
    def bytes_needed(shape, slots: int) -> int:
        return int(lib().k3moe_cache_bytes(Shape.of(shape), int(slots)))

    def fetch(self, counts, base: int = 0, stats=None, dev_status=None, stream=None):
        """Make the step's routed experts resident: expert base + i for counts[i] > 0
        (counts: int32 from k3moe_bucket)."""
        rc = lib().k3moe_cache_fetch(self.shape, self.slots, self.arena.data_ptr(), self.nbytes,
                                     self.host.cstruct(), _ptr(counts, torch.int32, "counts"), int(base),
                                     int(counts.numel()), _ptr(stats, torch.int64, "stats"),
                                     _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
        _check("k3moe_cache_fetch", rc)

    def layer_weights(self, layer: int, experts_per_layer: int) -> "Weights":
        """The device tables of one layer of a stack (offset by layer * experts_per_layer)."""
        w = Weights.__new__(Weights)
        off = 8 * layer * experts_per_layer
        c = self.weights._c
        w.ptrs, w.keep = [], [self.arena]
        w._c = _WeightsC(c.w13_codes + off, c.w13_scales + off, c.w2_codes + off, c.w2_scales + off)
        return w


def k3moe_quantize_mxfp4(x, codes, scales, stream=None):
    """MXFP4 quantisation of bf16 values x [n] (n a multiple of 32) into codes
    uint8 [n/2] (low nibble = even element) and E8M0 scales uint8 [n/32]."""
    n = x.numel() if isinstance(x, torch.Tensor) else 0
    rc = lib().k3moe_quantize_mxfp4(n, _ptr(x, _BF16, "x"), _ptr(codes, torch.uint8, "codes"),
                                    _ptr(scales, torch.uint8, "scales"), _stream(stream))
    _check("k3moe_quantize_mxfp4", rc)


def k3moe_selftest_bounded_wait(dev_status, dev_elapsed_ns, stream=None):
    """A bounded mbarrier wait that nothing completes: ORs K3MOE_DEV_TIMEOUT into
    dev_status (int32) and writes the wait's duration in ns to dev_elapsed_ns (int64)."""
    _check("k3moe_selftest_bounded_wait",
           lib().k3moe_selftest_bounded_wait(_ptr(dev_status, torch.int32, "dev_status"),
                                             _ptr(dev_elapsed_ns, torch.int64, "dev_elapsed_ns"), _stream(stream)))


def k3moe_combine(shape, Y, w, inv, out, out_f32=None, stream=None):
    rc = lib().k3moe_combine(Shape.of(shape), _ptr(Y, torch.float32, "Y"), _ptr(w, torch.float32, "w"),
                             _ptr(inv, torch.int32, "inv"), _ptr(out, _BF16, "out"),
                             _ptr(out_f32, torch.float32, "out_f32"), _stream(stream))
    _check("k3moe_combine", rc)


def k3moe_combine_residual(shape, Y, w, inv, residual, out, out_f32=None, stream=None):
    """out = bf16(residual + sum_j w[t, j] Y[inv[t k + j]]) (out may be residual)."""
    rc = lib().k3moe_combine_residual(Shape.of(shape), _ptr(Y, torch.float32, "Y"), _ptr(w, torch.float32, "w"),
                                      _ptr(inv, torch.int32, "inv"), _ptr(residual, _BF16, "residual"),
                                      _ptr(out, _BF16, "out"), _ptr(out_f32, torch.float32, "out_f32"),
                                      _stream(stream))
    _check("k3moe_combine_residual", rc)


def k3moe_layer(shape, logits, x, weights: Weights, idx, w, counts, offsets, perm, inv, Y, out, out_f32=None,
                mode=K3MOE_FFN_AUTO, ws=None, dev_status=None, stream=None):
    """route -> bucket -> expert FFN -> combine in one call (one workspace of
    k3moe_workspace_bytes(shape, K3MOE_OP_LAYER, mode) bytes)."""
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    rc = lib().k3moe_layer(Shape.of(shape), _ptr(logits, torch.float32, "logits"), _ptr(x, _BF16, "x"),
                           weights.cstruct(), _ptr(idx, torch.int32, "idx"), _ptr(w, torch.float32, "w"),
                           _ptr(counts, torch.int32, "counts"), _ptr(offsets, torch.int32, "offsets"),
                           _ptr(perm, torch.int32, "perm"), _ptr(inv, torch.int32, "inv"), _ptr(Y, torch.float32, "Y"),
                           _ptr(out, _BF16, "out"), _ptr(out_f32, torch.float32, "out_f32"), mode,
                           _ptr(ws, None, "ws"), ws_bytes, _ptr(dev_status, torch.int32, "dev_status"),
                           _stream(stream))
    _check("k3moe_layer", rc)
