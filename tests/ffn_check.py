"""Staged parity of the expert FFN against the oracle.

h = bf16(silu(g) u) is the GLU expert's one rounding point: floating point
decides a bf16 code there.  The GPU sums g and u in fp32 (its own order) and
the oracle in float64, so the two h can differ, and a single one-step difference
at a large |h| moves a row of Y by up to max|W2| * ulp(h) -- above 2e-3 RMS on
its own.  So the decision is checked for validity against a bound, and what
follows it is compared with the oracle applied to the GPU's decision:

  (a) h: every GPU element is the bf16 rounding (to nearest even) of some value
      in [hmin, hmax], the range of silu(g') u' over |g' - g| <= dg,
      |u' - u| <= du, widened by 2^-20 relative for the fp32 evaluation of
      silu(g) u; g, u are the oracle's exact sums and dg = gamma_d * sum|Wg x|,
      du = gamma_d * sum|Wu x| the standard bound of a d-deep fp32 summation
      (gamma_d = d u / (1 - d u)) with the kernel's depth d:
        GEMV / STREAM (CUDA cores, round to nearest): d = 16 + 2 + K/1024 + 5
          (16 products per half-chunk partial, its sum and the scale fma, the
          lane's chunks, the 5-level warp butterfly), with u = 2^-23 (twice the
          unit roundoff, a margin);
        GEMM W4A16 (tcgen05 kind::f16) and W4A4 (kind::mxf4): the tensor core's
          internal order and rounding are not documented, so d = K/16 + 16 (one
          step per K = 16 slice plus the slice's own sum) with u = 2^-23;
  (b) Y: the GPU's rows against the oracle's down projection of the GPU's h,
      max |err| <= 2e-3 RMS (W4A4: the oracle quantises that h to MXFP4 itself);
  (c) out: the GPU's fp32 output against the oracle's combine of (b)'s rows,
      max |err| <= 2e-3 RMS."""
from __future__ import annotations

import numpy as np
import torch

import mxfp4_expert_ffn_router_gb300 as k3
import oracle

TOL = 2e-3


def resolved_mode(s, mode):
    """The kernel family a mode runs for a shape (the library's AUTO rule)."""
    if mode != k3.K3MOE_FFN_AUTO:
        return mode
    A = s.T * s.k
    gemm_ok = s.H % 128 == 0 and s.I % 128 == 0
    return k3.K3MOE_FFN_GEMM if gemm_ok and 5 * A >= 4 * s.E else k3.K3MOE_FFN_GEMV


def gamma(s, mode) -> float:
    m = resolved_mode(s, mode)
    if m in (k3.K3MOE_FFN_GEMM, k3.K3MOE_FFN_W4A4):
        d = s.H / 16 + 16
    else:
        d = 16 + 2 + -(-s.H // 1024) + 5
    u = 2.0 ** -23
    return d * u / (1 - d * u)


def gpu_h(bufs, s, mode=None) -> np.ndarray:
    """The GPU's h (uint16 bf16 bits [A, I], bucket order) from the expert FFN
    workspace of a layer run (torch tensors or their host copies)."""
    mode = bufs["mode"] if mode is None else mode
    off = k3.k3moe_workspace_h_offset(s, mode)
    assert off >= 0
    A = s.T * s.k
    raw = bufs["ws_ffn"][off: off + A * s.I * 2]
    if isinstance(raw, torch.Tensor):
        raw = raw.cpu().numpy()
    return np.ascontiguousarray(raw).view(np.uint16).reshape(A, s.I)


def bf16_values(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def max_rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(np.square(ref.astype(np.float64)))))
    return float(np.max(np.abs(got.astype(np.float64) - ref))) / (rms if rms > 0 else 1.0)


def _key(bits: np.ndarray) -> np.ndarray:
    """Order-preserving integer of bf16 bit patterns (-0 and +0 both 0)."""
    b = np.asarray(bits, np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def _bf16_directed(v: np.ndarray, up: bool) -> np.ndarray:
    """Keys of the bf16 values next to v: the largest <= v (up=False) or the
    smallest >= v (up=True), through float32 nearest plus a correction step."""
    v = np.asarray(v, np.float64)
    f = v.astype(np.float32)
    if up:
        f = np.where(f.astype(np.float64) < v, np.nextafter(f, np.float32(np.inf)), f)
    else:
        f = np.where(f.astype(np.float64) > v, np.nextafter(f, np.float32(-np.inf)), f)
    bits = np.ascontiguousarray(f, np.float32).view(np.uint32)
    hi = (bits >> 16).astype(np.int64)
    low = bits & 0xFFFF
    neg = (bits >> 31) == 1
    mag = hi & 0x7FFF
    key = np.where(neg, -mag, mag)
    inexact = low != 0  # dropping the low 16 bits moved toward zero
    if up:
        key = np.where(inexact & ~neg, key + 1, key)
    else:
        key = np.where(inexact & neg, key - 1, key)
    return key


def _silu(z):
    return z / (1.0 + np.exp(-z))


ZMIN = -1.2784645427610738  # argmin of silu


def check_h(h_gpu: np.ndarray, sums: dict, g_bound: float) -> dict:
    """(a): each GPU h is a bf16 rounding of a value silu(g') u' within the bound."""
    g, u = sums["g"], sums["u"]
    dg, du = g_bound * sums["gabs"], g_bound * sums["uabs"]
    corners = [_silu(g + sg * dg) * (u + su * du) for sg in (-1, 1) for su in (-1, 1)]
    # silu's minimum inside [g - dg, g + dg] extends the range
    inside = (g - dg <= ZMIN) & (ZMIN <= g + dg)
    sm = _silu(ZMIN)
    corners += [np.where(inside, sm * (u - du), corners[0]), np.where(inside, sm * (u + du), corners[0])]
    lo = np.minimum.reduce(corners)
    hi = np.maximum.reduce(corners)
    lo = lo - 2.0 ** -20 * np.abs(lo)
    hi = hi + 2.0 ** -20 * np.abs(hi)
    k = _key(h_gpu)
    bad = (k < _bf16_directed(lo, up=False)) | (k > _bf16_directed(hi, up=True))
    nbad = int(bad.sum())
    if nbad:
        i = int(np.flatnonzero(bad.ravel())[0])
        raise AssertionError(f"{nbad} h elements outside their bound; first at {np.unravel_index(i, h_gpu.shape)}: "
                             f"gpu {float(bf16_values(h_gpu.ravel()[i:i + 1])[0])!r}, range "
                             f"[{float(lo.ravel()[i])!r}, {float(hi.ravel()[i])!r}]")
    return {"h_elements": int(h_gpu.size)}


def check_staged(s, r: dict, xbits, W, offsets, perm, w, inv, h_gpu, a4=False, mode=None) -> dict:
    """Whole-layer staged check (every bucket position) with the oracle in-process."""
    mode = r["mode"] if mode is None else mode
    hpre, h_ref, sums = oracle.expert_gateup(s, xbits, W, offsets, perm, a4=a4, sums=True)
    st = check_h(h_gpu, sums, gamma(s, mode))
    st["h_differs"] = int((h_gpu != h_ref).sum())
    Y = oracle.expert_down(s, h_gpu, W, offsets, a4=a4)
    out, _ = oracle.combine(s, Y, w, inv)
    st["y_err"] = max_rel_err(r["Y"], Y)
    st["out_err"] = max_rel_err(r["out_f32"], out)
    assert st["y_err"] <= TOL, st
    assert st["out_err"] <= TOL, st
    return st
