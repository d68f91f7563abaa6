"""Staged parity of the expert FFN against the oracle.

h = bf16(silu(g) u) is the GLU expert's one rounding point: floating point
decides a bf16 code there.  The GPU sums g and u in fp32 and the oracle in
float64, so an element whose exact value lies next to a rounding midpoint can
round to either neighbour, and one such flip at a large |h| moves a whole row
of Y by up to |W2| * ulp(h) -- enough to exceed 2e-3 RMS on its own.  So the
decision is compared where it is unique and checked for validity where it is
not, and everything after it is compared with the oracle applied to the GPU's
own decision:

  (a) h: every GPU element equals the oracle's bf16 rounding, except elements
      where the two are adjacent bf16 values and the oracle's unrounded value
      lies within TAU of an ulp of their midpoint (a near-tie); such elements are
      at most MAX_FLIP_FRAC of all;
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
TAU = 0.125
MAX_FLIP_FRAC = 0.02


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
    """Order-preserving integer of bf16 bit patterns (-0 and +0 both 0): adjacent
    finite values have keys one apart."""
    b = np.asarray(bits, np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def check_h(h_gpu: np.ndarray, h_ref: np.ndarray, hpre: np.ndarray) -> dict:
    """(a): equal values, or a near-tie flip between adjacent bf16 values."""
    diff = _key(h_gpu) != _key(h_ref)
    n = int(diff.sum())
    if n:
        ka, kb = _key(h_gpu[diff]), _key(h_ref[diff])
        assert np.all(np.abs(ka - kb) == 1), f"{int((np.abs(ka - kb) != 1).sum())} h elements off by > 1 bf16 step"
        va, vb = bf16_values(h_gpu[diff]), bf16_values(h_ref[diff])
        dist = np.abs(hpre[diff] - 0.5 * (va + vb)) / np.abs(va - vb)
        assert np.all(dist <= TAU), f"a flip away from a rounding tie: {float(dist.max()):.3g} ulp from the midpoint"
    frac = n / max(1, h_ref.size)
    assert frac <= MAX_FLIP_FRAC, frac
    return {"h_flips": n, "h_flip_frac": frac}


def check_staged(s, r: dict, xbits, W, offsets, perm, w, inv, h_gpu, a4=False) -> dict:
    """Whole-layer staged check (every bucket position) with the oracle in-process."""
    hpre, h_ref = oracle.expert_gateup(s, xbits, W, offsets, perm, a4=a4)
    st = check_h(h_gpu, h_ref, hpre)
    Y = oracle.expert_down(s, h_gpu, W, offsets, a4=a4)
    out, _ = oracle.combine(s, Y, w, inv)
    st["y_err"] = max_rel_err(r["Y"], Y)
    st["out_err"] = max_rel_err(r["out_f32"], out)
    assert st["y_err"] <= TOL, st
    assert st["out_err"] <= TOL, st
    return st
