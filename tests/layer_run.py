"""Helpers for the GPU tests: run one MoE layer through the C ABI (binding)."""
from __future__ import annotations

import numpy as np
import torch

import mxfp4_expert_ffn_router_gb300 as k3


def alloc_layer(s, device="cuda", mode=k3.K3MOE_FFN_AUTO, with_f32=True):
    A = s.T * s.k
    i32, f32 = torch.int32, torch.float32
    bufs = dict(
        status=torch.zeros(1, dtype=i32, device=device),
        idx=torch.empty((s.T, s.k), dtype=i32, device=device),
        w=torch.empty((s.T, s.k), dtype=f32, device=device),
        counts=torch.empty(s.E, dtype=i32, device=device),
        offsets=torch.empty(s.E + 1, dtype=i32, device=device),
        perm=torch.empty(A, dtype=i32, device=device),
        inv=torch.empty(A, dtype=i32, device=device),
        ws_bucket=torch.empty(max(1, k3.k3moe_workspace_bytes(s, k3.K3MOE_OP_BUCKET)),
                              dtype=torch.uint8, device=device),
        ws_ffn=torch.empty(max(1, k3.k3moe_workspace_bytes(s, k3.K3MOE_OP_EXPERT_FFN, mode)),
                           dtype=torch.uint8, device=device),
        Y=torch.empty((A, s.H), dtype=f32, device=device),
        out=torch.empty((s.T, s.H), dtype=torch.int16, device=device),
        out_f32=torch.empty((s.T, s.H), dtype=f32, device=device) if with_f32 else None,
    )
    return bufs


def run_layer(s, logits, x, weights, bufs=None, mode=k3.K3MOE_FFN_AUTO, stream=None):
    b = bufs if bufs is not None else alloc_layer(s, logits.device, mode)
    b["mode"] = mode  # which workspace layout holds h (see ffn_check.gpu_h)
    k3.k3moe_route(s, logits, b["idx"], b["w"], b["status"], stream=stream)
    k3.k3moe_bucket(s, b["idx"], b["counts"], b["offsets"], b["perm"], b["inv"], b["ws_bucket"],
                    b["status"], stream=stream)
    k3.k3moe_expert_ffn(s, x, weights, b["offsets"], b["perm"], b["Y"], mode, b["ws_ffn"],
                        b["status"], stream=stream)
    k3.k3moe_combine(s, b["Y"], b["w"], b["inv"], b["out"], b["out_f32"], stream=stream)
    return b


def host(b):
    torch.cuda.synchronize()
    return {k: (v.cpu().numpy() if isinstance(v, torch.Tensor) else v) for k, v in b.items()}


def bf16_rne_bits_of(f32: np.ndarray) -> np.ndarray:
    """Library rounding (torch) of fp32 values to bf16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(f32, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy()


def max_rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max |got - ref| / RMS(ref) -- the tolerance measure (bar: 2e-3)."""
    rms = float(np.sqrt(np.mean(np.square(ref.astype(np.float64))))) if ref.size else 1.0
    if ref.size == 0:
        return 0.0
    return float(np.max(np.abs(got.astype(np.float64) - ref))) / (rms if rms > 0 else 1.0)
