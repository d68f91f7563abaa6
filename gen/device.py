"""Device-resident copies of the synthetic workloads (torch; no MoE arithmetic).

Builds, on one CUDA device, the stacked MXFP4 expert tensors [E, ...] of a
workload from the counter-based generator, in batches of experts through a
pinned host staging buffer, plus its logits and activations."""
from __future__ import annotations

import numpy as np
import torch

from . import (CONFIGS, SCALE_HI, SCALE_LO, WEIGHT_SEED, Shape, expert_sizes, fill_experts,
               make_logits, make_x)


class DeviceExperts:
    """Stacked uint8 tensors w13c [E,2I,H/2], w13s [E,2I,H/32], w2c [E,H,I/2], w2s [E,H,I/32]."""

    def __init__(self, H: int, I: int, E: int, device="cuda", seed: int = WEIGHT_SEED,
                 batch_bytes: int = 1 << 30, slo: int = SCALE_LO, shi: int = SCALE_HI):
        self.H, self.I, self.E = H, I, E
        sz = expert_sizes(H, I)
        shapes = [(E, 2 * I, H // 2), (E, 2 * I, H // 32), (E, H, I // 2), (E, H, I // 32)]
        self.tensors = [torch.empty(s, dtype=torch.uint8, device=device) for s in shapes]
        per = sum(sz)
        nb = max(1, min(E, batch_bytes // per))
        stage = [torch.empty((nb,) + s[1:], dtype=torch.uint8).pin_memory() for s in shapes]
        for e0 in range(0, E, nb):
            e1 = min(E, e0 + nb)
            fill_experts(H, I, e0, e1, *[t.data_ptr() for t in stage], seed=seed, slo=slo, shi=shi)
            for dst, src in zip(self.tensors, stage):
                dst[e0:e1].copy_(src[: e1 - e0], non_blocking=True)
            torch.cuda.current_stream().synchronize()  # staging buffer reused next batch

    @property
    def bytes(self) -> int:
        return sum(t.numel() for t in self.tensors)

    def host_expert(self, e: int):
        """Host numpy copies of expert e's four tensors (read back from the device)."""
        return tuple(t[e].cpu().numpy() for t in self.tensors)


def device_inputs(name: str, s: Shape | None = None, device="cuda"):
    """(logits f32 [T,E], x bf16-bits int16 [T,H]) on the device plus host numpy copies."""
    s = s or CONFIGS[name]
    logits = make_logits(name, s)
    x = make_x(s)
    return (torch.from_numpy(logits).to(device), torch.from_numpy(x.view(np.int16)).to(device),
            logits, x)
