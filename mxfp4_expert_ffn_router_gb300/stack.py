"""A stack of routed MoE layers whose experts live in host memory, decoded
through one least-recently-used arena of expert slots in device memory.

This is the per-token expert workload of the kimi-k3-in-c engine ("running a
2.78T model in 8 GB", the expert-cache study: 92 MoE layers x 16 routed experts
= 1,472 expert requests per token, 25.83 GB of expert reads per token at a
budget too small for any expert to stay resident).  Every step runs in the
library's kernels, layer after layer on one stream: k3moe_route,
k3moe_bucket, k3moe_cache_fetch (the layer's slice of the arena's experts),
k3moe_expert_ffn on the arena's tables, k3moe_combine.  Nothing synchronises
the host inside a token.

The experts of logical layer l are host store l mod P (P physical layers held
in page-locked host memory); the arena caches logical experts (l, e), so hits,
misses and bytes are those of L distinct layers whatever P is.
"""
from __future__ import annotations


import torch

from . import (K3MOE_FFN_GEMV, K3MOE_OP_BUCKET, K3MOE_OP_EXPERT_FFN, ExpertCache, Shape, Weights,
               k3moe_bucket, k3moe_combine, k3moe_expert_ffn, k3moe_route, k3moe_workspace_bytes)


class HostExpertStore:
    """P physical layers of MXFP4 experts in page-locked host memory, stacked as
    [P * E, ...] per array, and device tables of L * E pointers (logical layer l
    -> physical l mod P)."""

    def __init__(self, H: int, I: int, E: int, P: int, L: int, fill, device="cuda"):
        shapes = [(P * E, 2 * I, H // 2), (P * E, 2 * I, H // 32), (P * E, H, I // 2), (P * E, H, I // 32)]
        self.arrays = [torch.empty(sh, dtype=torch.uint8, pin_memory=True) for sh in shapes]
        for p in range(P):  # fill(p, [four host addresses]) writes the E experts of physical layer p
            fill(p, [a[p * E].data_ptr() for a in self.arrays])
        self.H, self.I, self.E, self.P, self.L = H, I, E, P, L
        ptrs = []
        for a in self.arrays:
            per = a[0].numel()
            phys = (torch.arange(L, dtype=torch.int64) % P)[:, None] * E + torch.arange(E, dtype=torch.int64)[None, :]
            ptrs.append((a.data_ptr() + per * phys.reshape(-1)).to(device))
        self.weights = Weights(ptrs, keep=self.arrays)

    @property
    def bytes(self) -> int:
        return sum(a.numel() for a in self.arrays)


class CachedMoEStack:
    """L MoE layers of shape ``s`` (per layer: T tokens, E experts, top-k) over a
    host expert store, with an arena of ``slots`` expert slots."""

    def __init__(self, s, store: HostExpertStore, slots: int, device="cuda", mode: int = K3MOE_FFN_GEMV):
        self.s, self.store, self.slots, self.mode = Shape.of(s), store, int(slots), mode
        L, E = store.L, s.E
        self.arena_shape = Shape(s.T, s.H, s.I, L * E, s.k)
        self.arena = torch.empty(ExpertCache.bytes_needed(self.arena_shape, slots), dtype=torch.uint8, device=device)
        self.cache = ExpertCache(self.arena_shape, slots, store.weights, self.arena)
        self.layer_w = [self.cache.layer_weights(l, E) for l in range(L)]
        A = s.T * s.k
        i32, f32 = torch.int32, torch.float32
        self.stats = torch.zeros(4, dtype=torch.int64, device=device)
        self.status = torch.zeros(1, dtype=i32, device=device)
        self.idx = torch.empty((s.T, s.k), dtype=i32, device=device)
        self.w = torch.empty((s.T, s.k), dtype=f32, device=device)
        self.counts = torch.empty(E, dtype=i32, device=device)
        self.offsets = torch.empty(E + 1, dtype=i32, device=device)
        self.perm = torch.empty(A, dtype=i32, device=device)
        self.inv = torch.empty(A, dtype=i32, device=device)
        self.ws_b = torch.empty(max(1, k3moe_workspace_bytes(s, K3MOE_OP_BUCKET)), dtype=torch.uint8, device=device)
        self.ws_f = torch.empty(max(1, k3moe_workspace_bytes(s, K3MOE_OP_EXPERT_FFN, mode)), dtype=torch.uint8,
                                device=device)
        self.Y = torch.empty((A, s.H), dtype=f32, device=device)

    def layer(self, l: int, logits, x, out, out_f32=None, stream=None):
        """Layer l on one batch: logits f32 [T, E], x bf16 [T, H] -> out bf16 [T, H]."""
        s = self.s
        k3moe_route(s, logits, self.idx, self.w, self.status, stream=stream)
        k3moe_bucket(s, self.idx, self.counts, self.offsets, self.perm, self.inv, self.ws_b, self.status, stream=stream)
        self.cache.fetch(self.counts, l * s.E, self.stats, self.status, stream=stream)
        k3moe_expert_ffn(s, x, self.layer_w[l], self.offsets, self.perm, self.Y, self.mode, self.ws_f, self.status,
                         stream=stream)
        k3moe_combine(s, self.Y, self.w, self.inv, out, out_f32, stream=stream)

    def counters(self) -> dict:
        """Requests, raw hits, true resident hits and bytes copied host -> arena so far."""
        r, raw, true, by = (int(v) for v in self.stats.cpu().tolist())
        return {"requests": r, "raw_hits": raw, "true_resident_hits": true, "bytes_from_host": by}
