"""GPU tests of a stack of MoE layers over host-resident experts and one LRU
arena (mxfp4_expert_ffn_router_gb300.stack): every layer's output is bitwise
the output with that layer's experts resident in device memory, and is checked
in stages against the oracle (routing bit-exact, the FFN at its bf16 rounding
of h, then Y and out); the arena's counters follow the reference policy over
the logical experts (layer, expert) of the whole stack."""
import numpy as np
import pytest
import torch

import gen
import mxfp4_expert_ffn_router_gb300 as k3
import oracle
from ffn_check import check_staged, gpu_h
from layer_run import alloc_layer, host, run_layer
from mxfp4_expert_ffn_router_gb300.stack import CachedMoEStack, HostExpertStore
from oracle.cache_ref import LruArena

pytestmark = pytest.mark.gpu


def _fill(H, I, E):
    def fill(p, ptrs):
        gen.fill_experts(H, I, 0, E, *ptrs, seed=gen.WEIGHT_SEED + p)
    return fill


@pytest.mark.parametrize("L,P,T,H,I,E,k,slots", [(6, 2, 2, 256, 128, 32, 4, 16), (4, 2, 1, 7168, 1536, 64, 16, 24)])
def test_stack_layers_match_resident_experts_and_the_oracle(L, P, T, H, I, E, k, slots):
    s = gen.Shape(T, H, I, E, k)
    store = HostExpertStore(H, I, E, P, L, _fill(H, I, E))
    stack = CachedMoEStack(s, store, slots)
    ref = LruArena(L * E, slots, expert_bytes=s.expert_bytes())
    phys = [gen.expert_arrays(H, I, 0, E, seed=gen.WEIGHT_SEED + p) for p in range(P)]
    dev_w = [k3.Weights.from_stacked(*[torch.from_numpy(a).cuda() for a in arrs]) for arrs in phys]
    for tok in range(2):
        for l in range(L):
            seed = 100 + 7 * l + 1000 * tok
            logits = gen.normal_f32(seed, gen.stream(gen.KIND_LOGITS), T * E, 2.0).reshape(T, E)
            xbits = gen.normal_bf16_bits(seed, gen.stream(gen.KIND_X), T * H).reshape(T, H)
            lg = torch.from_numpy(logits).cuda()
            x = torch.from_numpy(xbits.view(np.int16)).cuda()
            out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
            out32 = torch.empty((T, H), dtype=torch.float32, device="cuda")
            stack.layer(l, lg, x, out, out32)
            torch.cuda.synchronize()
            assert int(stack.status.item()) == 0
            # the same layer with its experts resident in device memory
            r = host(run_layer(s, lg, x, dev_w[l % P], bufs=alloc_layer(s, mode=k3.K3MOE_FFN_GEMV),
                               mode=k3.K3MOE_FFN_GEMV))
            np.testing.assert_array_equal(out32.cpu().numpy().view(np.int32), r["out_f32"].view(np.int32))
            # against the oracle, staged at h (the stack's own workspace holds its h)
            idx, w, _ = oracle.route(s, logits)
            np.testing.assert_array_equal(stack.idx.cpu().numpy(), idx)
            counts, offsets, perm, inv = oracle.bucket(s, idx)
            W = oracle.Weights(E, {e: tuple(z[e] for z in phys[l % P]) for e in np.unique(idx)})
            rs = {"Y": stack.Y.cpu().numpy(), "out_f32": out32.cpu().numpy(), "mode": k3.K3MOE_FFN_GEMV}
            h = gpu_h({"ws_ffn": stack.ws_f, "mode": k3.K3MOE_FFN_GEMV}, s)
            check_staged(s, rs, xbits, W, offsets, perm, w, inv, h)
            ref.step(l * E + np.flatnonzero(counts))
            c = stack.counters()
            assert [c["requests"], c["raw_hits"], c["true_resident_hits"], c["bytes_from_host"]] == \
                [ref.requests, ref.raw_hits, ref.true_hits, ref.bytes], (tok, l)
