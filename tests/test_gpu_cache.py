"""GPU tests of the expert cache (k3moe_cache_*): experts in page-locked host
memory, an LRU arena of expert slots in device memory.

Each step routes and buckets on the GPU, makes the routed experts resident, and
runs the expert FFN on the arena's tables.  Checks per step: the FFN output is
bitwise the output with the experts resident in device memory (the arena holds
the right bytes and the tables point at them); the counters (requests, raw hits,
true resident hits, bytes copied) and the slot each expert occupies follow the
reference model of the policy (oracle/cache_ref.py); non-resident experts have
NULL table entries; a step that routes to more distinct experts than there are
slots is refused and reported."""
import numpy as np
import pytest
import torch

import gen
import mxfp4_expert_ffn_router_gb300 as k3
from layer_run import alloc_layer
from oracle.cache_ref import LruArena

pytestmark = pytest.mark.gpu


def _host_store(arrs):
    """Page-locked host copies of the stacked expert arrays, and a Weights whose
    device tables point at them."""
    pinned = [torch.from_numpy(np.ascontiguousarray(a)).pin_memory() for a in arrs]
    E = arrs[0].shape[0]
    ptrs = [(t.data_ptr() + t[0].numel() * torch.arange(E, dtype=torch.int64)).cuda() for t in pinned]
    return k3.Weights(ptrs, keep=pinned), pinned


def _tables(cache, E):
    """The arena's four pointer tables as int64 [4, E] (read from the arena tensor)."""
    c = cache.weights._c
    base = cache.arena.data_ptr()
    out = []
    for addr in (c.w13_codes, c.w13_scales, c.w2_codes, c.w2_scales):
        off = addr - base
        out.append(cache.arena[off: off + 8 * E].view(torch.int64).cpu().numpy())
    return np.stack(out)


@pytest.mark.parametrize("T,H,I,E,k,S", [(2, 256, 128, 40, 4, 12), (1, 7168, 2048, 64, 16, 20)])
def test_cache_steps_follow_the_policy_and_feed_the_ffn(T, H, I, E, k, S):
    s = gen.Shape(T, H, I, E, k)
    arrs = gen.expert_arrays(H, I, 0, E)
    host_w, _keep = _host_store(arrs)
    dev_w = k3.Weights.from_stacked(*[torch.from_numpy(a).cuda() for a in arrs])
    arena = torch.empty(k3.ExpertCache.bytes_needed(s, S), dtype=torch.uint8, device="cuda")
    cache = k3.ExpertCache(s, S, host_w, arena)
    stats = torch.zeros(4, dtype=torch.int64, device="cuda")
    ref = LruArena(E, S, expert_bytes=s.expert_bytes())
    b = alloc_layer(s, mode=k3.K3MOE_FFN_GEMV)
    rng = np.random.default_rng(E + S)
    xbits = gen.normal_bf16_bits(6, gen.stream(gen.KIND_X), T * H).reshape(T, H)
    x = torch.from_numpy(xbits.view(np.int16)).cuda()
    for step in range(12):
        # skew the logits so that some experts recur (hits) and others churn
        logits = rng.standard_normal((T, E)).astype(np.float32)
        logits[:, : E // 8] += 1.5
        lg = torch.from_numpy(logits).cuda()
        k3.k3moe_route(s, lg, b["idx"], b["w"], b["status"])
        k3.k3moe_bucket(s, b["idx"], b["counts"], b["offsets"], b["perm"], b["inv"], b["ws_bucket"], b["status"])
        cache.fetch(b["counts"], 0, stats, b["status"])
        Yc = torch.empty_like(b["Y"])
        k3.k3moe_expert_ffn(s, x, cache.weights, b["offsets"], b["perm"], Yc, k3.K3MOE_FFN_GEMV, b["ws_ffn"],
                            b["status"])
        k3.k3moe_expert_ffn(s, x, dev_w, b["offsets"], b["perm"], b["Y"], k3.K3MOE_FFN_GEMV, b["ws_ffn"],
                            b["status"])
        torch.cuda.synchronize()
        assert int(b["status"].item()) == 0
        np.testing.assert_array_equal(Yc.cpu().numpy().view(np.int32), b["Y"].cpu().numpy().view(np.int32))
        counts = b["counts"].cpu().numpy()
        ref.step(np.flatnonzero(counts))
        st = stats.cpu().numpy()
        assert list(st) == [ref.requests, ref.raw_hits, ref.true_hits, ref.bytes], (step, st)
        # tables: resident experts at slot addresses a + v * stride in the reference's slots, others NULL
        tab = _tables(cache, E)
        resident = sorted(ref.slot_of.items(), key=lambda kv: kv[1])
        for e in range(E):
            if e not in ref.slot_of:
                assert (tab[:, e] == 0).all(), (step, e)
        if len(resident) >= 2:
            (e0, v0), (e1, v1) = resident[0], resident[-1]
            stride = (int(tab[0, e1]) - int(tab[0, e0])) // (v1 - v0)
            assert stride >= s.expert_bytes()
            for e, v in resident:
                assert int(tab[0, e]) == int(tab[0, e0]) + (v - v0) * stride, (step, e)
    assert ref.true_hits > 0 and ref.bytes > 0  # both paths exercised


def test_cache_refuses_a_step_with_more_experts_than_slots():
    s = gen.Shape(4, 256, 128, 32, 4)
    arrs = gen.expert_arrays(256, 128, 0, 32)
    host_w, _keep = _host_store(arrs)
    arena = torch.empty(k3.ExpertCache.bytes_needed(s, 6), dtype=torch.uint8, device="cuda")
    cache = k3.ExpertCache(s, 6, host_w, arena)
    stats = torch.zeros(4, dtype=torch.int64, device="cuda")
    b = alloc_layer(s)
    idx = torch.arange(16, dtype=torch.int32, device="cuda").reshape(4, 4)  # 16 distinct experts > 6 slots
    k3.k3moe_bucket(s, idx, b["counts"], b["offsets"], b["perm"], b["inv"], b["ws_bucket"], b["status"])
    cache.fetch(b["counts"], 0, stats, b["status"])
    torch.cuda.synchronize()
    assert int(b["status"].item()) == k3.K3MOE_DEV_BOUNDS
    assert stats.cpu().numpy().tolist() == [0, 0, 0, 0]
    assert (_tables(cache, 32) == 0).all()
