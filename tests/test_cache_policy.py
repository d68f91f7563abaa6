"""Pins of the expert cache's reference model (oracle/cache_ref.py) against what
the pages and the mathematics fix, without any GPU."""
import numpy as np

from oracle.cache_ref import LruArena


def test_uniform_requests_hit_at_capacity_over_experts():
    """Independent uniform request sets over E experts with a full arena of C slots:
    every requested expert is resident with probability C/E, whatever the policy
    (closed form), so the long-run true resident hit rate is C/E."""
    E, C, U = 896, 224, 16
    rng = np.random.default_rng(0)
    a = LruArena(E, C)
    for _ in range(300):  # fill
        a.step(rng.choice(E, U, replace=False))
    r0, h0 = a.requests, a.true_hits
    for _ in range(3000):
        a.step(rng.choice(E, U, replace=False))
    rate = (a.true_hits - h0) / (a.requests - r0)
    assert abs(rate - C / E) < 0.01, rate
    assert a.raw_hits == a.requests


def test_pages_cyclic_layers_never_hit_below_one_token_of_slots():
    """92 layers x 16 experts = 1,472 requests per token.  With the same routing
    every token (the most favourable case) LRU still evicts each expert before
    its next use whenever the arena holds no more slots than the other 91 layers
    request (1,456): 0% true resident hits, as the pages report for the 8 GB
    budget (about 460 experts of 17.5 MB); with room for a whole token every
    request after the first token hits."""
    layers, E, k = 92, 896, 16
    rng = np.random.default_rng(1)
    routing = [rng.choice(E, k, replace=False) for _ in range(layers)]
    for slots, expect in ((1472 - 16, 0.0), (460, 0.0), (1472, 1.0)):
        a = LruArena(layers * E, slots)
        for tok in range(3):
            h0, r0 = a.true_hits, a.requests
            for l in range(layers):
                a.step(l * E + routing[l])
            if tok > 0:
                assert (a.true_hits - h0) / (a.requests - r0) == expect, (slots, tok)
        assert a.requests == 3 * 1472


def test_victim_order_hand_worked():
    a = LruArena(10, 3, expert_bytes=100)
    s = a.step([5, 1])                     # empty slots in index order
    assert s["placed"] == {1: 0, 5: 1} and s["true_hits"] == 0
    s = a.step([7])
    assert s["placed"] == {7: 2}
    s = a.step([1, 9])                     # 1 hits (slot 0); 9 takes the LRU slot not used now: slot 1 (5)
    assert s["true_hits"] == 1 and s["placed"] == {9: 1}
    s = a.step([2, 3])                     # slots 2 (step 2) then 0 (step 3, lower index than 1)
    assert s["placed"] == {2: 2, 3: 0}
    assert a.step([1, 2, 3, 4])["refused"] and a.requests == 7
    assert a.bytes == 6 * 100 and a.true_hits == 1
