"""ORACLE for the expert cache's policy and counters -- test infrastructure only.

A plain-Python statement of the least-recently-used expert arena that the
kimi-k3-in-c engine puts between its expert store and the matmul ("running a
2.78T model in 8 GB", the section on the trunk and the expert cache): an arena
of expert slots, a batch prefetch of each step's experts just before use, and
two counts per request -- a raw hit when the expert is in the arena when the
matmul asks for it (near 100% with the batch prefetch), and a true resident hit
when the expert stayed in the arena since the previous step (the measure of
reads avoided; 0% at an 8 GB budget, where all 1,472 requests of a token miss).

Readings where the pages are silent (the CUDA library states the same rule):
  * a step requests a set of experts (ascending ids); requested experts already
    in a slot are true resident hits and are marked used;
  * each missing expert, in ascending id order, takes the least recently used
    slot not used in this step -- slots ordered by the last step they were used
    in (never-used slots first), ties by slot index; the slot's previous expert
    leaves the arena;
  * after the batch prefetch every request is served from the arena, so raw
    hits = requests;
  * a step with more distinct experts than slots is refused (nothing changes).
Only the tests may import this module.
"""
from __future__ import annotations


class LruArena:
    def __init__(self, n_experts: int, n_slots: int, expert_bytes: int = 1):
        self.E, self.S, self.B = n_experts, n_slots, expert_bytes
        self.slot_of = {}                  # expert -> slot
        self.expert_of = [-1] * n_slots    # slot -> expert
        self.last = [-1] * n_slots         # slot -> last step it was used in
        self.step_no = 0
        self.requests = self.raw_hits = self.true_hits = self.bytes = 0

    def step(self, requested) -> dict:
        """One step over the requested expert ids; returns the step's counts and
        the slot each missing expert was given ({expert: slot})."""
        req = sorted(set(int(e) for e in requested))
        hits = [e for e in req if e in self.slot_of]
        misses = [e for e in req if e not in self.slot_of]
        used = {self.slot_of[e] for e in hits}
        free = sorted((v for v in range(self.S) if v not in used), key=lambda v: (self.last[v], v))
        if len(misses) > len(free):
            return {"refused": True, "requests": 0, "true_hits": 0, "misses": 0, "placed": {}}
        self.step_no += 1
        for v in used:
            self.last[v] = self.step_no
        placed = {}
        for e, v in zip(misses, free):
            old = self.expert_of[v]
            if old >= 0:
                del self.slot_of[old]
            self.expert_of[v] = e
            self.slot_of[e] = v
            self.last[v] = self.step_no
            placed[e] = v
        self.requests += len(req)
        self.raw_hits += len(req)
        self.true_hits += len(hits)
        self.bytes += len(misses) * self.B
        return {"refused": False, "requests": len(req), "true_hits": len(hits), "misses": len(misses),
                "placed": placed}
