"""The float64 oracle over large parity samples, run as N independent
single-threaded oracle processes.

The processes are started with ``spawn`` (never forked from a process that has
used the GPU).  Work is split by expert: a task is one routed expert and the
tokens of the sample routed to it, in the oracle's own bucket order.  Each
worker draws that expert's MXFP4 weights from the seeded generator (one thread)
and runs the oracle's expert FFN (``oracle.expert_ffn`` with one expert, k = 1)
on those tokens, so no process holds more than one expert's weights.  The
caller assembles the rows into the oracle's bucket order and runs the oracle's
combine: the arithmetic is the oracle's throughout, only its work is divided.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

import gen
import oracle


def _expert_rows(task):
    """One routed expert's oracle rows for the activation rows x_e ([n, H] bf16 bits):
    Y float64 [n, H]; with the GPU's h rows h_e ([n, I]) also the oracle's
    unrounded and rounded h, g, u and their magnitude sums (gate/up) and Y from
    the GPU's h (down)."""
    H, I, e, x_e, h_e, a4, seed = task
    n = x_e.shape[0]
    arrs = gen.expert_arrays(H, I, e, e + 1, seed=seed, nthreads=1)
    W = oracle.Weights(1, {0: tuple(z[0] for z in arrs)})
    s1 = gen.Shape(n, H, I, 1, 1)
    off, perm = np.array([0, n], np.int32), np.arange(n, dtype=np.int32)
    if h_e is None:
        return e, oracle.expert_ffn(s1, x_e, W, off, perm, a4=a4), None, None, None
    hpre, h_ref, sums = oracle.expert_gateup(s1, x_e, W, off, perm, a4=a4, sums=True)
    Y = oracle.expert_down(s1, h_e, W, off, a4=a4)
    return e, Y, hpre, h_ref, sums


def workers() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def sample_layer(s, xbits, idx, w, tokens, a4=False, seed=gen.WEIGHT_SEED, nproc=None, h_gpu=None, inv_gpu=None):
    """The oracle's layer restricted to the tokens ``tokens`` (sorted token ids).

    Without ``h_gpu``: returns (Y', out', inv') for the sub-batch, Y' float64
    [n k, H] in the oracle's bucket order of the sub-batch, out' float64 [n, H],
    inv' the position of assignment i k + j of the i-th sampled token in Y'.

    With the GPU's h (``h_gpu`` [A, I] in the GPU's bucket order, ``inv_gpu`` its
    inverse permutation): a dict with the sub-batch's GPU h rows, the oracle's
    unrounded and rounded h, its g, u, sum |Wg x| and sum |Wu x| ("sums"), Y' and
    out' computed from the GPU's h, and inv'."""
    tokens = np.asarray(tokens, np.int64)
    n = len(tokens)
    sub = gen.Shape(n, s.H, s.I, s.E, s.k)
    idx_s = np.ascontiguousarray(idx[tokens], np.int32)
    w_s = np.ascontiguousarray(w[tokens], np.float64)
    counts, offsets, perm, inv = oracle.bucket(sub, idx_s)
    staged = h_gpu is not None
    h_sub = None
    if staged:  # GPU h rows in the sub-batch's bucket order
        a_full = tokens[perm // s.k] * s.k + perm % s.k
        h_sub = np.ascontiguousarray(h_gpu[inv_gpu[a_full]])
    tasks = []
    for e in np.flatnonzero(counts):
        p0, p1 = int(offsets[e]), int(offsets[e + 1])
        rows = tokens[perm[p0:p1] // s.k]
        tasks.append((s.H, s.I, int(e), np.ascontiguousarray(xbits[rows]),
                      h_sub[p0:p1] if staged else None, bool(a4), seed))
    tasks.sort(key=lambda t: -t[3].shape[0])  # longest first
    Y = np.zeros((n * s.k, s.H), np.float64)
    hpre = np.zeros((n * s.k, s.I), np.float64) if staged else None
    h_ref = np.zeros((n * s.k, s.I), np.uint16) if staged else None
    sums = {k: np.zeros((n * s.k, s.I), np.float64) for k in ("g", "u", "gabs", "uabs")} if staged else None
    ctx = mp.get_context("spawn")
    with ctx.Pool(nproc or workers()) as pool:
        for e, rows, hp, hr, sm in pool.imap_unordered(_expert_rows, tasks):
            Y[offsets[e]:offsets[e + 1]] = rows
            if staged:
                hpre[offsets[e]:offsets[e + 1]] = hp
                h_ref[offsets[e]:offsets[e + 1]] = hr
                for key in sums:
                    sums[key][offsets[e]:offsets[e + 1]] = sm[key]
    out, _ = oracle.combine(sub, Y, w_s, inv)
    if not staged:
        return Y, out, inv
    return {"Y": Y, "out": out, "inv": inv, "hpre": hpre, "h_ref": h_ref, "h_gpu": h_sub, "sums": sums}


def hot_expert_sample(s, counts, offsets, perm, n_hot=32, tile=128, total=256, rng_seed=123):
    """Token ids covering every 128-token tile of the n_hot most loaded experts
    (the first position of each tile and the expert's last bucket position),
    the first and the last token, and seeded random tokens up to ``total``."""
    hot = np.argsort(-counts, kind="stable")[:n_hot]
    pick = {0, s.T - 1}
    for e in hot:
        p0, p1 = int(offsets[e]), int(offsets[e + 1])
        if p1 <= p0:
            continue
        for p in list(range(p0, p1, tile)) + [p1 - 1]:
            pick.add(int(perm[p] // s.k))
    rng = np.random.default_rng(rng_seed)
    while len(pick) < min(total, s.T):
        pick.add(int(rng.integers(0, s.T)))
    return np.array(sorted(pick), np.int64), hot
