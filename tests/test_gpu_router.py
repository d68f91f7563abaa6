"""GPU parity of the router entry point (k3moe_router): the router scores of every
expert for every token (x . wr[e], bf16 in, fp32 accumulation) and the top-k
route on them, against the float64 oracle.

Bars (the reading of the pages' selection on scores the GPU sums in fp32):
  * the fp32 logits are within the accumulation bound the header states of the
    oracle's float64 scores, element by element;
  * idx bit-exact and w within 1 fp32 ulp of the oracle's route applied to the
    GPU's own fp32 logits (the selection itself is exact);
  * against the oracle's router-then-route (float64 scores rounded once to
    fp32): the same set of experts on every token whose k-th and (k+1)-th
    oracle scores are more than twice the row's bound apart, and the same order
    on every token whose first k + 1 scores are all that far apart; scores
    closer than that may order either way (the selection on the GPU's own
    scores is still checked exactly)."""
import numpy as np
import pytest
import torch

import gen
import mxfp4_expert_ffn_router_gb300 as k3
import oracle

pytestmark = pytest.mark.gpu

U24 = 2.0 ** -24


def _gamma(d, u):
    return d * u / (1.0 - d * u)


def _bound(s, x_bits, wr_bits):
    """Per-element bound |logit_gpu - logit_exact| for the kernel the library picks."""
    import math
    xv = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).double().abs().numpy()
    wv = torch.from_numpy(wr_bits.view(np.int16)).view(torch.bfloat16).double().abs().numpy()
    mag = xv @ wv.T
    if s.T < 64:
        g = _gamma(math.ceil(s.H / 256) + 7, U24)
    else:
        g = _gamma(math.ceil(s.H / 16) + 16, 2 * U24)
    return g * mag + 1e-30


def _run(s, x_bits, wr_bits):
    dev = torch.device("cuda")
    x = torch.from_numpy(x_bits.view(np.int16)).to(dev)
    wr = torch.from_numpy(wr_bits.view(np.int16)).to(dev)
    logits = torch.full((s.T, s.E), float("nan"), dtype=torch.float32, device=dev)
    idx = torch.empty((s.T, s.k), dtype=torch.int32, device=dev)
    w = torch.empty((s.T, s.k), dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    k3.k3moe_router(s, x, wr, logits, idx, w, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return logits.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


def _check(s, x_bits, wr_bits):
    g_logits, g_idx, g_w = _run(s, x_bits, wr_bits)
    l64, l32, idx_o, w_o, bad = oracle.router(s, x_bits, wr_bits)
    bound = _bound(s, x_bits, wr_bits)
    err = np.abs(g_logits.astype(np.float64) - l64)
    assert np.all(err <= bound), float(np.max(err / bound))
    # the selection on the GPU's own scores is exact
    idx_g, w_g, _ = oracle.route(s, g_logits)
    np.testing.assert_array_equal(g_idx, idx_g)
    assert np.all(np.abs(g_w.astype(np.float64) - w_g) <= np.spacing(np.abs(w_g.astype(np.float32))) + 1e-45)
    # against the exact scores: the same set wherever the k-th and (k+1)-th are
    # well apart, the same order wherever every adjacent pair of the first k + 1 is
    srt = -np.sort(-l64, axis=1)
    tol = 2.0 * bound.max(axis=1)
    m = min(s.k + 1, s.E)
    gaps = srt[:, : m - 1] - srt[:, 1:m]
    set_clear = gaps[:, s.k - 1] > tol if s.k < s.E else np.ones(s.T, bool)
    order_clear = np.all(gaps > tol[:, None], axis=1)
    for t in np.flatnonzero(set_clear):
        assert set(g_idx[t].tolist()) == set(idx_o[t].tolist()), t
    for t in np.flatnonzero(order_clear):
        np.testing.assert_array_equal(g_idx[t], idx_o[t])
    if s.T >= 50:
        assert set_clear.mean() > 0.5  # the bound is tight enough to decide most tokens
    return g_logits, g_idx


@pytest.mark.parametrize("T,H,E,k", [
    (1, 7168, 896, 16),     # decode
    (8, 7168, 896, 16),     # speculative-verify batch
    (3, 256, 40, 4),        # ragged: E not a multiple of anything
    (63, 512, 896, 16),     # last size on the CUDA-core kernel
    (64, 512, 896, 16),     # first size on the tensor cores
    (200, 1024, 300, 8),    # ragged token and expert tiles
    (130, 96, 17, 3),       # H not a multiple of the 64-value K step: zero-filled tail
    (4096, 7168, 896, 16),  # prefill chunk
])
def test_router_matches_oracle(T, H, E, k):
    s = gen.Shape(T, H, 64, E, k)
    x = gen.normal_bf16_bits(21, gen.stream(gen.KIND_X), T * H).reshape(T, H)
    wr = gen.make_router(s)
    _check(s, x, wr)


def test_router_ties_go_to_the_lower_expert():
    """Duplicated router rows give exactly equal scores (same products, same
    order): the lower expert index must win, as in the route."""
    s = gen.Shape(5, 512, 64, 64, 8)
    x = gen.normal_bf16_bits(22, gen.stream(gen.KIND_X), s.T * s.H).reshape(s.T, s.H)
    wr = gen.make_router(s).copy()
    wr[40:48] = wr[0:8]  # experts 40..47 score exactly like 0..7
    g_logits, g_idx = _check(s, x, wr)
    np.testing.assert_array_equal(g_logits[:, 40:48], g_logits[:, 0:8])
    for t in range(s.T):
        for e in g_idx[t]:
            if 40 <= e < 48:
                assert e - 40 in g_idx[t]


def test_router_is_deterministic_and_handles_empty_batch():
    s = gen.Shape(300, 1024, 64, 128, 8)
    x = gen.normal_bf16_bits(23, gen.stream(gen.KIND_X), s.T * s.H).reshape(s.T, s.H)
    wr = gen.make_router(s)
    a = _run(s, x, wr)
    b = _run(s, x, wr)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u.view(np.int32), v.view(np.int32))
    e = gen.Shape(0, 1024, 64, 128, 8)
    k3.k3moe_router(e, torch.empty((0, 1024), dtype=torch.int16, device="cuda"),
                    torch.from_numpy(wr.view(np.int16)).cuda(), torch.empty((0, 128), device="cuda"),
                    torch.empty((0, 8), dtype=torch.int32, device="cuda"), torch.empty((0, 8), device="cuda"))
