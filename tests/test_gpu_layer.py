"""GPU tests of the whole-layer entry point (k3moe_layer): every output and
intermediate is bitwise what the four separate calls (route, bucket, expert
FFN, combine) write -- on the single-block decode front (T <= 4, E <= 1024,
T k <= 128) and on the four-call path -- including NaN rows, ties, absent
experts and the largest batch the front takes.  The separate calls are checked
against the oracle by the other GPU tests."""
import numpy as np
import pytest
import torch

import gen
import mxfp4_expert_ffn_router_gb300 as k3
import oracle
from layer_run import alloc_layer, host, run_layer

pytestmark = pytest.mark.gpu

KEYS = ("idx", "w", "counts", "offsets", "perm", "inv", "Y", "out", "out_f32", "status")


def _layer_call(s, lg, x, W, mode):
    b = alloc_layer(s, mode=mode)
    ws = torch.empty(max(1, k3.k3moe_workspace_bytes(s, k3.K3MOE_OP_LAYER, mode)), dtype=torch.uint8, device="cuda")
    k3.k3moe_layer(s, lg, x, W, b["idx"], b["w"], b["counts"], b["offsets"], b["perm"], b["inv"], b["Y"], b["out"],
                   b["out_f32"], mode, ws, b["status"])
    return host(b)


def _compare(s, logits, xbits, arrs, mode=k3.K3MOE_FFN_AUTO, present=None):
    lg = torch.from_numpy(np.ascontiguousarray(logits, np.float32)).cuda()
    x = torch.from_numpy(xbits.view(np.int16)).cuda()
    W = k3.Weights.from_stacked(*[torch.from_numpy(a).cuda() for a in arrs],
                                present=None if present is None else torch.from_numpy(present))
    one = _layer_call(s, lg, x, W, mode)
    four = host(run_layer(s, lg, x, W, bufs=alloc_layer(s, mode=mode), mode=mode))
    for key in KEYS:
        a, b = np.asarray(one[key]), np.asarray(four[key])
        np.testing.assert_array_equal(a.view(np.uint8), b.view(np.uint8), err_msg=key)
    return one


@pytest.mark.parametrize("T,H,I,E,k", [
    (1, 7168, 2048, 896, 16),    # decode
    (8, 7168, 2048, 896, 16),    # batch8
    (4, 512, 256, 64, 32),       # the largest batch the front takes (A = 128)
    (5, 512, 256, 64, 16),       # one token more: the four-call path
    (3, 256, 128, 1024, 5),      # E = 1024
    (4, 128, 64, 8, 2),          # tiny
])
def test_layer_is_bitwise_the_four_calls(T, H, I, E, k):
    s = gen.Shape(T, H, I, E, k)
    logits = gen.normal_f32(31, gen.stream(gen.KIND_LOGITS), T * E, 2.0).reshape(T, E)
    xbits = gen.normal_bf16_bits(31, gen.stream(gen.KIND_X), T * H).reshape(T, H)
    arrs = gen.expert_arrays(H, I, 0, E)
    r = _compare(s, logits, xbits, arrs)
    assert r["status"][0] == 0
    idx, _, _ = oracle.route(s, logits)
    np.testing.assert_array_equal(r["idx"], idx)


@pytest.mark.parametrize("rows", ["special", "zeros"])
def test_layer_front_special_rows_and_absent_experts(rows):
    s = gen.Shape(4, 256, 128, 40, 4)
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((s.T, s.E)).astype(np.float32)
    if rows == "special":
        logits[0] = 0.5                        # all equal: experts 0..3
        logits[1, 7] = np.nan                  # NaN row: 0..3, weights 1/4, flagged
        logits[2, [5, 9]] = np.inf             # two +inf picks share the weight
        logits[3] = -np.inf                    # all -inf: weights 1/4
    else:
        logits[0, :6] = [-0.0, 0.0, 1.0, 1.0, -0.0, 0.0]
        logits[0, 6:] = -1.0                   # ties and signed zeros
        logits[1, ::2] = 2.0                   # twenty-way tie at the top
    xbits = gen.normal_bf16_bits(32, gen.stream(gen.KIND_X), s.T * s.H).reshape(s.T, s.H)
    arrs = gen.expert_arrays(s.H, s.I, 0, s.E)
    present = np.ones(s.E, bool)
    present[[0, 9]] = False
    r = _compare(s, logits, xbits, arrs, present=present)
    assert r["status"][0] == (k3.K3MOE_DEV_NONFINITE if rows == "special" else 0)
    idx, w, _ = oracle.route(s, logits)
    np.testing.assert_array_equal(r["idx"], idx)


@pytest.mark.parametrize("mode", [k3.K3MOE_FFN_GEMM, k3.K3MOE_FFN_W4A4])
def test_layer_tensor_core_modes(mode):
    s = gen.Shape(96, 256, 128, 8, 2)
    logits = gen.normal_f32(33, gen.stream(gen.KIND_LOGITS), s.T * s.E, 1.0).reshape(s.T, s.E)
    xbits = gen.normal_bf16_bits(33, gen.stream(gen.KIND_X), s.T * s.H).reshape(s.T, s.H)
    r = _compare(s, logits, xbits, gen.expert_arrays(s.H, s.I, 0, s.E), mode=mode)
    assert r["status"][0] == 0
