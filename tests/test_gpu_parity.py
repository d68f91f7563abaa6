"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Bars: expert indices, counts, offsets, perm and inv bit-exact; routing weights
within 1 fp32 ulp of the oracle; the FFN staged at its bf16 rounding of h
(ffn_check): every GPU h element a bf16 rounding of a value within the kernel's
fp32 summation bound of the exact silu(g) u, then Y and the fp32 output within
max|err| <= 2e-3 * RMS of the oracle applied to the GPU's h; the bf16 output
equal to RNE(fp32 output)."""
import numpy as np
import pytest
import torch

import gen
import mxfp4_expert_ffn_router_gb300 as k3
import oracle
from ffn_check import check_staged, gpu_h
from layer_run import alloc_layer, bf16_rne_bits_of, host, max_rel_err, run_layer

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _experts_host(H, I, E, seed=gen.WEIGHT_SEED):
    a, b, c, d = gen.expert_arrays(H, I, 0, E, seed=seed)
    return a, b, c, d


def _device_weights(arrs, present=None):
    t = [torch.from_numpy(np.ascontiguousarray(z)).cuda() for z in arrs]
    return k3.Weights.from_stacked(*t, present=present)


def _check_route(s, logits, r):
    idx, w, bad = oracle.route(s, logits)
    np.testing.assert_array_equal(r["idx"], idx)
    wr = w.astype(np.float32)
    ulp = np.spacing(np.abs(wr))
    assert np.all(np.abs(r["w"].astype(np.float64) - w) <= ulp + 1e-45)
    return idx, w, bad


def _check_bucket(s, idx, r):
    counts, offsets, perm, inv = oracle.bucket(s, idx)
    np.testing.assert_array_equal(r["counts"], counts)
    np.testing.assert_array_equal(r["offsets"], offsets)
    np.testing.assert_array_equal(r["perm"], perm)
    np.testing.assert_array_equal(r["inv"], inv)
    return counts, offsets, perm, inv


def _full_check(s, logits, xbits, experts_np, r, a4=False, absent=()):
    """Routing and bucketing bit-exact; the FFN staged at its bf16 rounding of h
    (ffn_check): near-tie flips only, then Y and out against the oracle applied to
    the GPU's h; the bf16 output equal to RNE(fp32 output)."""
    idx, w, _ = _check_route(s, logits, r)
    counts, offsets, perm, inv = _check_bucket(s, idx, r)
    exps = {e: tuple(z[e] for z in experts_np) for e in np.unique(idx) if e not in absent}
    W = oracle.Weights(s.E, exps)
    st = check_staged(s, r, xbits, W, offsets, perm, w, inv, gpu_h(r, s), a4=a4)
    np.testing.assert_array_equal(r["out"], bf16_rne_bits_of(r["out_f32"]))
    Y = oracle.expert_down(s, gpu_h(r, s), W, offsets, a4=a4)
    out, _ = oracle.combine(s, Y, w, inv)
    assert st["out_err"] <= TOL
    return out


CASES = [  # T, H, I, E, k: several tiles and ragged tails
    (4, 128, 64, 8, 2),
    (1, 64, 32, 8, 8),
    (37, 256, 96, 24, 6),
    (129, 128, 64, 33, 3),
    (9, 7168, 64, 16, 4),
    (5, 96, 2048, 7, 2),
    (300, 64, 32, 5, 1),
    (3, 64, 64, 40, 32),
]


WIDE_CASES = [  # wider rows and experts (the GEMV kernels' exact and guarded instances)
    (1, 512, 512, 8, 2),
    (4, 384, 96, 8, 2),         # rows shorter than a warp's 32 chunks, guarded loops
    (70, 128, 32, 5, 3),        # smallest rows, 40+ tokens per expert
    (2, 8192, 4096, 3, 2),
    (5, 512, 512, 8, 2),
    (37, 1024, 512, 24, 6),
    (130, 512, 1024, 7, 3),
    (3, 7168, 512, 40, 32),
    (2, 4096, 4096, 3, 2),
    (8, 7168, 2048, 12, 4),
]


def _run_case(T, H, I, E, k, mode):
    s = gen.Shape(T, H, I, E, k)
    rng = np.random.default_rng(T * 1000 + E)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    xbits = gen.normal_bf16_bits(3, gen.stream(gen.KIND_X), T * H).reshape(T, H)
    experts = _experts_host(H, I, E)
    Wd = _device_weights(experts)
    b = alloc_layer(s, mode=mode)
    r = host(run_layer(s, torch.from_numpy(logits).cuda(), torch.from_numpy(xbits.view(np.int16)).cuda(), Wd,
                       bufs=b, mode=mode))
    assert r["status"][0] == 0
    _full_check(s, logits, xbits, experts, r)


@pytest.mark.parametrize("T,H,I,E,k", WIDE_CASES)
def test_gemv_mode_matches_oracle_wide(T, H, I, E, k):
    _run_case(T, H, I, E, k, k3.K3MOE_FFN_GEMV)


GEMM_CASES = [  # shapes the tcgen05 grouped GEMM accepts (H, 2I multiples of 128; I of 64)
    (8, 256, 128, 4, 2),
    (37, 512, 256, 8, 3),
    (300, 256, 128, 3, 2),      # experts with more than one 128-token tile
    (5, 7168, 2048, 16, 4),
    (130, 1024, 512, 6, 1),
]


@pytest.mark.parametrize("T,H,I,E,k", GEMM_CASES)
def test_gemm_mode_matches_oracle(T, H, I, E, k):
    _run_case(T, H, I, E, k, k3.K3MOE_FFN_GEMM)


def test_retired_stream_mode_is_the_gemv_mode():
    """K3MOE_FFN_STREAM is kept for callers that pass it and is served by the GEMV
    kernels: same workspace, same h and Y bit for bit."""
    T, H, I, E, k = 5, 512, 256, 8, 2
    s = gen.Shape(T, H, I, E, k)
    assert k3.k3moe_workspace_bytes(s, k3.K3MOE_OP_EXPERT_FFN, k3.K3MOE_FFN_STREAM) == \
        k3.k3moe_workspace_bytes(s, k3.K3MOE_OP_EXPERT_FFN, k3.K3MOE_FFN_GEMV)
    rng = np.random.default_rng(9)
    logits = torch.from_numpy(rng.standard_normal((T, E)).astype(np.float32)).cuda()
    xbits = gen.normal_bf16_bits(4, gen.stream(gen.KIND_X), T * H).reshape(T, H)
    Wd = _device_weights(_experts_host(H, I, E))
    got = {}
    for mode in (k3.K3MOE_FFN_GEMV, k3.K3MOE_FFN_STREAM):
        r = host(run_layer(s, logits, torch.from_numpy(xbits.view(np.int16)).cuda(), Wd,
                           bufs=alloc_layer(s, mode=mode), mode=mode))
        assert r["status"][0] == 0
        got[mode] = (gpu_h(r, s), r["Y"])
    np.testing.assert_array_equal(got[k3.K3MOE_FFN_GEMV][0], got[k3.K3MOE_FFN_STREAM][0])
    np.testing.assert_array_equal(got[k3.K3MOE_FFN_GEMV][1].view(np.int32), got[k3.K3MOE_FFN_STREAM][1].view(np.int32))


@pytest.mark.parametrize("mode", [k3.K3MOE_FFN_GEMV, k3.K3MOE_FFN_GEMM])
def test_absent_expert_and_hot_expert_both_modes(mode):
    s = gen.Shape(45, 512, 512, 6, 2)
    logits = np.random.default_rng(7).standard_normal((45, 6)).astype(np.float32)
    logits[:, 4] += 50.0  # expert 4 takes every token: many token chunks
    xbits = gen.normal_bf16_bits(4, gen.stream(gen.KIND_X), 45 * 512).reshape(45, 512)
    experts = _experts_host(512, 512, 6)
    present = np.ones(6, bool)
    idx, _, _ = oracle.route(s, logits)
    gone = int(idx[0, 1])
    present[gone] = False
    b = alloc_layer(s, mode=mode)
    r = host(run_layer(s, torch.from_numpy(logits).cuda(), torch.from_numpy(xbits.view(np.int16)).cuda(),
                       _device_weights(experts, present=torch.from_numpy(present)), bufs=b, mode=mode))
    assert r["status"][0] == 0 and r["counts"][4] == 45
    _full_check(s, logits, xbits, experts, r, absent=(gone,))


@pytest.mark.parametrize("T,H,I,E,k", CASES)
def test_small_shapes_match_oracle(T, H, I, E, k):
    s = gen.Shape(T, H, I, E, k)
    rng = np.random.default_rng(T * 1000 + E)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    xbits = gen.normal_bf16_bits(3, gen.stream(gen.KIND_X), T * H).reshape(T, H)
    experts = _experts_host(H, I, E)
    Wd = _device_weights(experts)
    r = host(run_layer(s, torch.from_numpy(logits).cuda(), torch.from_numpy(xbits.view(np.int16)).cuda(), Wd))
    assert r["status"][0] == 0
    _full_check(s, logits, xbits, experts, r)


def test_tiny_workload():
    s = gen.CONFIGS["tiny"]
    logits, xbits = gen.make_logits("tiny"), gen.make_x(s)
    experts = _experts_host(s.H, s.I, s.E)
    r = host(run_layer(s, torch.from_numpy(logits).cuda(), torch.from_numpy(xbits.view(np.int16)).cuda(),
                       _device_weights(experts)))
    _full_check(s, logits, xbits, experts, r)


def test_ties_signed_zeros_and_all_equal_rows():
    s = gen.Shape(6, 64, 32, 40, 5)
    rng = np.random.default_rng(5)
    logits = np.round(rng.standard_normal((6, 40)) * 2).astype(np.float32) / 2
    logits[0] = 0.25
    logits[1, :20] = -0.0
    logits[1, 20:] = 0.0
    logits[2, ::3] = 7.0
    xbits = gen.normal_bf16_bits(4, gen.stream(gen.KIND_X), 6 * 64).reshape(6, 64)
    experts = _experts_host(64, 32, 40)
    r = host(run_layer(s, torch.from_numpy(logits).cuda(), torch.from_numpy(xbits.view(np.int16)).cuda(),
                       _device_weights(experts)))
    _full_check(s, logits, xbits, experts, r)
    assert r["idx"][0].tolist() == [0, 1, 2, 3, 4]


def test_nan_row_flagged_and_infinities():
    s = gen.Shape(4, 64, 32, 16, 4)
    logits = np.random.default_rng(1).standard_normal((4, 16)).astype(np.float32)
    logits[1, 3] = np.nan
    logits[2] = -np.inf
    logits[3, 5] = np.inf
    logits[3, 9] = np.inf
    xbits = gen.normal_bf16_bits(4, gen.stream(gen.KIND_X), 4 * 64).reshape(4, 64)
    experts = _experts_host(64, 32, 16)
    r = host(run_layer(s, torch.from_numpy(logits).cuda(), torch.from_numpy(xbits.view(np.int16)).cuda(),
                       _device_weights(experts)))
    assert r["status"][0] & k3.K3MOE_DEV_NONFINITE
    idx, w, bad = oracle.route(s, logits)
    np.testing.assert_array_equal(r["idx"], idx)
    np.testing.assert_allclose(r["w"], w, rtol=1e-7, atol=0)
    assert bad.tolist() == [0, 1, 0, 0]
    _full_check(s, logits, xbits, experts, r)


def test_absent_expert_gives_zero_rows():
    s = gen.Shape(16, 128, 64, 8, 2)
    logits = np.random.default_rng(2).standard_normal((16, 8)).astype(np.float32)
    xbits = gen.normal_bf16_bits(4, gen.stream(gen.KIND_X), 16 * 128).reshape(16, 128)
    experts = _experts_host(128, 64, 8)
    present = np.ones(8, bool)
    present[3] = False
    r = host(run_layer(s, torch.from_numpy(logits).cuda(), torch.from_numpy(xbits.view(np.int16)).cuda(),
                       _device_weights(experts, present=torch.from_numpy(present))))
    assert r["status"][0] == 0
    _full_check(s, logits, xbits, experts, r, absent=(3,))
    lo, hi = r["offsets"][3], r["offsets"][4]
    assert hi > lo and not r["Y"][lo:hi].any()


def test_one_expert_takes_every_token():
    s = gen.Shape(45, 128, 64, 6, 2)
    logits = np.random.default_rng(7).standard_normal((45, 6)).astype(np.float32)
    logits[:, 4] += 50.0
    xbits = gen.normal_bf16_bits(4, gen.stream(gen.KIND_X), 45 * 128).reshape(45, 128)
    experts = _experts_host(128, 64, 6)
    r = host(run_layer(s, torch.from_numpy(logits).cuda(), torch.from_numpy(xbits.view(np.int16)).cuda(),
                       _device_weights(experts)))
    assert r["counts"][4] == 45
    _full_check(s, logits, xbits, experts, r)


def test_empty_batch():
    s = gen.Shape(0, 128, 64, 8, 2)
    b = alloc_layer(s)
    b["counts"].fill_(-5)
    b["offsets"].fill_(-5)
    k3.k3moe_route(s, torch.empty((0, 8), device="cuda"), b["idx"], b["w"], b["status"])
    k3.k3moe_bucket(s, b["idx"], b["counts"], b["offsets"], b["perm"], b["inv"], b["ws_bucket"], b["status"])
    torch.cuda.synchronize()
    assert not b["counts"].any() and not b["offsets"].any()


def test_maximum_hidden_and_intermediate():
    s = gen.Shape(2, 16384, 16384, 2, 1)
    logits = np.array([[1.0, 0.0], [0.0, 1.0]], np.float32)
    xbits = gen.normal_bf16_bits(4, gen.stream(gen.KIND_X), 2 * 16384).reshape(2, 16384)
    experts = _experts_host(16384, 16384, 2)
    r = host(run_layer(s, torch.from_numpy(logits).cuda(), torch.from_numpy(xbits.view(np.int16)).cuda(),
                       _device_weights(experts)))
    _full_check(s, logits, xbits, experts, r)


def test_maximum_experts_and_k():
    s = gen.Shape(5, 64, 32, 4096, 32)
    logits = np.random.default_rng(9).standard_normal((5, 4096)).astype(np.float32)
    xbits = gen.normal_bf16_bits(4, gen.stream(gen.KIND_X), 5 * 64).reshape(5, 64)
    experts = _experts_host(64, 32, 4096)
    r = host(run_layer(s, torch.from_numpy(logits).cuda(), torch.from_numpy(xbits.view(np.int16)).cuda(),
                       _device_weights(experts)))
    _full_check(s, logits, xbits, experts, r)


@pytest.mark.parametrize("E,k", [(100, 8), (200, 16), (512, 32), (1000, 16), (1024, 32), (1025, 16), (2000, 5)])
def test_route_every_keys_per_lane_instance(E, k):
    """The route's instances: a warp per token for E <= 1024 (4, 8, 16 and 32 keys
    per lane here), the block search above it; 37 tokens (several blocks of 8 warps
    and a ragged tail) with rows of ties, signed zeros, infinities and a NaN row."""
    T = 37
    s = gen.Shape(T, 64, 32, E, k)
    logits = np.random.default_rng(E).standard_normal((T, E)).astype(np.float32)
    logits[1] = np.round(logits[1])            # many ties at each value
    logits[2] = 0.0
    logits[2, ::3] = -0.0                      # all equal, signed zeros
    logits[3, [5, E - 1]] = np.inf             # two +inf picks share the weight
    logits[4] = -np.inf                        # all -inf: weights 1/k
    logits[5, E // 2] = np.nan                 # NaN row: experts 0..k-1, flagged
    b = alloc_layer(s, with_f32=False)
    k3.k3moe_route(s, torch.from_numpy(logits).cuda(), b["idx"], b["w"], b["status"])
    r = host(b)
    _check_route(s, logits, r)
    assert r["status"][0] == k3.K3MOE_DEV_NONFINITE


def test_large_bucket_multi_tile_bit_exact():
    s = gen.Shape(5000, 32, 32, 300, 7)  # A = 35000: the tiled bucketing path
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((5000, 300)).astype(np.float32)
    logits[:, 17] += 2.0
    b = alloc_layer(s, with_f32=False)
    lg = torch.from_numpy(logits).cuda()
    k3.k3moe_route(s, lg, b["idx"], b["w"], b["status"])
    k3.k3moe_bucket(s, b["idx"], b["counts"], b["offsets"], b["perm"], b["inv"], b["ws_bucket"], b["status"])
    r = host(b)
    idx, _, _ = _check_route(s, logits, r)
    _check_bucket(s, idx, r)


def test_deterministic_repeat():
    s = gen.Shape(33, 256, 128, 12, 4)
    logits = np.random.default_rng(8).standard_normal((33, 12)).astype(np.float32)
    xbits = gen.normal_bf16_bits(4, gen.stream(gen.KIND_X), 33 * 256).reshape(33, 256)
    Wd = _device_weights(_experts_host(256, 128, 12))
    lg, xd = torch.from_numpy(logits).cuda(), torch.from_numpy(xbits.view(np.int16)).cuda()
    a = host(run_layer(s, lg, xd, Wd))
    b = host(run_layer(s, lg, xd, Wd))
    for key in ("idx", "w", "perm", "Y", "out", "out_f32"):
        assert np.array_equal(a[key].view(np.uint8), b[key].view(np.uint8)), key


def test_bad_expert_index_is_reported_not_read():
    s = gen.Shape(3, 64, 32, 8, 2)
    b = alloc_layer(s)
    idx = torch.tensor([[0, 1], [9, 2], [-1, 3]], dtype=torch.int32, device="cuda")
    k3.k3moe_bucket(s, idx, b["counts"], b["offsets"], b["perm"], b["inv"], b["ws_bucket"], b["status"])
    r = host(b)
    assert r["status"][0] & k3.K3MOE_DEV_BOUNDS
    assert r["offsets"][-1] == 4 and r["inv"][2] == -1 and r["inv"][4] == -1


@pytest.mark.parametrize("mode", [k3.K3MOE_FFN_GEMV, k3.K3MOE_FFN_GEMM, k3.K3MOE_FFN_W4A4])
def test_misaligned_expert_is_reported_and_reads_as_absent(mode):
    """An expert whose pointers are all given but whose gate/up codes are not
    16-byte aligned: every mode checks the alignment before it reads through the
    pointer, reports K3MOE_DEV_BOUNDS, and gives that expert zero rows; the other
    experts are unaffected.  (The shifted pointer stays inside its allocation.)"""
    s = gen.Shape(24, 512, 512, 6, 2)
    logits = np.random.default_rng(11).standard_normal((24, 6)).astype(np.float32)
    xbits = gen.normal_bf16_bits(4, gen.stream(gen.KIND_X), 24 * 512).reshape(24, 512)
    experts = _experts_host(512, 512, 6)
    idx, _, _ = oracle.route(s, logits)
    bad = int(idx[0, 0])
    Wd = _device_weights(experts)
    ptrs = [p.clone() for p in Wd.ptrs]
    ptrs[0][bad] += 1  # w13 codes of expert `bad`, one byte off
    Wbad = k3.Weights(ptrs, keep=Wd.keep)
    b = alloc_layer(s, mode=mode)
    r = host(run_layer(s, torch.from_numpy(logits).cuda(), torch.from_numpy(xbits.view(np.int16)).cuda(),
                       Wbad, bufs=b, mode=mode))
    assert r["status"][0] & k3.K3MOE_DEV_BOUNDS
    assert not (r["status"][0] & k3.K3MOE_DEV_TIMEOUT)
    _full_check(s, logits, xbits, experts, r, a4=(mode == k3.K3MOE_FFN_W4A4), absent=(bad,))
    lo, hi = r["offsets"][bad], r["offsets"][bad + 1]
    assert hi > lo and not r["Y"][lo:hi].any()
