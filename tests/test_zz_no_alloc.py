"""k3moe_expert_ffn_noalloc: the expert FFN for callers that cannot allocate.

Some callers of this library cannot allocate device memory while they run a
layer (cudaMalloc/cudaFree may synchronise the device, a host framework may own
all device memory, or allocation calls may not be allowed where the layer runs).
For them the library offers an entry point with the same inputs and outputs as
k3moe_expert_ffn but no workspace argument: its scratch is a fixed device array
inside the library.  These tests call it through the C ABI and check that it
gives the result of the workspace entry point, within the parity tolerance of
the other GPU tests, on two calls in a row (the second call starts from the
array as the first call left it), and that it refuses a problem whose scratch
would not fit.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import gen
import mxfp4_expert_ffn_router_gb300 as k3
from layer_run import alloc_layer, max_rel_err

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _setup(T, H, I, E, k, mode):
    s = gen.Shape(T, H, I, E, k)
    rng = np.random.default_rng(1000 + T + E)
    logits = torch.from_numpy(rng.standard_normal((T, E)).astype(np.float32)).cuda()
    xbits = gen.normal_bf16_bits(5, gen.stream(gen.KIND_X), T * H).reshape(T, H)
    x = torch.from_numpy(xbits.view(np.int16)).cuda()
    a, b, c, d = gen.expert_arrays(H, I, 0, E)
    W = k3.Weights.from_stacked(*[torch.from_numpy(z).cuda() for z in (a, b, c, d)])
    buf = alloc_layer(s, mode=mode)
    k3.k3moe_route(s, logits, buf["idx"], buf["w"], buf["status"])
    k3.k3moe_bucket(s, buf["idx"], buf["counts"], buf["offsets"], buf["perm"], buf["inv"],
                    buf["ws_bucket"], buf["status"])
    return s, x, W, buf


@pytest.mark.parametrize("T,H,I,E,k,mode", [
    (1, 7168, 2048, 32, 16, k3.K3MOE_FFN_AUTO),    # decode-sized: AUTO picks the GEMV kernels
    (5, 512, 512, 8, 2, k3.K3MOE_FFN_STREAM),      # the retired STREAM mode: the GEMV kernels
    (4, 128, 64, 8, 2, k3.K3MOE_FFN_AUTO),         # the GEMV kernels
    (8, 7168, 2048, 48, 16, k3.K3MOE_FFN_GEMV),
])
def test_noalloc_matches_workspace_entry_point_twice(T, H, I, E, k, mode):
    s, x, W, buf = _setup(T, H, I, E, k, mode)
    A = s.T * s.k
    assert k3.k3moe_workspace_bytes(s, k3.K3MOE_OP_EXPERT_FFN, mode) <= k3.K3MOE_NOALLOC_SCRATCH_BYTES
    k3.k3moe_expert_ffn(s, x, W, buf["offsets"], buf["perm"], buf["Y"], mode, buf["ws_ffn"], buf["status"])
    torch.cuda.synchronize()
    ref = buf["Y"].cpu().numpy().astype(np.float64)
    for call in range(2):
        Y = torch.full((A, s.H), float("nan"), dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        k3.k3moe_expert_ffn_noalloc(s, x, W, buf["offsets"], buf["perm"], Y, mode, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, call
        got = Y.cpu().numpy()
        assert np.isfinite(got).all(), call
        assert max_rel_err(got, ref) <= TOL, (call, max_rel_err(got, ref))


def test_noalloc_auto_is_gemv_where_the_workspace_entry_point_picks_the_gemm():
    """T=8, E=48, k=16: k3moe_expert_ffn's AUTO takes the tensor-core GEMM (5A >=
    4E); the allocation-free entry point's AUTO takes the GEMV kernels: its
    output is bitwise the workspace entry point's GEMV output (the two modes are
    each checked against the oracle by the parity tests); GEMM and W4A4 are
    refused."""
    T, H, I, E, k = 8, 7168, 2048, 48, 16
    s, x, W, buf = _setup(T, H, I, E, k, k3.K3MOE_FFN_AUTO)
    assert k3.k3moe_workspace_bytes(s, k3.K3MOE_OP_EXPERT_FFN, k3.K3MOE_FFN_AUTO) == \
        k3.k3moe_workspace_bytes(s, k3.K3MOE_OP_EXPERT_FFN, k3.K3MOE_FFN_GEMM)
    A = s.T * s.k
    outs = {}
    for mode in (k3.K3MOE_FFN_AUTO, k3.K3MOE_FFN_GEMV):
        ws = torch.empty(k3.k3moe_workspace_bytes(s, k3.K3MOE_OP_EXPERT_FFN, mode), dtype=torch.uint8,
                         device="cuda")
        Y = torch.empty((A, s.H), dtype=torch.float32, device="cuda")
        k3.k3moe_expert_ffn(s, x, W, buf["offsets"], buf["perm"], Y, mode, ws, buf["status"])
        torch.cuda.synchronize()
        outs[mode] = Y.cpu().numpy()
    assert int(buf["status"].item()) == 0
    Y = torch.full((A, s.H), float("nan"), dtype=torch.float32, device="cuda")
    k3.k3moe_expert_ffn_noalloc(s, x, W, buf["offsets"], buf["perm"], Y, k3.K3MOE_FFN_AUTO, buf["status"])
    torch.cuda.synchronize()
    got = Y.cpu().numpy()
    np.testing.assert_array_equal(got.view(np.int32), outs[k3.K3MOE_FFN_GEMV].view(np.int32))
    assert not np.array_equal(outs[k3.K3MOE_FFN_AUTO].view(np.int32), got.view(np.int32))  # another kernel
    for mode in (k3.K3MOE_FFN_GEMM, k3.K3MOE_FFN_W4A4):
        with pytest.raises(k3.K3moeError) as err:
            k3.k3moe_expert_ffn_noalloc(s, x, W, buf["offsets"], buf["perm"], Y, mode, buf["status"])
        assert err.value.code == k3.K3MOE_ERR_UNSUPPORTED


def test_noalloc_refuses_problem_beyond_its_scratch():
    s = gen.Shape(4096, 7168, 2048, 896, 16)  # needs hundreds of MB of scratch
    assert k3.k3moe_workspace_bytes(s, k3.K3MOE_OP_EXPERT_FFN, 0) > k3.K3MOE_NOALLOC_SCRATCH_BYTES
    tiny = torch.zeros(64, dtype=torch.int32, device="cuda")
    W = k3.Weights([torch.zeros(896, dtype=torch.int64, device="cuda") for _ in range(4)])
    with pytest.raises(k3.K3moeError) as err:
        k3.k3moe_expert_ffn_noalloc(s, tiny.view(torch.int16), W, tiny, tiny, tiny.view(torch.float32))
    assert err.value.code == k3.K3MOE_ERR_NOALLOC_LIMIT
