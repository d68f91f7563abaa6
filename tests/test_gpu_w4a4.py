"""GPU parity of the W4A4 pieces: the MXFP4 activation quantiser (bit-exact
codes and scales against the oracle's quantiser, OCP Microscaling Formats v1.0
conversion rule) and the W4A4 expert-FFN mode (the tcgen05 GEMM on MXFP4
activations) against the oracle's A4 path."""
import numpy as np
import pytest
import torch

import gen
import oracle
import mxfp4_expert_ffn_router_gb300 as k3
from test_gpu_parity import GEMM_CASES, _device_weights, _experts_host, _full_check
from layer_run import alloc_layer, host, run_layer

pytestmark = pytest.mark.gpu


def _bf16_bits(v):
    """float64 values -> bf16 bit patterns (all values used here are exact in bf16)."""
    f = np.asarray(v, np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def _special_blocks():
    rng = np.random.default_rng(7)
    blocks = []
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    for e in (-10, 0, 3, 60):  # grid midpoints (ties) at several shared exponents, max 4 * 2^e
        b = np.zeros(32)
        b[:7] = mids * 2.0 ** e
        b[7:14] = -mids * 2.0 ** e
        b[14] = 4.0 * 2.0 ** e
        b[15:] = rng.standard_normal(17) * 2.0 ** e
        b = np.clip(b, -5.9 * 2.0 ** e, 5.9 * 2.0 ** e)
        blocks.append(b)
    blocks.append(np.zeros(32))                                   # all-zero block: scale byte 0
    b = np.full(32, -0.0); blocks.append(b)                        # negative zeros
    blocks.append(np.full(32, 7.0) * np.sign(rng.standard_normal(32)))  # saturation at 6
    blocks.append(rng.standard_normal(32) * 2.0 ** -130)           # tiny: shared exponent clamps at -127
    blocks.append(rng.standard_normal(32) * 2.0 ** 120)            # huge
    bits = [_bf16_bits(b) for b in blocks]
    nan_block = _bf16_bits(rng.standard_normal(32))
    nan_block[[3, 17]] = 0x7FC0                                     # NaN elements: code 0, ignored by amax
    bits.append(nan_block)
    bits.append(np.full(32, 0x7FC0, np.uint16))                     # all NaN
    return np.concatenate(bits)


@pytest.mark.parametrize("n_random", [0, 32 * 1000, 32 * 4099])
def test_quantize_matches_oracle_bit_exact(n_random):
    rng = np.random.default_rng(n_random + 1)
    v = rng.standard_normal(n_random) * 2.0 ** rng.integers(-40, 40, n_random // 32 if n_random else 0).repeat(32)
    bits = np.concatenate([_special_blocks(), _bf16_bits(v)])
    codes_ref, scales_ref = oracle.quant_mxfp4(bits)
    x = torch.from_numpy(bits.view(np.int16)).cuda()
    codes = torch.empty(bits.size // 2, dtype=torch.uint8, device="cuda")
    scales = torch.empty(bits.size // 32, dtype=torch.uint8, device="cuda")
    k3.k3moe_quantize_mxfp4(x, codes, scales)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(scales.cpu().numpy(), scales_ref)
    np.testing.assert_array_equal(codes.cpu().numpy(), codes_ref)


def test_quantize_rejects_bad_arguments():
    x = torch.zeros(48, dtype=torch.bfloat16, device="cuda")
    c = torch.zeros(24, dtype=torch.uint8, device="cuda")
    s = torch.zeros(2, dtype=torch.uint8, device="cuda")
    with pytest.raises(k3.K3moeError):
        k3.k3moe_quantize_mxfp4(x, c, s)  # 48 values: not whole blocks


@pytest.mark.parametrize("T,H,I,E,k", GEMM_CASES)
def test_w4a4_mode_matches_a4_oracle(T, H, I, E, k):
    s = gen.Shape(T, H, I, E, k)
    rng = np.random.default_rng(T * 1000 + E + 5)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    xbits = gen.normal_bf16_bits(3, gen.stream(gen.KIND_X), T * H).reshape(T, H)
    experts = _experts_host(H, I, E)
    Wd = _device_weights(experts)
    mode = k3.K3MOE_FFN_W4A4
    r = host(run_layer(s, torch.from_numpy(logits).cuda(), torch.from_numpy(xbits.view(np.int16)).cuda(), Wd,
                       bufs=alloc_layer(s, mode=mode), mode=mode))
    assert r["status"][0] == 0
    out_a4 = _full_check(s, logits, xbits, experts, r, a4=True)
    # the A4 result differs from the A16 one (reported, not gated): the quantiser is on the path
    idx, w, _ = oracle.route(s, logits)
    counts, offsets, perm, inv = oracle.bucket(s, idx)
    exps = {e: tuple(z[e] for z in experts) for e in np.unique(idx)}
    out_a16, _ = oracle.combine(s, oracle.expert_ffn(s, xbits, oracle.Weights(s.E, exps), offsets, perm), w, inv)
    assert not np.allclose(out_a4, out_a16, rtol=0, atol=0)


def test_w4a4_mode_rejects_unsupported_shape():
    s = gen.Shape(4, 96, 64, 8, 2)  # H not a multiple of 128
    assert k3.k3moe_workspace_bytes(s, k3.K3MOE_OP_EXPERT_FFN, k3.K3MOE_FFN_W4A4) == 0
