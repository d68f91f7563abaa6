"""GPU parity on the full-size workloads (896 experts, H=7168, I=2048; 21 GB of
MXFP4 weights resident), in the launch configuration the benchmark times.

Decode (T=1), the 8-token batch (through the GEMV and the tensor-core GEMM
modes, each against the same oracle), the speculative-verify batches of 2 to 16
tokens and the I=1536 decode layer are checked in full against the oracle.
For the 4096- and 2048-token prefill workloads the routing and bucketing are
checked bit-exactly on every token; the outputs of at least 256 tokens --
covering every 64-position span of the 32 most loaded experts' buckets and
their last positions, the first and the last token -- are checked against the
oracle, both the combined rows and every one of their expert output rows Y.
The FFN is checked in stages at its bf16 rounding of h (ffn_check): each GPU h
element must be a bf16 rounding of a value within the fp32 summation bound of
the exact silu(g) u, and Y and the output are compared with the oracle applied
to the GPU's h."""
import numpy as np
import pytest
import torch

import gen
import oracle
from gen.device import DeviceExperts, device_inputs
from layer_run import alloc_layer, bf16_rne_bits_of, host, max_rel_err, run_layer
from ffn_check import check_h, gamma, gpu_h
from oracle_pool import hot_expert_sample, sample_layer
import mxfp4_expert_ffn_router_gb300 as k3

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module")
def experts_2048():
    dx = DeviceExperts(7168, 2048, 896)
    yield dx
    del dx
    torch.cuda.empty_cache()


def _weights(dx):
    return k3.Weights.from_stacked(*dx.tensors)


def _route_bucket_exact(s, logits, r):
    idx, w, _ = oracle.route(s, logits)
    np.testing.assert_array_equal(r["idx"], idx)
    assert np.all(np.abs(r["w"].astype(np.float64) - w) <= np.spacing(np.abs(w.astype(np.float32))) + 1e-45)
    counts, offsets, perm, inv = oracle.bucket(s, idx)
    for key, ref in (("counts", counts), ("offsets", offsets), ("perm", perm), ("inv", inv)):
        np.testing.assert_array_equal(r[key], ref, err_msg=key)
    return idx, w, counts, offsets, perm, inv


def _staged(s, r, xbits, idx, w, inv, tokens, a4=False):
    """Staged FFN parity (ffn_check) on the given tokens: the GPU's h near-tie
    flips only, then its Y rows and fp32 outputs against the oracle applied to
    the GPU's h, the oracle running as parallel single-threaded processes."""
    d = sample_layer(s, xbits, idx, w, tokens, a4=a4, h_gpu=gpu_h(r, s), inv_gpu=inv)
    st = check_h(d["h_gpu"], d["sums"], gamma(s, r["mode"]))
    st["h_differs"] = int((d["h_gpu"] != d["h_ref"]).sum())
    n = len(tokens)
    a_ids = (np.asarray(tokens)[:, None] * s.k + np.arange(s.k)[None, :]).ravel()
    got_Y = r["Y"][inv[a_ids]]
    ref_Y = d["Y"][d["inv"][np.arange(n * s.k)]]
    st["y_err"] = max_rel_err(got_Y, ref_Y)
    st["out_err"] = max_rel_err(r["out_f32"][tokens], d["out"])
    print(st)
    assert st["y_err"] <= TOL, st
    assert st["out_err"] <= TOL, st
    return st


def _full(name, dx, s=None, mode=k3.K3MOE_FFN_AUTO):
    """The whole layer against the oracle: routing and bucketing bit-exact, the
    FFN staged at the bf16 rounding of h over every token."""
    s = s or gen.CONFIGS[name]
    lg, xd, logits, xbits = device_inputs(name, s)
    r = host(run_layer(s, lg, xd, _weights(dx), bufs=alloc_layer(s, mode=mode), mode=mode))
    assert r["status"][0] == 0
    idx, w, counts, offsets, perm, inv = _route_bucket_exact(s, logits, r)
    _staged(s, r, xbits, idx, w, inv, np.arange(s.T))
    np.testing.assert_array_equal(r["out"], bf16_rne_bits_of(r["out_f32"]))
    return r


@pytest.mark.parametrize("mode", [k3.K3MOE_FFN_AUTO, k3.K3MOE_FFN_GEMV])
def test_decode(experts_2048, mode):
    r = _full("decode", experts_2048, mode=mode)
    assert len(np.unique(r["idx"])) == 16


@pytest.mark.parametrize("mode", [k3.K3MOE_FFN_GEMV, k3.K3MOE_FFN_GEMM])
def test_batch8_gemv_and_gemm_against_one_oracle(experts_2048, mode):
    """The per-token (GEMV) and batched (tensor-core GEMM) paths each agree with the
    same oracle on the 8-token batch; the chunk-union prefill of the kimi-k3-in-c
    CHANGELOG ("[1.0.0] Added") requires the batched path to give the per-token
    path's tokens."""
    r = _full("batch8", experts_2048, mode=mode)
    shared = set(r["idx"][0, :8].tolist())
    for t in range(1, 4):
        assert set(r["idx"][t, :8].tolist()) == shared


@pytest.mark.parametrize("T", [2, 4, 12, 16])
@pytest.mark.parametrize("mode", [k3.K3MOE_FFN_GEMV, k3.K3MOE_FFN_GEMM])
def test_spec_verify_batches(experts_2048, T, mode):
    """Speculative-verify batches ("--spec N" of the kimi-k3-in-c CHANGELOG, block
    "[1.0.0] Added"): T tokens, half of them sharing 8 of their top-16 experts."""
    name = f"spec{T}"
    r = _full(name, experts_2048, mode=mode)
    if T >= 4:
        shared = set(r["idx"][0, :8].tolist())
        for t in range(1, T // 2):
            assert set(r["idx"][t, :8].tolist()) == shared


def test_decode_i1536():
    dx = DeviceExperts(7168, 1536, 896)
    _full("decode_i1536", dx, gen.CONFIGS["decode_i1536"])


@pytest.mark.parametrize("name,mode", [("prefill", k3.K3MOE_FFN_AUTO), ("skewed", k3.K3MOE_FFN_AUTO),
                                       ("prefill", k3.K3MOE_FFN_W4A4), ("skewed", k3.K3MOE_FFN_W4A4)])
def test_prefill_sampled(experts_2048, name, mode):
    """AUTO takes the W4A16 tensor-core GEMM here; W4A4 takes the block-scaled FP4
    GEMM and is checked against the oracle's A4 path.  The sample covers every
    token tile of the 32 most loaded experts (the hottest skewed expert has
    about 1,640 tokens, 13 tiles of 128)."""
    s = gen.CONFIGS[name]
    lg, xd, logits, xbits = device_inputs(name, s)
    r = host(run_layer(s, lg, xd, _weights(experts_2048), bufs=alloc_layer(s, mode=mode), mode=mode))
    assert r["status"][0] == 0
    idx, w, counts, offsets, perm, inv = _route_bucket_exact(s, logits, r)
    np.testing.assert_array_equal(r["out"], bf16_rne_bits_of(r["out_f32"]))
    sample, hot = hot_expert_sample(s, counts, offsets, perm, n_hot=32, tile=64, total=256)
    assert len(sample) >= 256
    for e in hot:  # the last bucket position of every hot expert is in the sample
        assert perm[offsets[e + 1] - 1] // s.k in set(sample.tolist())
    _staged(s, r, xbits, idx, w, inv, sample, a4=mode == k3.K3MOE_FFN_W4A4)
