"""The staged FFN checker itself (CPU): h values that any fp32 summation within
the stated bound could produce pass, and planted mistakes in h are caught."""
import numpy as np
import pytest

import gen
import mxfp4_expert_ffn_router_gb300 as k3
import oracle
from ffn_check import _bf16_directed, _key, check_h, gamma


def _case():
    s = gen.Shape(6, 256, 64, 5, 2)
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((s.T, s.E)).astype(np.float32)
    xbits = gen.normal_bf16_bits(15, gen.stream(gen.KIND_X), s.T * s.H).reshape(s.T, s.H)
    arrs = gen.expert_arrays(s.H, s.I, 0, s.E)
    W = oracle.Weights(s.E, {e: tuple(z[e] for z in arrs) for e in range(s.E)})
    idx, w, _ = oracle.route(s, logits)
    counts, offsets, perm, inv = oracle.bucket(s, idx)
    hpre, h, sums = oracle.expert_gateup(s, xbits, W, offsets, perm, sums=True)
    return s, hpre, h, sums


def test_directed_rounding_brackets_every_value():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000), [0.0, -0.0, 1.0, -1.0]])
    lo, hi = _bf16_directed(v, up=False), _bf16_directed(v, up=True)
    assert np.all(lo <= hi) and np.all(hi - lo <= 1)
    # the oracle's (pinned) rounding to nearest lies between them
    rne = _key(np.array([oracle.bf16_rne(float(a)) for a in v], np.uint16))
    assert np.all((lo <= rne) & (rne <= hi))


def test_oracle_h_and_fp32_perturbations_pass():
    s, hpre, h, sums = _case()
    gb = gamma(s, k3.K3MOE_FFN_GEMV)
    check_h(h, sums, gb)
    # g and u off by a fraction of the bound: the rounding of silu(g') u' still passes
    g2 = sums["g"] + 0.5 * gb * sums["gabs"]
    u2 = sums["u"] - 0.5 * gb * sums["uabs"]
    v = g2 / (1.0 + np.exp(-g2)) * u2
    h2 = np.array([oracle.bf16_rne(float(a)) for a in v.ravel()], np.uint16).reshape(v.shape)
    check_h(h2, sums, gb)


@pytest.mark.parametrize("steps", [2, -3, 40])
def test_planted_h_mistakes_are_caught(steps):
    s, hpre, h, sums = _case()
    bad = h.copy()
    i = int(np.argmax(np.abs(hpre)))  # a large |h|: its bound spans at most two bf16 values
    r, c = np.unravel_index(i, h.shape)
    bad[r, c] = np.uint16(int(bad[r, c]) + steps)
    with pytest.raises(AssertionError):
        check_h(bad, sums, gamma(s, k3.K3MOE_FFN_GEMV))


def test_sign_flip_is_caught():
    s, hpre, h, sums = _case()
    bad = h.copy()
    i = int(np.argmax(np.abs(hpre)))
    bad.ravel()[i] ^= np.uint16(0x8000)
    with pytest.raises(AssertionError):
        check_h(bad, sums, gamma(s, k3.K3MOE_FFN_GEMM))
