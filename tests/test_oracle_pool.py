"""The parallel oracle runner used by the full-size parity samples: its
assembled rows are bitwise the oracle's own batched layer (route, bucket, FFN,
combine) on the same tokens, and bitwise the oracle's per-token path."""
import numpy as np

import gen
import oracle
from oracle_pool import hot_expert_sample, sample_layer


def test_sample_layer_is_the_oracle_layer():
    s = gen.Shape(64, 256, 128, 16, 4)
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((s.T, s.E)).astype(np.float32)
    xbits = gen.normal_bf16_bits(9, gen.stream(gen.KIND_X), s.T * s.H).reshape(s.T, s.H)
    idx, w, _ = oracle.route(s, logits)
    counts, offsets, perm, inv = oracle.bucket(s, idx)
    sample, hot = hot_expert_sample(s, counts, offsets, perm, n_hot=4, tile=8, total=24)
    assert len(sample) >= 24 and sample[0] == 0 and sample[-1] == s.T - 1
    for e in hot:
        for p in range(offsets[e], offsets[e + 1], 8):
            assert perm[p] // s.k in sample
    for a4 in (False, True):
        Y, out, inv_s = sample_layer(s, xbits, idx, w, sample, a4=a4, nproc=2)
        arrs = gen.expert_arrays(s.H, s.I, 0, s.E)
        W = oracle.Weights(s.E, {e: tuple(z[e] for z in arrs) for e in range(s.E)})
        sub = gen.Shape(len(sample), s.H, s.I, s.E, s.k)
        c2, o2, p2, i2 = oracle.bucket(sub, idx[sample])
        Yb = oracle.expert_ffn(sub, xbits[sample], W, o2, p2, a4=a4)
        np.testing.assert_array_equal(Y, Yb)
        np.testing.assert_array_equal(inv_s, i2)
        for i, t in enumerate(sample):
            ref = oracle.moe_token(s, xbits[t], idx[t], w[t], W, a4=a4)
            np.testing.assert_array_equal(out[i], ref)


def test_staged_sample_uses_the_given_h():
    """With the oracle's own h in place of the GPU's, the staged rows are the
    oracle's layer bit for bit, and the h it reports is the oracle's rounding."""
    s = gen.Shape(32, 128, 64, 12, 3)
    rng = np.random.default_rng(6)
    logits = rng.standard_normal((s.T, s.E)).astype(np.float32)
    xbits = gen.normal_bf16_bits(14, gen.stream(gen.KIND_X), s.T * s.H).reshape(s.T, s.H)
    idx, w, _ = oracle.route(s, logits)
    counts, offsets, perm, inv = oracle.bucket(s, idx)
    arrs = gen.expert_arrays(s.H, s.I, 0, s.E)
    W = oracle.Weights(s.E, {e: tuple(z[e] for z in arrs) for e in range(s.E)})
    for a4 in (False, True):
        hpre, h, sums = oracle.expert_gateup(s, xbits, W, offsets, perm, a4=a4, sums=True)
        sample = np.array([0, 3, 7, 31])
        d = sample_layer(s, xbits, idx, w, sample, a4=a4, nproc=2, h_gpu=h, inv_gpu=inv)
        Y, out, inv_s = sample_layer(s, xbits, idx, w, sample, a4=a4, nproc=2)
        np.testing.assert_array_equal(d["Y"], Y)
        np.testing.assert_array_equal(d["out"], out)
        np.testing.assert_array_equal(d["h_ref"], d["h_gpu"])
        for key in ("g", "u", "gabs", "uabs"):  # the sub-batch's rows of the whole batch's sums
            np.testing.assert_array_equal(d["sums"][key][inv_s[np.arange(len(sample) * s.k)]],
                                          sums[key][inv[(sample[:, None] * s.k + np.arange(s.k)[None, :]).ravel()]])
        a_full = sample[:, None] * s.k + np.arange(s.k)[None, :]
        np.testing.assert_array_equal(d["h_gpu"][inv_s[np.arange(len(sample) * s.k)]], h[inv[a_full.ravel()]])
