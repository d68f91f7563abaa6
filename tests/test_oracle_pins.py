"""Pins for the oracle: each oracle function is checked against something other
than itself -- a published table, a closed form, brute force, or a library
routine -- so that a dropped term, a wrong sign or index or a transposed
operand fails at least one test.  CPU only."""
import math
import os

import numpy as np
import pytest
import torch

import gen
import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Library rounding: torch's float32 -> bfloat16 (round to nearest even)."""
    t = torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _bf16_values(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- scalar codecs
def test_e2m1_matches_ocp_table():
    rows = [l.split() for l in open(os.path.join(GOLD, "e2m1_values.txt")) if l[0] != "#"]
    assert len(rows) == 16
    for code, val in rows:
        got = oracle.e2m1(int(code))
        assert got == float(val)
        assert math.copysign(1.0, got) == math.copysign(1.0, float(val))  # code 8 is -0


def test_e8m0_all_bytes_match_library():
    # library decode of E8M0 (torch.float8_e8m0fnu) and the closed form 2^(b-127)
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
    for b in range(255):
        assert oracle.e8m0(b) == math.ldexp(1.0, b - 127) == lib[b]
    assert math.isnan(oracle.e8m0(255)) and math.isnan(lib[255])


def test_bf16_value_roundtrip_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = np.array([oracle.bf16_value(int(b)) for b in bits[::7]])
    sel = ref[::7]
    same = (got == sel) | (np.isnan(got) & np.isnan(sel))
    assert same.all()


def test_bf16_rne_matches_library_on_float32_values():
    rng = np.random.default_rng(3)
    v = np.concatenate([
        rng.standard_normal(4000).astype(np.float32),
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
        (rng.standard_normal(2000) * 1e-38).astype(np.float32),  # bf16 subnormals
        # exact ties: a bf16 value plus half its quantum
        (np.float32(1.0) + np.float32(2.0 ** -8)) * np.ones(1, np.float32),
        np.array([1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 3.0e38, -3.3e38, 0.0, -0.0], np.float32),
    ])
    ref = _bf16_bits_from_f32(v)
    got = np.array([oracle.bf16_rne(float(x)) for x in v], np.uint16)
    np.testing.assert_array_equal(got, ref)


def test_bf16_rne_double_inputs_hand_worked():
    cases = [
        (1.0 + 2.0 ** -8, 0x3F80),                 # tie -> even (1.0)
        (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),    # just above the tie -> up
        (1.0 + 3 * 2.0 ** -8, 0x3F82),             # tie between odd 0x3F81 and even 0x3F82
        (2.0 ** -133, 0x0001),                     # smallest subnormal
        (2.0 ** -134, 0x0000),                     # tie with zero -> even (0)
        (1.5 * 2.0 ** -134, 0x0001),
        (-(2.0 ** -134), 0x8000),
        ((2 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),    # tie at the top -> even = overflow to inf
        ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),    # largest finite
        (float("inf"), 0x7F80), (-float("inf"), 0xFF80), (-0.0, 0x8000),
    ]
    for v, bits in cases:
        assert oracle.bf16_rne(v) == bits, (v, hex(oracle.bf16_rne(v)), hex(bits))
    assert oracle.bf16_rne(float("nan")) & 0x7FFF > 0x7F80


def test_silu_library_and_identities():
    z = np.linspace(-30, 30, 601)
    ref = torch.nn.functional.silu(torch.from_numpy(z)).numpy()
    got = np.array([oracle.silu(float(a)) for a in z])
    np.testing.assert_allclose(got, ref, rtol=1e-14, atol=1e-300)
    assert oracle.silu(0.0) == 0.0
    for a in (0.3, 1.7, 9.0):  # silu(a) - silu(-a) = a
        assert abs(oracle.silu(a) - oracle.silu(-a) - a) < 1e-14


# ---------------------------------------------------------------- MXFP4 quantiser
_E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _brute_quant(vals: np.ndarray):
    """Brute force: scale from floor(log2 amax) - 2; each element takes the
    E2M1 code whose value times the scale is nearest, ties to the even code;
    magnitudes beyond 6 * scale saturate."""
    amax = np.abs(vals).max()
    if amax == 0:
        return 0, [0] * len(vals)
    shared = int(math.floor(math.log2(amax))) - 2
    shared = max(-127, min(127, shared))
    X = 2.0 ** shared
    codes = []
    for v in vals:
        best = None
        for c in range(8):
            d = abs(abs(v) - _E2M1[c] * X)
            if best is None or d < best[0] or (d == best[0] and c % 2 == 0 and best[1] % 2 == 1):
                best = (d, c)
        codes.append(best[1] | (8 if v < 0 else 0))
    return shared + 127, codes


def _unpack(codes: np.ndarray, n: int):
    out = []
    for i in range(n):
        b = int(codes[i // 2])
        out.append(b & 0xF if i % 2 == 0 else b >> 4)
    return out


def test_quant_hand_worked_block():
    # amax 6.5 -> floor(log2) = 2 -> shared exponent 0 -> X = 1
    vals = np.array([1.0, 0.25, 0.75, -5.0, 6.5, 2.5, -3.5, 1.25] + [0.0] * 24, np.float32)
    codes, scales = oracle.quant_mxfp4(_bf16_bits_from_f32(vals))
    assert scales[0] == 127
    # 1->1.0 (2); .25 tie->0 (0); .75 tie->1.0 (2); -5 tie->-4 (14); 6.5 sat->6 (7);
    # 2.5 tie->2 (4); -3.5 tie->-4 (14); 1.25 tie->1.0 (2)
    assert _unpack(codes, 8) == [2, 0, 2, 14, 7, 4, 14, 2]


def test_quant_brute_force_random_blocks():
    rng = np.random.default_rng(11)
    for trial in range(60):
        scale = 2.0 ** rng.integers(-20, 20)
        v = (rng.standard_normal(32) * scale).astype(np.float32)
        if trial % 5 == 0:
            v[rng.integers(0, 32, 8)] = 0.0
        if trial % 7 == 0:  # values exactly on E2M1 midpoints
            v[:8] = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0], np.float32) * scale
        bits = _bf16_bits_from_f32(v)
        vb = _bf16_values(bits)
        codes, scales = oracle.quant_mxfp4(bits)
        sb, bc = _brute_quant(vb)
        assert scales[0] == sb
        assert _unpack(codes, 32) == bc
        # decoded |v - q| <= half the local grid step (or saturation)
        X = 2.0 ** (int(scales[0]) - 127)
        dec = np.array([oracle.e2m1(c) * X for c in bc])
        assert np.all(np.abs(dec) <= 6 * X)
        assert np.all((np.abs(vb - dec) <= X) | (np.abs(vb) > 6 * X))


def test_quant_zero_block():
    codes, scales = oracle.quant_mxfp4(np.zeros(32, np.uint16))
    assert scales[0] == 0 and not codes.any()


# ---------------------------------------------------------------- routing
def _brute_topk(row: np.ndarray, k: int):
    order = sorted(range(len(row)), key=lambda e: (-float(row[e]), e))
    return order[:k]


@pytest.mark.parametrize("E,k", [(8, 2), (64, 16), (896, 16), (33, 33)])
def test_route_matches_brute_force_sort(E, k):
    rng = np.random.default_rng(E * 100 + k)
    T = 24
    l = rng.standard_normal((T, E)).astype(np.float32)
    l[3] = 0.5                                  # all equal
    l[4, : E // 2] = 1.0                        # many ties
    l[5] = np.round(l[5] * 2) / 2               # coarse values, ties
    l[6, 0], l[6, 1 % E] = -0.0, 0.0            # signed zeros compare equal
    s = gen.Shape(T, 32, 32, E, k)
    idx, w, bad = oracle.route(s, l)
    assert not bad.any()
    for t in range(T):
        assert idx[t].tolist() == _brute_topk(l[t], k)
        sel = l[t, idx[t]].astype(np.float64)
        ref = torch.softmax(torch.from_numpy(sel), 0).numpy()  # library softmax
        np.testing.assert_allclose(w[t], ref, rtol=1e-14)
        assert abs(w[t].sum() - 1.0) < 1e-14
        # renormalised full softmax restricted to the top k gives the same weights
        full = torch.softmax(torch.from_numpy(l[t].astype(np.float64)), 0).numpy()
        np.testing.assert_allclose(w[t], full[idx[t]] / full[idx[t]].sum(), rtol=1e-12)
    assert idx[3].tolist() == list(range(k)) and np.allclose(w[3], 1.0 / k)


def test_route_special_rows():
    E, k = 16, 4
    l = np.zeros((4, E), np.float32)
    l[0, 5] = np.nan
    l[1] = -np.inf
    l[2, 7] = np.inf
    l[2, 3] = np.inf
    l[3] = -np.inf
    l[3, 9] = 2.0
    s = gen.Shape(4, 32, 32, E, k)
    idx, w, bad = oracle.route(s, l)
    assert bad.tolist() == [1, 0, 0, 0]
    assert idx[0].tolist() == [0, 1, 2, 3] and np.allclose(w[0], 0.25)
    assert idx[1].tolist() == [0, 1, 2, 3] and np.allclose(w[1], 0.25)
    assert idx[2].tolist() == [3, 7, 0, 1] and w[2].tolist() == [0.5, 0.5, 0.0, 0.0]
    assert idx[3].tolist() == [9, 0, 1, 2] and w[3].tolist() == [1.0, 0.0, 0.0, 0.0]


# ---------------------------------------------------------------- bucketing
@pytest.mark.parametrize("T,E,k", [(1, 896, 16), (37, 8, 2), (300, 64, 8), (5, 3, 3)])
def test_bucket_invariants_and_library_sort(T, E, k):
    rng = np.random.default_rng(T + E)
    idx = rng.integers(0, E, (T, k)).astype(np.int32)
    if E > 3:
        idx[: T // 2] = rng.integers(0, 3, (T // 2, k))  # skew
    s = gen.Shape(T, 32, 32, E, k)
    counts, offsets, perm, inv = oracle.bucket(s, idx)
    flat = idx.ravel()
    np.testing.assert_array_equal(counts, np.bincount(flat, minlength=E))
    assert offsets[0] == 0 and offsets[-1] == T * k and np.all(np.diff(offsets) >= 0)
    np.testing.assert_array_equal(perm, np.argsort(flat, kind="stable"))  # library stable sort
    np.testing.assert_array_equal(inv[perm], np.arange(T * k))
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)


# ---------------------------------------------------------------- FFN + combine
def _dense_weights(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Dequantise with the OCP table (golden) and 2^(s-127) -- no oracle code."""
    table = np.array([float(l.split()[1]) for l in open(os.path.join(GOLD, "e2m1_values.txt"))
                      if l[0] != "#"])
    lo, hi = codes & 0xF, codes >> 4
    nib = np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)
    sc = np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=1)
    return table[nib] * sc


def _bf16_round_vec(v: np.ndarray) -> np.ndarray:
    return np.array([oracle.bf16_value(oracle.bf16_rne(float(a))) for a in v.ravel()]).reshape(v.shape)


def _dense_moe(s, logits, xbits, experts, a4=False, absent=()):
    """out = sum over ALL experts of gate_e(x) * FFN_e(x), gate_e = 0 off the top k,
    with dense dequantised matrices and library matmul/softmax."""
    x = _bf16_values(xbits).reshape(s.T, s.H)
    if a4:
        x = np.stack([_a4_values(xbits[t]) for t in range(s.T)])
    out = np.zeros((s.T, s.H))
    for t in range(s.T):
        top = _brute_topk(logits[t], s.k)
        sel = torch.softmax(torch.from_numpy(logits[t, top].astype(np.float64)), 0).numpy()
        gate = np.zeros(s.E)
        gate[top] = sel
        for e in range(s.E):
            if gate[e] == 0.0 or e in absent:
                continue
            W13 = _dense_weights(experts[e][0], experts[e][1])
            W2 = _dense_weights(experts[e][2], experts[e][3])
            g, u = W13[: s.I] @ x[t], W13[s.I:] @ x[t]
            h = _bf16_round_vec(torch.nn.functional.silu(torch.from_numpy(g)).numpy() * u)
            if a4:
                hb = np.array([oracle.bf16_rne(float(a)) for a in h], np.uint16)
                h = _a4_values(hb)
            out[t] += gate[e] * (W2 @ h)
    return out


def _a4_values(bits: np.ndarray) -> np.ndarray:
    codes, scales = oracle.quant_mxfp4(bits)
    n = bits.size
    table = [oracle.e2m1(c) for c in range(16)]
    return np.array([table[c] * 2.0 ** (int(scales[i // 32]) - 127)
                     for i, c in enumerate(_unpack(codes, n))])


def _tiny_case(T, H, I, E, k, seed):
    s = gen.Shape(T, H, I, E, k)
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    xbits = gen.normal_bf16_bits(seed, gen.stream(gen.KIND_X), T * H).reshape(T, H)
    a, b, c, d = gen.expert_arrays(H, I, 0, E, seed=seed)
    experts = {e: (a[e], b[e], c[e], d[e]) for e in range(E)}
    return s, logits, xbits, experts


@pytest.mark.parametrize("T,H,I,E,k,seed", [(4, 128, 64, 8, 2, 0), (3, 64, 96, 5, 3, 7),
                                             (6, 32, 32, 4, 4, 9), (2, 96, 32, 12, 1, 4)])
def test_layer_equals_dense_float64_moe(T, H, I, E, k, seed):
    s, logits, xbits, experts = _tiny_case(T, H, I, E, k, seed)
    W = oracle.Weights(E, experts)
    out, ob = oracle.moe_layer(s, logits, xbits, W)
    ref = _dense_moe(s, logits, xbits, experts)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    # the bf16 output is the RNE rounding of the float64 output
    assert all(oracle.bf16_rne(float(v)) == int(b) for v, b in zip(out.ravel(), ob.ravel()))


def test_layer_a4_equals_dense_float64_moe():
    s, logits, xbits, experts = _tiny_case(3, 64, 64, 6, 2, 5)
    W = oracle.Weights(s.E, experts)
    out, _ = oracle.moe_layer(s, logits, xbits, W, a4=True)
    ref = _dense_moe(s, logits, xbits, experts, a4=True)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_absent_expert_contributes_zero():
    s, logits, xbits, experts = _tiny_case(5, 64, 32, 6, 2, 3)
    idx, _, _ = oracle.route(s, logits)
    gone = int(idx[0, 0])
    exp2 = dict(experts)
    exp2[gone] = (experts[gone][0], None, experts[gone][2], experts[gone][3])
    out, _ = oracle.moe_layer(s, logits, xbits, oracle.Weights(s.E, exp2))
    ref = _dense_moe(s, logits, xbits, experts, absent=(gone,))
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_per_token_path_is_bit_identical_to_batched():
    s, logits, xbits, experts = _tiny_case(7, 64, 64, 5, 3, 8)
    W = oracle.Weights(s.E, experts)
    out, _ = oracle.moe_layer(s, logits, xbits, W)
    idx, w, _ = oracle.route(s, logits)
    for t in range(s.T):
        row = oracle.moe_token(s, xbits[t], idx[t], w[t], W)
        assert np.array_equal(row, out[t])


def _one_hot_matrix(rows, K, col_of_row, code, scale_byte):
    codes = np.zeros((rows, K // 2), np.uint8)
    for r in range(rows):
        c = col_of_row(r)
        codes[r, c // 2] |= np.uint8(code << (4 * (c % 2)))
    return codes, np.full((rows, K // 32), scale_byte, np.uint8)


def test_hand_worked_identity_experts():
    """T=1, H=I=32, E=3, k=2, logits (1, 1, .5): experts 0 and 1 win with weight 1/2.
    Expert 0: g = x, u = 2x, y = h.  Expert 1: g = -x, u = 1.5x, y_r = 0.5 h_{r+1}.
    Expected out_r = (h0_r + 0.5 h1_{r+1}) / 2, h = bf16(silu(g) u)."""
    H = I = 32
    x = np.array([(r - 16) / 8 for r in range(H)], np.float32)
    xbits = _bf16_bits_from_f32(x)[None, :]
    e0g = _one_hot_matrix(I, H, lambda r: r, 2, 127)     # +1.0
    e0u = _one_hot_matrix(I, H, lambda r: r, 2, 128)     # +1.0 * 2
    e1g = _one_hot_matrix(I, H, lambda r: r, 10, 127)    # -1.0
    e1u = _one_hot_matrix(I, H, lambda r: r, 5, 126)     # 3.0 * 0.5
    w2_0 = _one_hot_matrix(H, I, lambda r: r, 2, 127)
    w2_1 = _one_hot_matrix(H, I, lambda r: (r + 1) % I, 4, 125)  # 2.0 * 0.25
    experts = {
        0: (np.concatenate([e0g[0], e0u[0]]), np.concatenate([e0g[1], e0u[1]]), *w2_0),
        1: (np.concatenate([e1g[0], e1u[0]]), np.concatenate([e1g[1], e1u[1]]), *w2_1),
        2: (np.zeros((2 * I, H // 2), np.uint8), np.zeros((2 * I, 1), np.uint8),
            np.zeros((H, I // 2), np.uint8), np.zeros((H, 1), np.uint8)),
    }
    s = gen.Shape(1, H, I, 3, 2)
    logits = np.array([[1.0, 1.0, 0.5]], np.float32)
    out, _ = oracle.moe_layer(s, logits, xbits, oracle.Weights(3, experts))
    xv = x.astype(np.float64)
    silu = lambda z: z / (1.0 + np.exp(-z))
    h0 = _bf16_values(_bf16_bits_from_f32((silu(xv) * 2 * xv)))  # products exact in f32 here?
    h0 = np.array([oracle.bf16_value(oracle.bf16_rne(float(silu(a) * 2 * a))) for a in xv])
    h1 = np.array([oracle.bf16_value(oracle.bf16_rne(float(silu(-a) * 1.5 * a))) for a in xv])
    expect = 0.5 * h0 + 0.5 * (0.5 * np.roll(h1, -1))
    np.testing.assert_array_equal(out[0], expect)


def test_k1_output_equals_single_expert_output():
    s, logits, xbits, experts = _tiny_case(4, 64, 32, 6, 1, 12)
    W = oracle.Weights(s.E, experts)
    out, _ = oracle.moe_layer(s, logits, xbits, W)
    idx, w, _ = oracle.route(s, logits)
    counts, offsets, perm, inv = oracle.bucket(s, idx)
    Y = oracle.expert_ffn(s, xbits, W, offsets, perm)
    assert np.allclose(w, 1.0)
    np.testing.assert_array_equal(out, Y[inv])


# ---------------------------------------------------------------- byte accounting
def _pages():
    vals = {}
    for l in open(os.path.join(GOLD, "pages_numbers.txt")):
        if l.strip() and l[0] != "#":
            key, val = l.split()[:2]
            vals[key] = float(val)
    return vals


def test_expert_bytes_reproduce_pages_totals():
    """Packed MXFP4 bytes per expert = 3*H*I*(1/2 + 1/32).  At H*I = 7168*1536 it
    gives exactly the pages' 25.83 GB per token over 1,472 requests and the
    1.45 TB expert total over 82,432 expert weight sets."""
    p = _pages()
    assert p["moe_layers"] * p["experts_per_token"] == p["expert_requests_per_step"]
    be = gen.Shape(1, 7168, 1536, 896, 16).expert_bytes()
    assert be == 17547264
    assert round(be * p["expert_requests_per_step"] / 1e9, 2) == p["expert_bytes_per_token_gb"]
    assert round(be * p["expert_weight_sets"] / 1e12, 2) == p["expert_weights_total_tb"]
    assert p["expert_weight_sets"] == p["moe_layers"] * p["experts_per_layer"]
    assert abs(be / (3 * 7168 * 1536) - p["bytes_per_param_nominal"]) < 0.04


# ----------------------------------------------------------------------------- router
def _bf16_f64(bits):
    """bf16 bit patterns -> float64 through torch (a library decode, not the oracle's)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(
        torch.float64).numpy()


@pytest.mark.parametrize("T,H,E", [(3, 128, 8), (5, 512, 40), (2, 7168, 16)])
def test_router_logits_match_library_matmul(T, H, E):
    """The router scores against numpy's float64 matrix product of the library-
    decoded bf16 operands (a different summation order: agreement to 1e-13 of
    the sum of |products|)."""
    s = gen.Shape(T, H, 64, E, 1)
    x = gen.normal_bf16_bits(11, gen.stream(gen.KIND_X), T * H).reshape(T, H)
    wr = gen.make_router(s)
    got = oracle.router_logits(s, x, wr)
    xv, wv = _bf16_f64(x), _bf16_f64(wr)
    ref = xv @ wv.T
    mag = np.abs(xv) @ np.abs(wv).T
    assert np.all(np.abs(got - ref) <= 1e-13 * mag)
    assert got.shape == (T, E)


def test_router_logits_exact_on_integers_and_one_hot():
    """Small integers are exact in bf16 and their products and sums exact in
    double: the scores equal numpy's int64 product bit for bit.  A one-hot token
    picks one column of the router matrix (catches a transposed operand)."""
    rng = np.random.default_rng(3)
    T, H, E = 4, 256, 24
    s = gen.Shape(T, H, 64, E, 1)
    xi = rng.integers(-15, 16, (T, H))
    wi = rng.integers(-15, 16, (E, H))
    as_bits = lambda a: (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    got = oracle.router_logits(s, as_bits(xi), as_bits(wi))
    np.testing.assert_array_equal(got, (xi @ wi.T).astype(np.float64))
    oh = np.zeros((T, H))
    cols = [0, 7, 100, 255]
    for t, c in enumerate(cols):
        oh[t, c] = 1.0
    got = oracle.router_logits(s, as_bits(oh), as_bits(wi))
    np.testing.assert_array_equal(got, wi[:, cols].T.astype(np.float64))


def test_router_routes_on_the_fp32_rounding_of_its_scores():
    """Router then route = the route (itself pinned by brute force) applied to the
    scores rounded once to float32 by numpy."""
    s = gen.Shape(6, 512, 64, 96, 16)
    x = gen.normal_bf16_bits(12, gen.stream(gen.KIND_X), s.T * s.H).reshape(s.T, s.H)
    wr = gen.make_router(s)
    l64, l32, idx, w, bad = oracle.router(s, x, wr)
    np.testing.assert_array_equal(l64, oracle.router_logits(s, x, wr))
    np.testing.assert_array_equal(l32, l64.astype(np.float32))
    idx2, w2, _ = oracle.route(s, l64.astype(np.float32))
    np.testing.assert_array_equal(idx, idx2)
    np.testing.assert_array_equal(w, w2)
    assert not bad.any()
    # scores have the decode workload's spread (standard deviation about 2)
    assert 1.5 < float(np.std(l64)) < 2.5


# ----------------------------------------------------------------------------- FFN halves
@pytest.mark.parametrize("a4", [False, True])
def test_ffn_halves_compose_to_the_ffn_and_match_dense_math(a4):
    """gate/up then down on its own h is bitwise the oracle's expert FFN; hpre is
    silu(g) u from dense dequantised matrices (golden E2M1 table, library silu)
    to 1e-12 and h its bf16 rounding; down on arbitrary bf16 rows is the dense
    product W2 h (A4: of the h row's MXFP4 values)."""
    s, logits, xbits, experts = _tiny_case(5, 128, 64, 6, 2, 11)
    W = oracle.Weights(s.E, experts)
    idx, w, _ = oracle.route(s, logits)
    counts, offsets, perm, inv = oracle.bucket(s, idx)
    Y, h_ffn = oracle.expert_ffn(s, xbits, W, offsets, perm, a4=a4, want_h=True)
    hpre, h, sums = oracle.expert_gateup(s, xbits, W, offsets, perm, a4=a4, sums=True)
    np.testing.assert_array_equal(h, h_ffn)
    np.testing.assert_array_equal(oracle.expert_down(s, h, W, offsets, a4=a4), Y)
    assert all(oracle.bf16_rne(float(v)) == int(b) for v, b in zip(hpre.ravel(), h.ravel()))
    x = _bf16_values(xbits).reshape(s.T, s.H)
    hr = gen.normal_bf16_bits(13, gen.stream(gen.KIND_X), s.T * s.k * s.I).reshape(s.T * s.k, s.I)
    Yr = oracle.expert_down(s, hr, W, offsets, a4=a4)
    for e in range(s.E):
        W13 = _dense_weights(experts[e][0], experts[e][1])
        W2 = _dense_weights(experts[e][2], experts[e][3])
        for p in range(offsets[e], offsets[e + 1]):
            xt = _a4_values(xbits[perm[p] // s.k]) if a4 else x[perm[p] // s.k]
            g, u = W13[: s.I] @ xt, W13[s.I:] @ xt
            ref = torch.nn.functional.silu(torch.from_numpy(g)).numpy() * u
            np.testing.assert_allclose(hpre[p], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
            for key, ref_v in (("g", g), ("u", u), ("gabs", np.abs(W13[: s.I]) @ np.abs(xt)),
                               ("uabs", np.abs(W13[s.I:]) @ np.abs(xt))):
                np.testing.assert_allclose(sums[key][p], ref_v, rtol=1e-12, atol=1e-12 * np.abs(ref_v).max())
            hv = _a4_values(hr[p]) if a4 else _bf16_values(hr[p])
            ref_y = W2 @ hv
            np.testing.assert_allclose(Yr[p], ref_y, rtol=1e-12, atol=1e-12 * np.abs(ref_y).max())
