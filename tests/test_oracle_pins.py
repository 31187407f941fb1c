"""Pins of the fp64 oracle against what the pages and the mathematics fix.

None of these tests re-types an oracle formula: each compares the oracle with
a hand-derived value, a closed form, an invariant, a special case that reduces
to a textbook routine, or a brute-force evaluation written as plain loops.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as O

RNG = np.random.default_rng(1234)


# ----------------------------------------------------------------------------
# number formats
# ----------------------------------------------------------------------------

def test_bf16_bits_known_values():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x4300, 0x3C23], dtype=np.uint16)
    want = [1.0, -2.0, 0.0, -0.0, 128.0, 0.00994873046875]
    assert O.bf16_bits_to_f64(bits).tolist() == want


def test_f32_to_bf16_round_half_even():
    # 1 + 2^-8 lies half-way between 1 and 1 + 2^-7: ties to the even code 0x3F80.
    # 1 + 3*2^-8 lies half-way between 1 + 2^-7 (odd code) and 1 + 2^-6: goes up.
    # 1 + 2^-8 + 2^-20 is above the half-way point: rounds up.
    v = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20, -(1 + 2 ** -8)], dtype=np.float32)
    assert O.f32_to_bf16_bits(v).tolist() == [0x3F80, 0x3F82, 0x3F81, 0xBF80]


# ----------------------------------------------------------------------------
# PackedInt4Linear storage
# ----------------------------------------------------------------------------

def test_unpack_golden_words(golden_dir):
    with open(os.path.join(golden_dir, "int4_words.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        assert int(c["int32"]) & 0xFFFFFFFF == int(c["word_hex"], 16)
        got = O.unpack_int4(np.array([[c["int32"]]], dtype=np.int32))[0].tolist()
        assert got == c["values"], c["word_hex"]


def test_unpack_every_value_in_every_position():
    # one non-zero nibble per word: all 16 codes x 8 positions
    for j in range(8):
        for code in range(16):
            word = np.array([[code << (4 * j)]], dtype=np.uint32).view(np.int32)
            got = O.unpack_int4(word)[0]
            want = np.zeros(8, dtype=np.int64)
            want[j] = code - 16 if code >= 8 else code
            assert got.tolist() == want.tolist()


def test_pack_unpack_round_trip():
    w = RNG.integers(0, 2 ** 32, size=(512, 2048), dtype=np.uint64).astype(np.uint32).view(np.int32)
    assert np.array_equal(O.pack_int4(O.unpack_int4(w)), w)
    q = RNG.integers(-8, 8, size=(33, 64))
    assert np.array_equal(O.unpack_int4(O.pack_int4(q)), q)
    # columns of a multi-word row land at 8i+j
    q = np.arange(16) % 16 - 8  # -8..7
    words = O.pack_int4(q[None, :])
    assert O.unpack_int4(words)[0].tolist() == q.tolist()


def test_pack_rejects_out_of_range():
    with pytest.raises(ValueError):
        O.pack_int4(np.array([[8] * 8]))
    with pytest.raises(ValueError):
        O.pack_int4(np.array([[0] * 7]))


def test_dequantize_group_scales():
    # row 0: all q = 1, group scales 0.5 / 2.0 -> 32 copies of each
    q = np.ones((2, 64), dtype=np.int64)
    q[1] = -8
    packed = O.pack_int4(q)
    scale = np.array([[0x3F00, 0x4000], [0x3F80, 0x3C23]], dtype=np.uint16)  # 0.5, 2.0 ; 1.0, 0.00994873046875
    W = O.dequantize(packed, scale)
    assert W[0, :32].tolist() == [0.5] * 32 and W[0, 32:].tolist() == [2.0] * 32
    assert W[1, :32].tolist() == [-8.0] * 32
    assert W[1, 32:].tolist() == [-8 * 0.00994873046875] * 32
    with pytest.raises(ValueError):
        O.dequantize(packed, scale[:, :1])


# ----------------------------------------------------------------------------
# router
# ----------------------------------------------------------------------------

def test_sigmoid_closed_forms():
    assert O.sigmoid(0.0) == 0.5
    assert abs(O.sigmoid(math.log(3.0)) - 0.75) < 1e-15
    z = RNG.normal(size=100) * 5
    assert np.allclose(O.sigmoid(-z), 1 - O.sigmoid(z), atol=1e-15)


def _brute_route(x, W, b, k, renorm):
    T, E = x.shape[0], W.shape[0]
    idx, wts = [], []
    for t in range(T):
        s = []
        for e in range(E):
            z = sum(float(x[t, h]) * float(W[e, h]) for h in range(x.shape[1]))
            s.append(1.0 / (1.0 + math.exp(-z)))
        ranked = sorted(range(E), key=lambda e: (-(s[e] + float(b[e])), e))[:k]
        w = [s[e] for e in ranked]
        if renorm:
            tot = sum(w) + 1e-20
            w = [v / tot for v in w]
        idx.append(ranked)
        wts.append(w)
    return np.array(idx), np.array(wts)


@pytest.mark.parametrize("renorm", [True, False])
def test_route_matches_brute_force(renorm):
    x = RNG.normal(size=(6, 24))
    W = RNG.normal(size=(10, 24)) * 0.3
    b = RNG.normal(size=10) * 0.05
    rt = O.route(x, W, b, 3, renorm)
    idx, w = _brute_route(x, W, b, 3, renorm)
    assert np.array_equal(rt.idx, idx)
    assert np.allclose(rt.weight, w, rtol=1e-13, atol=0)


def test_route_ranks_by_biased_score_weights_by_unbiased():
    # x = 0: every logit is 0 and every affinity 0.5, so the bias alone ranks.
    E, k = 6, 2
    b = np.array([0.0, 0.3, -0.1, 0.2, 0.0, 0.05])
    rt = O.route(np.zeros((1, 4)), np.ones((E, 4)), b, k, renorm=False)
    assert rt.idx[0].tolist() == [1, 3]
    assert rt.weight[0].tolist() == [0.5, 0.5]          # unbiased affinities
    rt = O.route(np.zeros((1, 4)), np.ones((E, 4)), b, k, renorm=True)
    assert rt.weight[0].tolist() == [0.5 / (1.0 + 1e-20)] * 2


def test_route_ties_go_to_lower_expert():
    b = np.zeros(5)
    rt = O.route(np.zeros((1, 3)), np.zeros((5, 3)), b, 3)
    assert rt.idx[0].tolist() == [0, 1, 2]


def test_route_k_equals_E_and_k_one():
    x = RNG.normal(size=(5, 16))
    W = RNG.normal(size=(7, 16))
    b = RNG.normal(size=7) * 0.01
    rt = O.route(x, W, b, 7)
    assert all(sorted(r) == list(range(7)) for r in rt.idx.tolist())
    assert np.allclose(rt.weight.sum(1), 1.0, atol=1e-15)
    rt1 = O.route(x, W, b, 1)
    assert np.all(rt1.weight == 1.0)    # s / (s + 1e-20) == 1 in float64
    assert np.all(np.isinf(O.topk_gap(rt.r, 7)))


def test_renorm_sums_to_one_and_gap():
    x = RNG.normal(size=(50, 32))
    W = RNG.normal(size=(20, 32)) * 0.2
    rt = O.route(x, W, np.zeros(20), 4)
    assert np.allclose(rt.weight.sum(1), 1.0, rtol=0, atol=4e-16)
    gap = O.topk_gap(rt.r, 4)
    for t in range(50):
        srt = sorted(rt.r[t], reverse=True)
        assert gap[t] == srt[3] - srt[4]


# ----------------------------------------------------------------------------
# dispatch
# ----------------------------------------------------------------------------

def _random_topk(T, E, k):
    return np.stack([RNG.permutation(E)[:k] for _ in range(T)])


@pytest.mark.parametrize("T,E,k", [(1, 4, 2), (37, 9, 3), (200, 16, 8), (64, 64, 1)])
def test_dispatch_invariants_and_brute_force(T, E, k):
    idx = _random_topk(T, E, k)
    d = O.dispatch(idx, E)
    assert d.counts.sum() == T * k and d.offsets[-1] == T * k and d.offsets[0] == 0
    assert np.array_equal(np.diff(d.offsets), d.counts)
    assert np.array_equal(np.bincount(d.row_token, minlength=T), np.full(T, k))
    # brute force: sort (expert, token) pairs
    pairs = sorted((int(idx[t, j]), t, j) for t in range(T) for j in range(k))
    assert [p[1] for p in pairs] == d.row_token.tolist()
    assert [p[2] for p in pairs] == d.row_slot.tolist()
    # inverse permutation: gather then scatter is the identity
    for t in range(T):
        for j in range(k):
            r = d.inv_row[t * k + j]
            assert d.row_token[r] == t and d.row_slot[r] == j
            assert d.offsets[idx[t, j]] <= r < d.offsets[idx[t, j] + 1]
    assert sorted(d.inv_row.tolist()) == list(range(T * k))


def test_dispatch_idle_experts():
    idx = np.array([[2, 0], [0, 2], [2, 0]])
    d = O.dispatch(idx, 5)
    assert d.counts.tolist() == [3, 0, 3, 0, 0]
    assert d.offsets.tolist() == [0, 3, 3, 6, 6, 6]
    assert d.row_token.tolist() == [0, 1, 2, 0, 1, 2]
    assert d.row_slot.tolist() == [1, 0, 1, 0, 1, 0]


# ----------------------------------------------------------------------------
# act_bits = 8
# ----------------------------------------------------------------------------

def test_quantizer_golden(golden_dir):
    with open(os.path.join(golden_dir, "quantizer_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        q, s = O.quantize_rows_int8(np.array([c["v"]], dtype=np.float32))
        assert q[0].tolist() == c["q"]
        assert float(s[0]) == c["scale"]


def _f32_half_ulp(x) -> Fraction:
    """Half the spacing of the float32 values around x (normal range)."""
    return Fraction(2) ** (math.floor(math.log2(abs(float(x)))) - 24)


def test_quantizer_float32_tie_case_by_exact_arithmetic(golden_dir):
    # The golden row [a, a/2, -a/2] that separates float32 from float64
    # quantisation, checked with exact rationals: the stored scale is the
    # float32 nearest a/127; the exact quotient (a/2)/s is not a tie, but the
    # float32 nearest to it is the tie 63.5, so rint gives the even code 64.
    with open(os.path.join(golden_dir, "quantizer_cases.json")) as f:
        c = json.load(f)["cases"][4]
    a, v, s = Fraction(c["v"][0]), Fraction(c["v"][1]), Fraction(c["scale"])
    assert float(np.float32(c["scale"])) == c["scale"]          # s is a float32 value
    assert abs(s - a / 127) <= _f32_half_ulp(s)
    tie = Fraction(127, 2)
    quo = v / s
    assert quo < tie and tie - quo < _f32_half_ulp(tie)
    assert c["q"] == [127, 64, -64]


def test_quantizer_identity_on_int8_rows():
    x = RNG.integers(-127, 128, size=(20, 96)).astype(np.float32)
    x[:, 5] = 127.0
    q, s = O.quantize_rows_int8(x)
    assert np.all(s == 1.0) and np.array_equal(q, x.astype(np.int8))


def test_quantizer_bounds_and_rounding():
    v = (RNG.normal(size=(40, 300)) * RNG.uniform(0.01, 100, size=(40, 1))).astype(np.float32)
    q, s = O.quantize_rows_int8(v)
    assert q.dtype == np.int8 and np.abs(q.astype(int)).max() <= 127
    # amax maps to +-127 and every code is within half a step of v / scale
    for r in range(40):
        sc = Fraction(float(s[r]))
        assert sc == Fraction(float(np.float32(np.abs(v[r]).max()) / np.float32(127)))
        for c in range(0, 300, 7):
            assert abs(Fraction(float(v[r, c])) / sc - int(q[r, c])) <= Fraction(1, 2) + Fraction(1, 10 ** 5)
    # rows are independent
    q2, s2 = O.quantize_rows_int8(v[::-1])
    assert np.array_equal(q2, q[::-1]) and np.array_equal(s2, s[::-1])


def _brute_partials(qx, qw):
    R, K = qx.shape
    N = qw.shape[0]
    P = np.zeros((R, N, K // 32), dtype=np.int64)
    for r in range(R):
        for n in range(N):
            for c in range(K):
                P[r, n, c // 32] += int(qx[r, c]) * int(qw[n, c])
    return P


def test_group_partials_brute_force_and_extremes():
    qx = RNG.integers(-127, 128, size=(3, 96)).astype(np.int8)
    qw = RNG.integers(-8, 8, size=(5, 96))
    P = O.int4_group_partials(qx, O.pack_int4(qw))
    assert np.array_equal(P, _brute_partials(qx, qw))
    # worst-case magnitude 32*8*127 per group
    qx = np.full((1, 64), 127, dtype=np.int8)
    qw = np.full((2, 64), -8)
    assert O.int4_group_partials(qx, O.pack_int4(qw)).tolist() == [[[-32512, -32512]] * 2]


def test_group_partials_int32_bound_rejected():
    K = 2 ** 31 // (8 * 127) // 32 * 32 + 32   # first multiple of 32 with K*8*127 >= 2^31
    assert K * 8 * 127 >= 2 ** 31 and (K - 32) * 8 * 127 < 2 ** 31
    with pytest.raises(ValueError):
        O.int4_group_partials(np.zeros((1, K), np.int8), np.zeros((1, K // 8), np.int32))


# ----------------------------------------------------------------------------
# the int16 / int64 reading of act_bits = 16
# ----------------------------------------------------------------------------

def test_quantizer_int16_identity_on_int16_rows():
    x = RNG.integers(-32767, 32768, size=(12, 96)).astype(np.float32)
    x[:, 7] = -32767.0
    q, s = O.quantize_rows_int16(x)
    assert q.dtype == np.int16
    assert np.all(s == 1.0) and np.array_equal(q, x.astype(np.int16))


def test_quantizer_int16_bounds_and_rounding():
    v = (RNG.normal(size=(20, 200)) * RNG.uniform(0.01, 100, size=(20, 1))).astype(np.float32)
    v[3] = 0.0
    q, s = O.quantize_rows_int16(v)
    assert np.abs(q.astype(int)).max() <= 32767
    assert s[3] == 0 and not q[3].any()
    for r in range(20):
        if r == 3:
            continue
        sc = Fraction(float(s[r]))
        assert sc == Fraction(float(np.float32(np.abs(v[r]).max()) / np.float32(32767)))
        assert np.abs(q[r].astype(int)).max() == 32767
        for c in range(0, 200, 9):
            # float32 division: the quotient (up to 32767) carries 2^-9 of rounding
            assert abs(Fraction(float(v[r, c])) / sc - int(q[r, c])) <= Fraction(1, 2) + Fraction(1, 2 ** 8)
    # half steps round to even codes (scale 1)
    q, s = O.quantize_rows_int16(np.array([[32767.0, 0.5, 1.5, 2.5, -2.5, -100.5]], np.float32))
    assert s[0] == 1.0 and q[0].tolist() == [32767, 0, 2, 2, -2, -100]


def test_quantizer_int16_float32_tie_case_by_exact_arithmetic():
    # the row [a, a/2, -a/2] separates float32 from float64 quantisation: the
    # exact quotient (a/2)/s lies below the tie 16383.5 by less than half a
    # float32 ulp there, so the float32 quotient is the tie itself and rint
    # gives the even code 16384 (float64 would give 16383)
    a = np.float32(1.925695538520813)
    q, s = O.quantize_rows_int16(np.array([[a, a / np.float32(2), -a / np.float32(2)]], np.float32))
    assert q[0].tolist() == [32767, 16384, -16384]
    sc, v = Fraction(float(s[0])), Fraction(float(a / np.float32(2)))
    assert abs(sc - Fraction(float(a)) / 32767) <= _f32_half_ulp(s[0])
    tie = Fraction(32767, 2)
    assert v / sc < tie and tie - v / sc < _f32_half_ulp(tie)


def test_int16_group_partials_brute_force_and_extremes():
    q16 = RNG.integers(-32767, 32768, size=(3, 96)).astype(np.int16)
    qw = RNG.integers(-8, 8, size=(4, 96))
    assert np.array_equal(O.int16_group_partials(q16, O.pack_int4(qw)), _brute_partials(q16, qw))
    q16 = np.full((1, 64), -32767, dtype=np.int16)
    qw = np.full((1, 64), -8)
    assert O.int16_group_partials(q16, O.pack_int4(qw)).tolist() == [[[32 * 8 * 32767] * 2]]
    K = 2 ** 31 // (8 * 32767) // 32 * 32 + 32   # first multiple of 32 past the int32 bound
    assert K * 8 * 32767 >= 2 ** 31 and (K - 32) * 8 * 32767 < 2 ** 31
    with pytest.raises(ValueError):
        O.int16_group_partials(np.zeros((1, K), np.int16), np.zeros((1, K // 8), np.int32))


def test_int4_linear_int16_reduces_to_an_integer_matmul():
    # integer rows holding +-32767 (scale 1) and unit weight scales: y is the
    # integer product x qw^T, computed here with Python integers
    x = RNG.integers(-32767, 32768, size=(4, 64))
    x[:, 0] = 32767
    qw = RNG.integers(-8, 8, size=(3, 64))
    ones = np.full((3, 2), ONE, dtype=np.uint16)
    y = O.int4_linear_int16(x.astype(np.float64), O.pack_int4(qw), ones)
    want = [[sum(int(x[r, c]) * int(qw[n, c]) for c in range(64)) for n in range(3)] for r in range(4)]
    assert y.tolist() == want
    # a group scale multiplies its group's partial only
    sc = ones.copy()
    sc[1, 1] = 0x4000  # 2.0 for group 1 of output 1
    y2 = O.int4_linear_int16(x.astype(np.float64), O.pack_int4(qw), sc)
    g1 = [sum(int(x[r, c]) * int(qw[1, c]) for c in range(32, 64)) for r in range(4)]
    assert np.array_equal(y2[:, 1] - y[:, 1], np.array(g1, dtype=np.float64))


# ----------------------------------------------------------------------------
# PackedInt4Linear and the expert
# ----------------------------------------------------------------------------

ONE = 0x3F80  # bf16 1.0


def test_int4_linear_unit_scales_is_integer_matmul():
    qw = RNG.integers(-8, 8, size=(7, 64))
    u = RNG.integers(-127, 128, size=(4, 64)).astype(np.float64)
    u[:, 0] = 127
    scale = np.full((7, 2), ONE, dtype=np.uint16)
    want = [[sum(int(u[r, c]) * int(qw[n, c]) for c in range(64)) for n in range(7)] for r in range(4)]
    y16 = O.int4_linear(u, O.pack_int4(qw), scale, 16)
    y8 = O.int4_linear(u, O.pack_int4(qw), scale, 8)
    assert y16.tolist() == want
    assert y8.tolist() == want          # sc = 1, q = u: the integer accumulator itself


def test_int4_linear_exact_mode_close_to_w4a16():
    qw = RNG.integers(-8, 8, size=(16, 256))
    scale = O.f32_to_bf16_bits(RNG.uniform(0.002, 0.01, size=(16, 8)).astype(np.float32))
    u = O.round_bf16(RNG.normal(size=(5, 256)))
    y16 = O.int4_linear(u, O.pack_int4(qw), scale, 16)
    y8 = O.int4_linear(u, O.pack_int4(qw), scale, 8)
    # int8 activations carry a relative error below one half step (1/254 of max|u|)
    bound = (np.abs(u).max(1, keepdims=True) / 254) * np.abs(O.dequantize(O.pack_int4(qw), scale)).sum(1)[None, :]
    assert np.all(np.abs(y8 - y16) <= bound * 1.0001)


def _brute_expert(u, ex, act_bits=16):
    """Plain loops of down(SiLU(gate u) * up u) with explicit unpack and scales."""
    def lin(vec, packed, scale):
        N, K8 = packed.shape
        out = []
        for n in range(N):
            acc = 0.0
            for i in range(K8):
                word = int(packed[n, i]) & 0xFFFFFFFF
                for j in range(8):
                    code = (word >> (4 * j)) & 0xF
                    qv = code - 16 if code >= 8 else code
                    c = 8 * i + j
                    acc += vec[c] * qv * float(O.bf16_bits_to_f64(scale[n, c // 32]))
            out.append(acc)
        return out
    g = lin(u, ex["gate_packed"], ex["gate_scale"])
    up = lin(u, ex["up_packed"], ex["up_scale"])
    h = [gv / (1.0 + math.exp(-gv)) * uv for gv, uv in zip(g, up)]
    return lin(h, ex["down_packed"], ex["down_scale"])


def _random_expert(D, I):
    def sc(n, k):
        return O.f32_to_bf16_bits(RNG.uniform(0.02, 0.2, size=(n, k // 32)).astype(np.float32))
    return {
        "gate_packed": O.pack_int4(RNG.integers(-8, 8, size=(I, D))), "gate_scale": sc(I, D),
        "up_packed": O.pack_int4(RNG.integers(-8, 8, size=(I, D))), "up_scale": sc(I, D),
        "down_packed": O.pack_int4(RNG.integers(-8, 8, size=(D, I))), "down_scale": sc(D, I),
    }


def test_expert_matches_brute_force_loops():
    ex = _random_expert(64, 32)
    u = O.round_bf16(RNG.normal(size=(2, 64)))
    y = O.expert_ffn(u, ex, 16)
    for r in range(2):
        assert np.allclose(y[r], _brute_expert(u[r], ex), rtol=1e-12, atol=1e-12)


def _brute_q8(vals):
    """Per-row int8 codes and scale of a list of values, one float32 operation at a time."""
    a = np.float32(0.0)
    for v in vals:
        a = max(a, abs(np.float32(v)))
    s = np.float32(a / np.float32(127))
    if s == 0:
        return [0] * len(vals), s
    return [int(min(max(np.rint(np.float32(np.float32(v) / s)), -127), 127)) for v in vals], s


def _brute_expert_exact(u, ex):
    """Plain loops of the act_bits=8 expert: each linear takes the bf16 value
    of its input, quantises it per row to int8, sums integer products per
    32-column group, and scales by the group scale and the row scale."""
    def lin(vec, packed, scale):
        q, sx = _brute_q8(O.round_bf16(np.array(vec, dtype=np.float64)).tolist())
        N, K8 = packed.shape
        out = []
        for n in range(N):
            acc = 0.0
            for g in range(K8 * 8 // 32):
                P = 0
                for c in range(32 * g, 32 * g + 32):
                    code = (int(packed[n, c // 8]) & 0xFFFFFFFF) >> (4 * (c % 8)) & 0xF
                    P += q[c] * (code - 16 if code >= 8 else code)
                acc += float(O.bf16_bits_to_f64(scale[n, g])) * P
            out.append(float(sx) * acc)
        return out
    g = lin(u, ex["gate_packed"], ex["gate_scale"])
    up = lin(u, ex["up_packed"], ex["up_scale"])
    h = [gv / (1.0 + math.exp(-gv)) * uv for gv, uv in zip(g, up)]
    return lin(h, ex["down_packed"], ex["down_scale"])


def test_exact_expert_matches_brute_force_loops():
    # u is not bf16-valued (as after the latent projection): both the input
    # and h are rounded to bf16 before their int8 quantisation
    ex = _random_expert(64, 32)
    u = RNG.normal(size=(3, 64))
    y = O.expert_ffn(u, ex, 8)
    for r in range(3):
        assert np.allclose(y[r], _brute_expert_exact(u[r], ex), rtol=1e-12, atol=1e-12)


def test_expert_closed_form_swiglu():
    # u = 1, every gate/up weight 1 * 2^-5 over 32 inputs -> G = U = 1;
    # down weights 1 * 2^-5 over 32 hidden -> y = SiLU(1) * 1 = 1 / (1 + e^-1).
    D = I = 32
    ones = O.pack_int4(np.ones((32, 32), dtype=np.int64))
    s = np.full((32, 1), 0x3D00, dtype=np.uint16)   # 2^-5
    ex = {"gate_packed": ones, "gate_scale": s, "up_packed": ones, "up_scale": s,
          "down_packed": ones, "down_scale": s}
    y = O.expert_ffn(np.ones((1, D)), ex, 16)
    assert np.allclose(y, 1.0 / (1.0 + math.exp(-1.0)), rtol=1e-15)
    # negative gate: SiLU(-1) * 1 = -1 / (1 + e)
    ex["gate_packed"] = O.pack_int4(-np.ones((32, 32), dtype=np.int64))
    y = O.expert_ffn(np.ones((1, D)), ex, 16)
    assert np.allclose(y, -1.0 / (1.0 + math.e), rtol=1e-15)


def test_rmsnorm_closed_form():
    c, eps = -3.0, 1e-6
    g = O.f32_to_bf16_bits(np.array([1.0, 0.5, 2.0, -1.0], np.float32))
    y = O.rmsnorm(np.full((1, 4), c), g, eps)
    base = c / math.sqrt(c * c + eps)
    assert np.allclose(y[0], [base, 0.5 * base, 2 * base, -base], rtol=1e-15)
    v = np.array([[3.0, -4.0]])   # mean square 12.5
    y = O.rmsnorm(v, np.full(2, ONE, np.uint16), 0.0)
    assert np.allclose(y, v / math.sqrt(12.5), rtol=1e-15)


# ----------------------------------------------------------------------------
# the layer
# ----------------------------------------------------------------------------

def _small_params(E=5, D=64, I=32, k=2, act_bits=16, latent=None, renorm=True):
    experts = [_random_expert(D, I) for _ in range(E)]
    H = latent[0].shape[1] if latent else D
    p = O.LayerParams(k=k, renorm=renorm, act_bits=act_bits,
                      w_router=RNG.normal(size=(E, H)) * 0.2, bias=RNG.normal(size=E) * 0.01,
                      expert=lambda e: experts[e], E=E)
    if latent:
        p.lat_down, p.lat_norm, p.lat_up = latent
    return p


@pytest.mark.parametrize("act_bits", [16, 8])
def test_sorted_dispatch_equals_per_token_definition(act_bits):
    p = _small_params(E=6, k=3, act_bits=act_bits)
    x = O.round_bf16(RNG.normal(size=(17, 64)))
    a = O.moe_forward(x, p)
    b = O.moe_forward_sorted(x, p)
    assert np.allclose(a, b.out, rtol=1e-12, atol=1e-12 * np.abs(a).max())
    # evaluating a subset of tokens gives the same rows
    sub = O.moe_forward(x, p, tokens=[3, 11, 0])
    assert np.allclose(sub, a[[3, 11, 0]], rtol=1e-12, atol=1e-14)


def test_sorted_dispatch_with_single_row_and_idle_experts():
    # 10 rows over 24 experts: most experts hold one row or none, so the
    # sorted path must neither skip a one-row segment nor touch an empty one
    p = _small_params(E=24, k=2)
    x = O.round_bf16(RNG.normal(size=(5, 64)))
    counts = O.dispatch(O.route(x, p.w_router, p.bias, p.k).idx, p.E).counts
    assert (counts == 1).any() and (counts == 0).any()
    a = O.moe_forward(x, p)
    assert np.allclose(O.moe_forward_sorted(x, p).out, a, rtol=1e-12, atol=1e-12 * np.abs(a).max())


def test_single_expert_layer_is_the_textbook_mlp():
    p = _small_params(E=1, k=1)
    x = O.round_bf16(RNG.normal(size=(3, 64)))
    y = O.moe_forward(x, p)
    for t in range(3):
        assert np.allclose(y[t], _brute_expert(x[t], p.expert(0)), rtol=1e-12, atol=1e-12)


def test_layer_brute_force_two_tokens():
    p = _small_params(E=4, k=2, D=32, I=32)
    x = O.round_bf16(RNG.normal(size=(2, 32)))
    y = O.moe_forward(x, p)
    idx, w = _brute_route(x, p.w_router, p.bias, 2, True)
    for t in range(2):
        want = np.zeros(32)
        for j in range(2):
            want += w[t, j] * np.array(_brute_expert(x[t], p.expert(int(idx[t, j]))))
        assert np.allclose(y[t], want, rtol=1e-12, atol=1e-12)


def test_renorm_off_scales_by_raw_affinities():
    p = _small_params(E=4, k=2, renorm=False)
    x = O.round_bf16(RNG.normal(size=(3, 64)))
    y = O.moe_forward(x, p)
    rt = O.route(x, p.w_router, p.bias, 2, False)
    for t in range(3):
        want = sum(rt.s[t, e] * O.expert_ffn(x[t:t + 1], p.expert(int(e)))[0] for e in rt.idx[t])
        assert np.allclose(y[t], want, rtol=1e-12)


def test_latent_identity_projections_reduce_to_rmsnorm_of_moe():
    D = 64
    eye = np.where(np.eye(D) > 0, ONE, 0).astype(np.uint16)
    gain = O.f32_to_bf16_bits(RNG.uniform(0.5, 1.5, size=D).astype(np.float32))
    p = _small_params(latent=(eye, gain, eye))
    x = O.round_bf16(RNG.normal(size=(4, D)))
    y = O.moe_forward(x, p)
    p_plain = O.LayerParams(k=p.k, renorm=p.renorm, act_bits=16, w_router=p.w_router, bias=p.bias,
                            expert=p.expert, E=p.E)
    want = O.rmsnorm(O.moe_forward(x, p_plain), gain, p.eps)
    assert np.allclose(y, want, rtol=1e-12, atol=1e-12)


def test_latent_norm_precedes_up_projection():
    # down = I and up = 2 I (2.0 is exact in bf16): out = 2 RMSNorm(moe(x)).
    # Normalising after the up-projection would give RMSNorm(2 moe(x)) = RMSNorm(moe(x)).
    D = 64
    eye = np.where(np.eye(D) > 0, ONE, 0).astype(np.uint16)
    two = np.where(np.eye(D) > 0, 0x4000, 0).astype(np.uint16)
    gain = np.full(D, ONE, np.uint16)
    p = _small_params(latent=(eye, gain, two))
    x = O.round_bf16(RNG.normal(size=(3, D)))
    y = O.moe_forward(x, p)
    p_plain = O.LayerParams(k=p.k, renorm=p.renorm, act_bits=16, w_router=p.w_router, bias=p.bias,
                            expert=p.expert, E=p.E)
    m = O.moe_forward(x, p_plain)
    want = 2.0 * m / np.sqrt(np.mean(m * m, axis=1, keepdims=True) + p.eps)
    assert np.allclose(y, want, rtol=1e-12, atol=1e-12)


def test_latent_projection_orientation():
    # [out, in] layout: lat_down [L, H] maps H -> L; lat_up [H, L] maps L -> H.
    H, L = 8, 32
    down = np.zeros((L, H), np.uint16)
    down[np.arange(L), np.arange(L) % H] = ONE      # latent c copies x[c mod H]
    p = _small_params(D=L, latent=(down, None, np.zeros((H, L), np.uint16)))
    x = O.round_bf16(RNG.normal(size=(2, H)))
    u = O.expert_input(x, p)
    assert np.array_equal(u, x[:, np.arange(L) % H])


# ----------------------------------------------------------------------------
# int4 weight quantiser (ExactLinear.from_weight with four bits, group 32)
# ----------------------------------------------------------------------------

def _bf16_exact(v):
    """The float32 values of v, asserting each is exactly a bf16."""
    v = np.asarray(v, dtype=np.float32)
    assert np.array_equal(O.round_bf16(v).astype(np.float32), v)
    return v


def test_weight_quantiser_recovers_exact_codes():
    # scales with at most 5 significant bits times codes of at most 3 bits are
    # exact bf16 values; a group whose largest |code| is 7 recovers (q, s)
    N, K = 6, 128
    q = RNG.integers(-7, 8, size=(N, K))
    q[:, ::32] = np.where(RNG.random((N, K // 32)) < 0.5, 7, -7)
    mant = RNG.integers(16, 32, size=(N, K // 32))
    expo = RNG.integers(-14, -3, size=(N, K // 32))
    s = np.ldexp(mant.astype(np.float64), expo)
    w = _bf16_exact(q * np.repeat(s, 32, axis=1))
    packed, s_bits = O.quantize_weight_int4(w)
    assert np.array_equal(O.unpack_int4(packed), q)
    assert np.array_equal(O.bf16_bits_to_f64(s_bits), s)


def test_weight_quantiser_error_bound_and_range():
    w = O.round_bf16(RNG.normal(size=(16, 256)) * RNG.uniform(1e-3, 10, size=(16, 1))).astype(np.float32)
    packed, s_bits = O.quantize_weight_int4(w)
    q = O.unpack_int4(packed)
    s = np.repeat(O.bf16_bits_to_f64(s_bits), 32, axis=1)
    assert q.min() >= -8 and q.max() <= 7
    # every code is within half a step of w / s (s is the stored bf16 scale)
    assert np.all(np.abs(w / s - q) <= 0.5 + 2.0 ** -20)  # fp32 division, ulp(8) = 2^-20
    # the scale is a/7 rounded to bf16: within 2^-8 relative of the group's max/7
    amax = np.abs(w).reshape(16, 8, 32).max(axis=-1)
    rel = np.abs(O.bf16_bits_to_f64(s_bits) * 7 / amax - 1)
    assert rel.max() <= 2.0 ** -8
    # the largest magnitude of each group maps to +-7
    assert np.all(np.abs(q).reshape(16, 8, 32).max(axis=-1) == 7)


def test_weight_quantiser_zero_group_and_half_ties():
    w = np.zeros((2, 64), dtype=np.float32)
    # group 1 of row 0: max 7 (s = 1), values on half steps round to even codes
    w[0, 32:40] = [7.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, -3.5]
    packed, s_bits = O.quantize_weight_int4(w)
    q = O.unpack_int4(packed)
    assert s_bits.tolist() == [[0, 0x3F80], [0, 0]]
    assert q[0, 32:40].tolist() == [7, 0, 2, 2, 0, -2, -2, -4]
    assert not q[1].any() and not q[0, :32].any()


# ----------------------------------------------------------------------------
# int8 weight quantiser (ExactLinear.from_weight with eight bits, group 32)
# ----------------------------------------------------------------------------

def test_weight_quantiser_int8_recovers_exact_codes():
    # a group whose largest |code| is 127 and whose scale has at most one
    # significant bit: 127 * 2^e / 127 is the scale itself, and code * 2^e is
    # an exact bf16 for |code| <= 127 (7 significant bits), so (q, s) come back
    N, K = 6, 128
    q = RNG.integers(-127, 128, size=(N, K))
    q[:, ::32] = np.where(RNG.random((N, K // 32)) < 0.5, 127, -127)
    s = np.ldexp(1.0, RNG.integers(-20, 4, size=(N, K // 32)))
    w = _bf16_exact(q * np.repeat(s, 32, axis=1))
    q8, s_bits = O.quantize_weight_int8(w)
    assert q8.dtype == np.int8
    assert np.array_equal(q8.astype(np.int64), q)
    assert np.array_equal(O.bf16_bits_to_f64(s_bits), s)


def test_weight_quantiser_int8_error_bound_and_range():
    w = O.round_bf16(RNG.normal(size=(16, 256)) * RNG.uniform(1e-3, 10, size=(16, 1))).astype(np.float32)
    q, s_bits = O.quantize_weight_int8(w)
    q = q.astype(np.int64)
    s = np.repeat(O.bf16_bits_to_f64(s_bits), 32, axis=1)
    assert q.min() >= -127 and q.max() <= 127
    # every code is within half a step of w / s (fp32 division, ulp(128) = 2^-16)
    assert np.all(np.abs(w / s - q) <= 0.5 + 2.0 ** -16)
    # the scale is a/127 rounded to bf16: within 2^-8 relative of the group's max/127
    amax = np.abs(w).reshape(16, 8, 32).max(axis=-1)
    rel = np.abs(O.bf16_bits_to_f64(s_bits) * 127 / amax - 1)
    assert rel.max() <= 2.0 ** -8
    # the largest magnitude of each group maps to +-127 (|w| / s <= 127 (1 + 2^-9))
    assert np.all(np.abs(q).reshape(16, 8, 32).max(axis=-1) == 127)


def test_weight_quantiser_int8_zero_group_and_half_ties():
    w = np.zeros((2, 64), dtype=np.float32)
    # group 1 of row 0: max 127 (s = 1), values on half steps round to even codes
    w[0, 32:41] = [127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, -126.5, 125.5]
    q, s_bits = O.quantize_weight_int8(w)
    assert s_bits.tolist() == [[0, 0x3F80], [0, 0]]
    assert q[0, 32:41].tolist() == [127, 0, 2, 2, 0, -2, -2, -126, 126]
    assert not q[1].any() and not q[0, :32].any()


def test_weight_quantisers_agree_on_a_shared_grid():
    # a group of codes in [-7, 7] with max 7 and scale s: the int4 quantiser
    # recovers the codes with scale s, the int8 one the same values with
    # scale 7 s / 127 rounded to bf16 (brute force: each code from one float32
    # division, rounded half to even)
    q = np.array([[7, -7, 3, 0, -1, 5, 2, -4] * 4], dtype=np.int64)
    s = 0.0625
    w = _bf16_exact(q * s)
    q4, _ = O.quantize_weight_int4(w)
    assert np.array_equal(O.unpack_int4(q4), q)
    q8, s8 = O.quantize_weight_int8(w)
    s8f = np.float32(O.bf16_bits_to_f64(s8)[0, 0])
    assert s8f == np.float32(O.round_bf16(np.float32(7 * s) / np.float32(127)))
    want = [int(np.rint(np.float32(v) / s8f)) for v in w[0]]
    assert q8[0].tolist() == want


# ----------------------------------------------------------------------------
# shared expert
# ----------------------------------------------------------------------------

def test_shared_expert_closed_form_special_case():
    """x = e_0, up(x) = 1 for every feature, gate(x) = v, down a permutation:
    out = P bf16(SiLU(v)), with SiLU written out from the exponential."""
    H = I = 8
    v = np.array([-3.0, -1.0, -0.5, 0.0, 0.25, 1.0, 2.0, 5.0])
    gate = np.zeros((I, H)); gate[:, 0] = v
    up = np.zeros((I, H)); up[:, 0] = 1.0
    perm = [3, 0, 7, 1, 6, 2, 5, 4]
    down = np.zeros((H, I))
    for r, c in enumerate(perm):
        down[r, c] = 1.0
    x = np.zeros((1, H)); x[0, 0] = 1.0
    bits = lambda a: O.f32_to_bf16_bits(a.astype(np.float32))
    out = O.shared_expert(x, bits(gate), bits(up), bits(down))
    silu = np.array([t / (1.0 + math.exp(-t)) for t in v])
    want = O.round_bf16(silu)[perm]
    assert np.array_equal(out[0], want)
    # gate and up swapped: SiLU(1) * v instead (a transposed role fails here)
    out2 = O.shared_expert(x, bits(up), bits(gate), bits(down))
    assert np.array_equal(out2[0], O.round_bf16(v * (1.0 / (1.0 + math.exp(-1.0))))[perm])


def test_shared_expert_hidden_order_and_down_scaling():
    rng = np.random.default_rng(5)
    H, I = 64, 48
    bits = lambda a: O.f32_to_bf16_bits(a.astype(np.float32))
    gate, up, down = (bits(rng.normal(size=s) * 0.1) for s in [(I, H), (I, H), (H, I)])
    x = rng.normal(size=(5, H))
    ref = O.shared_expert(x, gate, up, down)
    # reordering the hidden features consistently changes nothing
    p = rng.permutation(I)
    assert np.allclose(O.shared_expert(x, gate[p], up[p], down[:, p]), ref, rtol=1e-12, atol=1e-14)
    # doubling the down weights (exact in bf16) doubles the output exactly
    d2 = O.f32_to_bf16_bits(2 * O.bf16_bits_to_f64(down).astype(np.float32))
    assert np.array_equal(O.shared_expert(x, gate, up, d2), 2 * ref)


def test_layer_adds_the_shared_expert_on_the_full_width_input():
    # Latent layer (H = 8 -> L = 32) with a shared expert on the full width H.
    H, L, Is = 8, 32, 16
    rng = np.random.default_rng(11)
    bits = lambda a: O.f32_to_bf16_bits(a.astype(np.float32))
    down = np.zeros((L, H), np.uint16)
    down[np.arange(L), np.arange(L) % H] = ONE
    up = bits(rng.normal(size=(H, L)) * 0.1)
    p = _small_params(D=L, latent=(down, np.full(L, ONE, np.uint16), up))
    p.w_router = rng.normal(size=(p.E, H)) * 0.2
    sg, su, sd = (bits(rng.normal(size=s) * 0.2) for s in [(Is, H), (Is, H), (H, Is)])
    x = O.round_bf16(rng.normal(size=(4, H)))
    routed = O.moe_forward(x, p)
    shared = O.shared_expert(x, sg, su, sd)
    assert np.abs(routed).max() > 0 and np.abs(shared).max() > 0
    p.shared_gate, p.shared_up, p.shared_down = sg, su, sd
    # a shared expert with zero down weights changes nothing
    p.shared_down = np.zeros_like(sd)
    assert np.array_equal(O.moe_forward(x, p), routed)
    # routed experts with zero codes leave exactly the shared expert
    p.shared_down = sd
    zero = {key: (np.zeros_like(v) if key.endswith("_packed") else v) for key, v in p.expert(0).items()}
    p.expert = lambda e: zero
    assert np.array_equal(O.moe_forward(x, p), shared)
    assert np.array_equal(O.moe_forward_sorted(x, p).out, shared)
