"""Pins for the CPU oracle: checks against facts that do not come from the
oracle itself (page figures, hand-derived examples, exact rational arithmetic,
closed forms, textbook special cases and invariants). CPU only."""

import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
import wq_inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _facts():
    out = {}
    with open(os.path.join(GOLDEN, "page_facts.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *v = line.split()
            out[k] = v
    return out


# ---------------------------------------------------------------- layout pins

def test_golden_row_lengths_from_model_card():
    f = _facts()
    assert O.packed_words_per_row(5120, 6) == int(f["dense_words_b6_k5120"][0])
    # the word-aligned formula the page quotes gives a different length
    assert 5120 // (32 // 6) == int(f["word_aligned_words_b6_k5120"][0])
    assert [int(b) for b in f["supported_bits"]] == list(range(2, 9))


def test_golden_hand_worked_b5_example():
    rows = {}
    with open(os.path.join(GOLDEN, "pack_b5_worked.txt")) as fh:
        for line in fh:
            if line.strip() and not line.startswith("#"):
                k, *v = line.split()
                rows[k] = v
    bits = int(rows["bits"][0])
    codes = np.array([[int(c) for c in rows["codes"]]])
    words = [int(w, 16) for w in rows["words"]]
    assert O.pack(codes, bits)[0].tolist() == words
    assert O.unpack(np.array([words], dtype=np.uint32), codes.shape[1], bits)[0].tolist() \
        == codes[0].tolist()


@pytest.mark.parametrize("bits", range(2, 9))
@pytest.mark.parametrize("K", [128, 5120])
def test_round_trip_random_and_extremes(bits, K):
    g = np.random.default_rng(bits * 1000 + K)
    N = 3
    codes = g.integers(0, 1 << bits, size=(N, K))
    codes[1, :] = 0
    codes[2, :] = (1 << bits) - 1
    packed = O.pack(codes, bits)
    assert packed.shape == (N, (K * bits + 31) // 32)
    assert np.array_equal(O.unpack(packed, K, bits), codes)
    # extremes: all-zero row packs to zero words, all-ones row to a run of ones
    assert not packed[1].any()
    ones = K * bits
    full, rem = divmod(ones, 32)
    assert np.all(packed[2, :full] == 0xFFFFFFFF)
    if rem:
        assert packed[2, full] == (1 << rem) - 1


@pytest.mark.parametrize("bits", range(2, 9))
def test_pack_equals_big_integer_construction(bits):
    """Independent statement of the layout: the row is the little-endian
    32-bit word sequence of the integer sum_k q_k * 2^(k*bits)."""
    g = np.random.default_rng(77 + bits)
    K = 96
    codes = g.integers(0, 1 << bits, size=(2, K))
    packed = O.pack(codes, bits)
    for r in range(2):
        U = 0
        for k in range(K):
            U += int(codes[r, k]) << (k * bits)
        nwords = (K * bits + 31) // 32
        expect = [(U >> (32 * i)) & 0xFFFFFFFF for i in range(nwords)]
        assert packed[r].tolist() == expect


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_dense_layout_equals_word_aligned_formula_when_bits_divides_32(bits):
    """Model card "Findings": the word-aligned kernel reads code `col` from
    word col // (32 // bits) at shift (col % (32 // bits)) * bits. When bits
    divides 32 the dense layout must be exactly that."""
    g = np.random.default_rng(5 + bits)
    K = 256
    codes = g.integers(0, 1 << bits, size=(4, K))
    pf = 32 // bits
    aligned = np.zeros((4, K // pf), dtype=np.uint64)
    for col in range(K):
        aligned[:, col // pf] |= codes[:, col].astype(np.uint64) << np.uint64((col % pf) * bits)
    assert np.array_equal(O.pack(codes, bits), aligned.astype(np.uint32))


def test_out_of_range_codes_counted_and_masked():
    codes = np.array([[0, 31, 32, 255, 7]])
    assert O.count_out_of_range(codes, 5) == 2
    assert O.unpack(O.pack(codes, 5), 5, 5)[0].tolist() == [0, 31, 0, 31, 7]


# ---------------------------------------------------------------- GEMM pins

def _frac_bf16(bits16):
    return Fraction(float(O.bf16_bits_to_f32(np.array([bits16], dtype=np.uint16))[0]))


@pytest.mark.parametrize("bits", [2, 5, 6, 7, 8])
def test_wna16_brute_force_exact_rationals(bits):
    M, K, N = 3, 128, 4
    x = I.make_x(M, K, 11 + bits)
    q = I.make_codes(N, K, bits, 12 + bits)
    s = I.make_scales(N, K // 128, 13 + bits)
    y = O.wna16_ref(x, q, s, bits)
    z = 1 << (bits - 1)
    for m in range(M):
        for n in range(N):
            exact = Fraction(0)
            mag = Fraction(0)
            for k in range(K):
                term = _frac_bf16(x[m, k]) * _frac_bf16(s[n, k // 128]) * (int(q[n, k]) - z)
                exact += term
                mag += abs(term)
            assert abs(Fraction(float(y[m, n])) - exact) <= mag * Fraction(1, 2**45)


@pytest.mark.parametrize("bits", [3, 5, 6, 7, 8])
@pytest.mark.parametrize("c_kind", ["zero_point", "min", "max"])
def test_wna16_closed_form_constant_codes(bits, c_kind):
    """All codes equal c: y[m, n] = sum_g s[n, g] * (c - z) * sum_{k in g} x[m, k];
    c = z gives y == 0 exactly."""
    M, K, N = 2, 384, 5
    z = 1 << (bits - 1)
    c = {"zero_point": z, "min": 0, "max": (1 << bits) - 1}[c_kind]
    x = I.make_x(M, K, 21)
    s = I.make_scales(N, K // 128, 22)
    q = np.full((N, K), c, dtype=np.int64)
    y = O.wna16_ref(x, q, s, bits)
    xf = O.bf16_bits_to_f64(x).reshape(M, K // 128, 128).sum(axis=2)   # [M, G]
    sf = O.bf16_bits_to_f64(s)                                          # [N, G]
    expect = (c - z) * xf @ sf.T
    if c == z:
        assert np.all(y == 0.0)
    else:
        np.testing.assert_allclose(y, expect, rtol=1e-12, atol=1e-12)


def test_b8_unit_scales_is_plain_int8_matmul():
    M, K, N = 3, 256, 7
    x = I.make_x(M, K, 31)
    q = I.make_codes(N, K, 8, 32)
    one = np.full((N, K // 128), 0x3F80, dtype=np.uint16)  # bf16 1.0
    y = O.wna16_ref(x, q, one, 8)
    w_int8 = q.astype(np.int64) - 128          # int8 weights in [-128, 127]
    ref = O.bf16_bits_to_f64(x) @ w_int8.T.astype(np.float64)
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-13)


def test_scale_sign_symmetry_and_all_negative():
    M, K, N, bits = 2, 512, 6, 6
    x = I.make_x(M, K, 41)
    q = I.make_codes(N, K, bits, 42)
    s = I.make_scales(N, K // 128, 43)
    y = O.wna16_ref(x, q, s, bits)
    flip = s.copy()
    flip[3, 2] ^= np.uint16(0x8000)        # flip the sign of one group scale
    zero = s.copy()
    zero[3, 2] = 0
    y_flip = O.wna16_ref(x, q, flip, bits)
    y_zero = O.wna16_ref(x, q, zero, bits)
    # y(s) = y(zero) + c, y(flip) = y(zero) - c
    np.testing.assert_allclose(y + y_flip, 2 * y_zero, rtol=1e-12, atol=1e-12)
    assert not np.allclose(y[:, 3], y_flip[:, 3])
    others = [n for n in range(N) if n != 3]
    assert np.array_equal(y[:, others], y_flip[:, others])
    neg = s ^ np.uint16(0x8000)
    assert np.array_equal(O.wna16_ref(x, q, neg, bits), -y)


# ---------------------------------------------------------------- act-quant pins

def _bf16(vals):
    return I._to_bf16_bits(np.array(vals, dtype=np.float32))


def test_act_quant_half_way_cases_round_to_even():
    # amax = 127 makes sx exactly 1.0, so x/sx = x and the halves are exact
    row = [127.0, 2.5, 3.5, -2.5, 0.5, 1.5, -0.5, 126.5, -126.5, 0.0]
    xq, sx = O.act_quant_ref(_bf16([row]))
    assert sx[0] == np.float32(1.0)
    assert xq[0].tolist() == [127, 2, 4, -2, 0, 2, 0, 126, -126, 0]


def test_act_quant_invariants():
    x = I.make_x_outliers(16, 1024, 51)
    x[3] = 0                        # an all-zero row
    xq, sx = O.act_quant_ref(x)
    xf = O.bf16_bits_to_f32(x)
    assert xq.dtype == np.int8
    assert np.all(np.abs(xq.astype(np.int32)) <= 127)
    assert sx[3] == 0 and not xq[3].any()
    for m in range(16):
        if m == 3:
            continue
        assert np.max(np.abs(xq[m].astype(np.int32))) == 127
        assert sx[m] == np.float32(np.max(np.abs(xf[m])) / np.float32(127))
        nz = xq[m] != 0
        assert np.all(np.sign(xq[m][nz]) == np.sign(xf[m][nz]))
        # reconstruction error at most half a step
        err = np.abs(xq[m].astype(np.float64) * sx[m] - xf[m].astype(np.float64))
        assert np.all(err <= 0.5 * np.float64(sx[m]) * (1 + 1e-6))


def _nearest_f32(q: Fraction) -> np.float32:
    """The float32 nearest to the rational q, ties to the even significand:
    IEEE round-to-nearest of an exact quotient, decided by comparing exact
    distances of the float32 values around float(q)."""
    f = np.float32(float(q))
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    return min(cands, key=lambda c: (abs(Fraction(float(c)) - q),
                                     int(np.array([c], dtype=np.float32).view(np.uint32)[0]) & 1))


def _round_half_even(v: Fraction) -> int:
    lo = v.numerator // v.denominator
    d = v - lo
    if d != Fraction(1, 2):
        return lo + (d > Fraction(1, 2))
    return lo + (lo % 2)


def test_act_quant_is_ieee_division_then_round_half_even():
    """In exact rational arithmetic: sx is amax / 127 rounded once to
    float32; xq is x / sx rounded once to float32, then to the nearest
    integer, ties to even, clamped to +-127 ("int8 activations (W4A8)"
    discussion, "Under the hood": per-token dynamic int8; the division and
    rounding details are this oracle's stated reading). Row m holds amax and
    +-amax/2 for every bf16 amax in [64, 128): x / sx then lies within
    rounding of 63.5, where a reciprocal multiply or a second rounding step
    decides differently for some rows."""
    rows = []
    extra = O.bf16_bits_to_f32(I.make_x(128, 4, 57))          # |x| < 64
    for m in range(128):
        a = float(O.bf16_bits_to_f32(np.array([0x4280 | m], dtype=np.uint16))[0])
        row = [a, a / 2, -a / 2, a / 4] + extra[m].tolist()
        rows.append([-v for v in row] if m % 2 else row)
    x = _bf16(rows)
    xq, sx = O.act_quant_ref(x)
    xf = O.bf16_bits_to_f32(x)
    for m in range(len(rows)):
        amax = max(abs(Fraction(float(v))) for v in xf[m])
        s = _nearest_f32(amax / 127)
        assert sx[m] == s
        for k in range(xf.shape[1]):
            ratio = _nearest_f32(Fraction(float(xf[m, k])) / Fraction(float(s)))
            want = max(-127, min(127, _round_half_even(Fraction(float(ratio)))))
            assert int(xq[m, k]) == want, (m, k)


def test_w4a8_group_acc_sums_to_integer_matmul_and_unit_scales():
    M, K, N = 4, 384, 5
    x = I.make_x_outliers(M, K, 61)
    q = I.make_codes(N, K, 4, 62)
    xq, sx = O.act_quant_ref(x)
    acc = O.w4a8_group_acc(xq, q)
    full = xq.astype(np.int64) @ (q.astype(np.int64) - 8).T
    assert np.array_equal(acc.sum(axis=2), full)
    # unit group scales and unit token scales: y is that integer matmul
    one = np.full((N, K // 128), 0x3F80, dtype=np.uint16)
    y = O.w4a8_ref_from_quant(xq, np.ones(M, np.float32), q, one)
    assert np.array_equal(y, full.astype(np.float64))
    # widening is lossless: q - 8 covers [-8, 7] exactly
    assert (q.astype(np.int64) - 8).min() >= -8 and (q.astype(np.int64) - 8).max() <= 7


def test_w4a8_brute_force_exact_rationals():
    """Tiny W4A8 layer summed term by term in exact rationals: the integer
    group sums over k // 128, each scaled by the token's float32 scale and the
    group's bf16 scale ("int8 activations (W4A8)" discussion, "Under the hood":
    integer accumulation of widened int4 weights, then the scales)."""
    M, K, N = 2, 384, 3
    x = I.make_x_outliers(M, K, 65)
    q = I.make_codes(N, K, 4, 66)
    s = I.make_scales(N, K // 128, 67)
    xq, sx = O.act_quant_ref(x)
    y = O.w4a8_ref_from_quant(xq, sx, q, s)
    for m in range(M):
        for n in range(N):
            exact = Fraction(0)
            mag = Fraction(0)
            for g in range(K // 128):
                acc = sum(int(xq[m, k]) * (int(q[n, k]) - 8) for k in range(128 * g, 128 * g + 128))
                term = Fraction(float(sx[m])) * _frac_bf16(s[n, g]) * acc
                exact += term
                mag += abs(term)
            assert abs(Fraction(float(y[m, n])) - exact) <= mag * Fraction(1, 2**45)


def test_w4a8_close_to_wna16_b4():
    """Reported, not a parity gate: the activation-quantization loss is small
    relative to the output with 1% outlier channels."""
    M, K, N = 8, 1024, 16
    x = I.make_x_outliers(M, K, 71)
    q = I.make_codes(N, K, 4, 72)
    s = I.make_scales(N, K // 128, 73)
    y8, _, _ = O.w4a8_ref(x, q, s)
    y16 = O.wna16_ref(x, q, s, 4)
    rel = np.linalg.norm(y8 - y16) / np.linalg.norm(y16)
    assert rel < 0.05


# ---------------------------------------------------------------- gather pins

def test_bf16_rne_hand_cases():
    one = 1.0
    cases = {
        one: 0x3F80,
        one + 2.0**-8: 0x3F80,              # tie between 1 and 1+2^-7 -> even (1)
        one + 3 * 2.0**-8: 0x3F82,          # tie between 1+2^-7 and 1+2^-6 -> even
        one + 2.0**-8 + 2.0**-20: 0x3F81,   # above the tie -> up
        -2.0: 0xC000,
        -0.0: 0x8000,
        float("inf"): 0x7F80,
    }
    vals = np.array(list(cases.keys()), dtype=np.float32)
    assert O.f32_to_bf16_bits_rne(vals).tolist() == list(cases.values())


@pytest.mark.parametrize("bits", [3, 5, 6, 8])
def test_gather_is_rounded_dequant_with_ids_out_of_range(bits):
    V, D, T = 9, 256, 7
    q = I.make_codes(V, D, bits, 81)
    s = I.make_scales(V, D // 128, 82)
    ids = np.array([0, 8, 3, -1, 9, 3, 100], dtype=np.int32)
    out, bad = O.qembed_ref(ids, q, s, bits)
    assert bad == 3
    w = O.dequant(q, s, bits)
    for t, i in enumerate(ids):
        got = O.bf16_bits_to_f64(out[t])
        if i < 0 or i >= V:
            assert np.all(out[t] == 0)
            continue
        # bf16 RNE (8 significant bits): relative error at most 2^-8
        assert np.all(np.abs(got - w[i]) <= np.abs(w[i]) * 2.0**-8)


def _bf16_bits_of_rational(v: Fraction) -> int:
    """bf16 bits of the rational v in the normal range, rounded to nearest
    with ties to the even significand, from the format's definition (sign,
    8-bit exponent with bias 127, 8 significant bits)."""
    if v == 0:
        return 0
    sign = 0x8000 if v < 0 else 0
    a, e = abs(v), 0
    while a >= 2:
        a, e = a / 2, e + 1
    while a < 1:
        a, e = a * 2, e - 1
    m = _round_half_even(a * 128)          # 128..256
    if m == 256:
        m, e = 128, e + 1
    return sign | ((e + 127) << 7) | (m - 128)


def test_gather_exact_products_round_half_even():
    """Every gathered element equals the exact product s * (q - z) rounded to
    bf16 once, ties to even, computed in rationals. Scales 1 + k/128 (and
    their negatives) against every 8-bit code give products with 9 to 16
    significant bits, many exactly halfway between two bf16 values, with both
    neighbours' parities."""
    bits, z = 8, 128
    scales_bits = [0x3F80 + k for k in range(1, 16)] + [0xBF80 + k for k in range(1, 16)]
    rows, srows = [], []
    for sb in scales_bits:
        rows += [list(range(0, 128)), list(range(128, 256))]
        srows += [[sb], [sb]]
    q = np.array(rows, dtype=np.int64)                     # V = 60 rows, D = 128
    s = np.array(srows, dtype=np.uint16)
    out, bad = O.qembed_ref(np.arange(len(rows)), q, s, bits)
    assert bad == 0
    ties = {0: 0, 1: 0}
    for r in range(len(rows)):
        sv = _frac_bf16(s[r, 0])
        for d in range(128):
            v = sv * (int(q[r, d]) - z)
            if v != 0:
                a = abs(v)
                while a >= 2:
                    a /= 2
                while a < 1:
                    a *= 2
                t = a * 128
                if t - int(t) == Fraction(1, 2):
                    ties[int(t) % 2] += 1
            want = _bf16_bits_of_rational(v) if v != 0 else (0x8000 if sv < 0 else 0)
            assert int(out[r, d]) == want, (r, d)
    assert ties[0] > 0 and ties[1] > 0, ties


def test_gather_negative_zero_and_unit_scale_b8():
    q = np.array([[128] * 128 + [0] * 128], dtype=np.int64)   # V=1, D=256
    s = np.array([[0xBF80, 0x3F80]], dtype=np.uint16)         # -1.0, +1.0
    out, bad = O.qembed_ref(np.array([0]), q, s, 8)
    assert bad == 0
    assert np.all(out[0, :128] == 0x8000)                       # -1 * 0 = -0.0
    assert np.all(O.bf16_bits_to_f32(out[0, 128:]) == -128.0)


# ---------------------------------------------------------------- byte counts

def test_page_byte_counts_pin_group_128_scales():
    f = _facts()
    V, D = int(f["vocab"][0]), int(f["hidden"][0])
    gib = 2.0**30
    bf16 = O.bf16_matrix_bytes(V, D) / gib
    assert round(bf16, 2) == float(f["bf16_vocab_layer_gib"][0])
    assert round(2 * bf16, 2) == float(f["bf16_both_vocab_layers_gib"][0])
    q8 = O.quantized_matrix_bytes(V, D, 8, group=128) / gib
    saving = 2 * bf16 - 2 * q8
    assert round(saving, 2) == float(f["int8_vocab_saving_gib"][0])
    # per-row scales would free 2.37 GiB instead, so the printed figure pins
    # group-128 scale granularity
    per_row = 2 * bf16 - 2 * O.quantized_matrix_bytes(V, D, 8, group=D) / gib
    assert round(per_row, 2) != float(f["int8_vocab_saving_gib"][0])


def test_stack_allocation():
    bits = [I.stack_layer_bits(l) for l in range(64)]
    assert bits[:10] == [7] * 10 and bits[54:] == [7] * 10
    assert bits[10:54] == [5, 6] * 22


# ---------------------------------------------------------------- asymmetric groups

def _zeros(N, G, bits, seed):
    return np.random.default_rng(seed).integers(0, 1 << bits, size=(N, G)).astype(np.uint8)


@pytest.mark.parametrize("bits", [4, 5, 6, 7, 8])
def test_zp_brute_force_exact_rationals(bits):
    """w = s (q - zp[n, g]) against exact rational arithmetic on a tiny
    shape with a different zero point in every (row, group)."""
    M, K, N = 2, 256, 3
    x = I.make_x(M, K, 41 + bits)
    q = I.make_codes(N, K, bits, 42 + bits)
    s = I.make_scales(N, K // 128, 43 + bits)
    zp = _zeros(N, K // 128, bits, 44 + bits)
    y = O.wna16_zp_ref(x, q, s, zp, bits)
    for m in range(M):
        for n in range(N):
            exact = Fraction(0)
            mag = Fraction(0)
            for k in range(K):
                term = _frac_bf16(x[m, k]) * _frac_bf16(s[n, k // 128]) * (int(q[n, k]) - int(zp[n, k // 128]))
                exact += term
                mag += abs(term)
            assert abs(Fraction(float(y[m, n])) - exact) <= mag * Fraction(1, 2**45)


@pytest.mark.parametrize("bits", [5, 6, 8])
def test_zp_closed_form_constant_codes(bits):
    """All codes c: y[m, n] = sum_g s[n, g] (c - zp[n, g]) sum_{k in g} x[m, k];
    codes equal to each group's zero point give y == 0 exactly."""
    M, K, N = 2, 384, 5
    G = K // 128
    x = I.make_x(M, K, 51)
    s = I.make_scales(N, G, 52)
    zp = _zeros(N, G, bits, 53)
    c = (1 << bits) - 1
    q = np.full((N, K), c, dtype=np.int64)
    y = O.wna16_zp_ref(x, q, s, zp, bits)
    xg = O.bf16_bits_to_f64(x).reshape(M, G, 128).sum(axis=2)              # [M, G]
    coef = O.bf16_bits_to_f64(s) * (c - zp.astype(np.float64))             # [N, G]
    np.testing.assert_allclose(y, xg @ coef.T, rtol=1e-12, atol=1e-12)
    qz = np.repeat(zp.astype(np.int64), 128, axis=1)
    assert np.all(O.wna16_zp_ref(x, qz, s, zp, bits) == 0.0)


@pytest.mark.parametrize("bits", [5, 6, 7, 8])
def test_zp_at_half_range_is_the_symmetric_layer(bits):
    M, K, N = 3, 256, 6
    x = I.make_x(M, K, 61)
    q = I.make_codes(N, K, bits, 62)
    s = I.make_scales(N, K // 128, 63)
    zp = np.full((N, K // 128), 1 << (bits - 1), dtype=np.uint8)
    assert np.array_equal(O.wna16_zp_ref(x, q, s, zp, bits), O.wna16_ref(x, q, s, bits))


def test_zp_shift_invariance():
    """Shifting the codes and the zero point of a group by the same amount
    leaves the dequantized weights, hence y, unchanged."""
    bits, M, K, N = 6, 2, 256, 4
    x = I.make_x(M, K, 71)
    s = I.make_scales(N, K // 128, 72)
    rng = np.random.default_rng(73)
    q = rng.integers(0, 40, size=(N, K))
    zp = rng.integers(0, 40, size=(N, K // 128)).astype(np.uint8)
    d = np.array([[3, 17], [0, 23], [11, 5], [20, 1]])                    # per (row, group)
    q2 = q + np.repeat(d, 128, axis=1)
    zp2 = (zp.astype(np.int64) + d).astype(np.uint8)
    assert np.array_equal(O.wna16_zp_ref(x, q, s, zp, bits), O.wna16_zp_ref(x, q2, s, zp2, bits))


def test_zp_uses_the_low_bits_of_each_byte():
    bits, M, K, N = 5, 2, 256, 3
    x = I.make_x(M, K, 81)
    q = I.make_codes(N, K, bits, 82)
    s = I.make_scales(N, K // 128, 83)
    zp = _zeros(N, K // 128, bits, 84)
    high = (zp | np.uint8(0xE0)).astype(np.uint8)                          # bits 5..7 set
    assert np.array_equal(O.wna16_zp_ref(x, q, s, high, bits), O.wna16_zp_ref(x, q, s, zp, bits))
    assert O.zero_points_used(np.array([0xFF], dtype=np.uint8), 5)[0] == 31


# ---------------------------------------------------------------- mixture of experts

def _moe_case(E, N, K, bits, counts, seed):
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    M = int(off[-1])
    x = I.make_x(M, K, seed)
    q = np.stack([I.make_codes(N, K, bits, seed + 1 + e) for e in range(E)])
    s = np.stack([I.make_scales(N, K // 128, seed + 50 + e) for e in range(E)])
    return off, x, q, s


def test_moe_brute_force_exact_rationals():
    """Three experts, ragged token counts including an empty expert: every
    output against exact rational arithmetic with that token's expert."""
    bits, N, K = 6, 3, 128
    off, x, q, s = _moe_case(4, N, K, bits, [2, 0, 1, 2], 400)
    y = O.moe_ref(x, off, q, s, bits)
    z = 1 << (bits - 1)
    for m in range(x.shape[0]):
        e = int(np.searchsorted(off, m, side="right")) - 1
        for n in range(N):
            exact = sum(_frac_bf16(x[m, k]) * _frac_bf16(s[e, n, k // 128]) * (int(q[e, n, k]) - z)
                        for k in range(K))
            mag = sum(abs(_frac_bf16(x[m, k]) * _frac_bf16(s[e, n, k // 128]) * (int(q[e, n, k]) - z))
                      for k in range(K))
            assert abs(Fraction(float(y[m, n])) - exact) <= mag * Fraction(1, 2**45)


def test_moe_with_one_expert_or_equal_experts_is_the_dense_layer():
    bits, N, K = 5, 7, 256
    off, x, q, s = _moe_case(1, N, K, bits, [9], 410)
    assert np.array_equal(O.moe_ref(x, off, q, s, bits), O.wna16_ref(x, q[0], s[0], bits))
    off, x, q, s = _moe_case(3, N, K, bits, [4, 1, 3], 420)
    qe = np.repeat(q[:1], 3, axis=0)
    se = np.repeat(s[:1], 3, axis=0)
    assert np.array_equal(O.moe_ref(x, off, qe, se, bits), O.wna16_ref(x, q[0], s[0], bits))


def test_moe_rows_follow_their_expert():
    """Reordering the experts together with their token blocks permutes the
    output rows the same way."""
    bits, N, K = 7, 5, 256
    counts = [3, 1, 4]
    off, x, q, s = _moe_case(3, N, K, bits, counts, 430)
    y = O.moe_ref(x, off, q, s, bits)
    perm = [2, 0, 1]
    blocks = [np.arange(off[e], off[e + 1]) for e in range(3)]
    rows = np.concatenate([blocks[e] for e in perm])
    off2 = np.concatenate([[0], np.cumsum([counts[e] for e in perm])])
    y2 = O.moe_ref(x[rows], off2, q[perm], s[perm], bits)
    assert np.array_equal(y2, y[rows])
