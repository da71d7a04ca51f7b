"""Planted mistakes in the CPU oracle: each case replaces one oracle function
with a copy that carries one plausible error (a flipped bit order, a wrong
zero point or group index, a reciprocal multiply, truncation instead of
round-to-nearest-even, a dropped factor ...) and checks that at least one of
the oracle's pins fails. The pins are the functions of test_oracle_pins.py,
run here against the mutated oracle. CPU only; the mistakes live in
monkeypatched copies and never touch the oracle module on disk.

A mistake that no valid input can expose (say, floor instead of ceil in the
row length when K is a multiple of 128) is not listed: no pin could catch it
and none needs to.
"""

import numpy as np
import pytest

import oracle
import oracle.wq_oracle as W
import test_oracle_pins as P

# ------------------------------------------------------------ the pins, small


def _pin_calls():
    calls = [("row lengths", P.test_golden_row_lengths_from_model_card, ()),
             ("hand-worked b5", P.test_golden_hand_worked_b5_example, ()),
             ("out of range", P.test_out_of_range_codes_counted_and_masked, ()),
             ("b8 int8 matmul", P.test_b8_unit_scales_is_plain_int8_matmul, ()),
             ("sign symmetry", P.test_scale_sign_symmetry_and_all_negative, ()),
             ("half-way rounding", P.test_act_quant_half_way_cases_round_to_even, ()),
             ("act-quant invariants", P.test_act_quant_invariants, ()),
             ("act-quant exact division", P.test_act_quant_is_ieee_division_then_round_half_even, ()),
             ("w4a8 integer path", P.test_w4a8_group_acc_sums_to_integer_matmul_and_unit_scales, ()),
             ("w4a8 brute force", P.test_w4a8_brute_force_exact_rationals, ()),
             ("w4a8 vs wna16", P.test_w4a8_close_to_wna16_b4, ()),
             ("bf16 rne", P.test_bf16_rne_hand_cases, ()),
             ("gather -0.0", P.test_gather_negative_zero_and_unit_scale_b8, ()),
             ("gather exact rounding", P.test_gather_exact_products_round_half_even, ()),
             ("page byte counts", P.test_page_byte_counts_pin_group_128_scales, ())]
    for b in range(2, 9):
        calls.append((f"round trip b{b}", P.test_round_trip_random_and_extremes, (b, 128)))
        calls.append((f"big integer b{b}", P.test_pack_equals_big_integer_construction, (b,)))
    for b in (2, 4, 8):
        calls.append((f"word-aligned b{b}", P.test_dense_layout_equals_word_aligned_formula_when_bits_divides_32,
                      (b,)))
    for b in (5, 8):
        calls.append((f"brute force b{b}", P.test_wna16_brute_force_exact_rationals, (b,)))
        calls.append((f"gather b{b}", P.test_gather_is_rounded_dequant_with_ids_out_of_range, (b,)))
    for b in (5, 6):
        for kind in ("zero_point", "min", "max"):
            calls.append((f"closed form b{b} {kind}", P.test_wna16_closed_form_constant_codes, (b, kind)))
    for b in (5, 8):
        calls.append((f"zp brute force b{b}", P.test_zp_brute_force_exact_rationals, (b,)))
        calls.append((f"zp closed form b{b}", P.test_zp_closed_form_constant_codes, (b,)))
        calls.append((f"zp at half range b{b}", P.test_zp_at_half_range_is_the_symmetric_layer, (b,)))
    calls.append(("zp shift invariance", P.test_zp_shift_invariance, ()))
    calls.append(("moe brute force", P.test_moe_brute_force_exact_rationals, ()))
    calls.append(("moe dense reductions", P.test_moe_with_one_expert_or_equal_experts_is_the_dense_layer, ()))
    calls.append(("moe row order", P.test_moe_rows_follow_their_expert, ()))
    calls.append(("zp low bits", P.test_zp_uses_the_low_bits_of_each_byte, ()))
    return calls


# a loose comparison the pins file reports without gating parity on it; a
# mistake it alone notices is not counted as caught
REPORTED_ONLY = {"w4a8 vs wna16"}


def _failing_pins():
    failed = []
    for name, fn, args in _pin_calls():
        try:
            fn(*args)
        except Exception:  # an assertion, or an error the mistake provokes
            failed.append(name)
    return failed


# ------------------------------------------------------------ the mistakes
# Each is a small edit of the function it replaces; the comment says which.

def _pack_msb(codes, bits):
    """pack with bit j of a word stored at position 31 - j."""
    c = np.asarray(codes).astype(np.int64)
    N, K = c.shape
    words = np.zeros((N, W.packed_words_per_row(K, bits)), dtype=np.uint64)
    for k in range(K):
        col = c[:, k].astype(np.uint64)
        for j in range(bits):
            p = k * bits + j
            words[:, p // 32] |= ((col >> np.uint64(j)) & np.uint64(1)) << np.uint64(31 - p % 32)
    return words.astype(np.uint32)


def _unpack_msb(packed, K, bits):
    w = np.asarray(packed, dtype=np.uint32).astype(np.uint64)
    codes = np.zeros((w.shape[0], K), dtype=np.uint64)
    for k in range(K):
        for j in range(bits):
            p = k * bits + j
            codes[:, k] |= ((w[:, p // 32] >> np.uint64(31 - p % 32)) & np.uint64(1)) << np.uint64(j)
    return codes.astype(np.int64)


def _pack_codes_msb_first(codes, bits):
    """pack with the code's own bits reversed (its top bit first in the stream)."""
    c = np.asarray(codes).astype(np.int64)
    N, K = c.shape
    words = np.zeros((N, W.packed_words_per_row(K, bits)), dtype=np.uint64)
    for k in range(K):
        col = c[:, k].astype(np.uint64)
        for j in range(bits):
            p = k * bits + (bits - 1 - j)
            words[:, p // 32] |= ((col >> np.uint64(j)) & np.uint64(1)) << np.uint64(p % 32)
    return words.astype(np.uint32)


def _unpack_codes_msb_first(packed, K, bits):
    w = np.asarray(packed, dtype=np.uint32).astype(np.uint64)
    codes = np.zeros((w.shape[0], K), dtype=np.uint64)
    for k in range(K):
        for j in range(bits):
            p = k * bits + (bits - 1 - j)
            codes[:, k] |= ((w[:, p // 32] >> np.uint64(p % 32)) & np.uint64(1)) << np.uint64(j)
    return codes.astype(np.int64)


def _pack_word_aligned(codes, bits):
    """pack that starts a new word when a code would straddle one (the older
    word-aligned layout), with the dense row length kept."""
    c = np.asarray(codes).astype(np.int64)
    N, K = c.shape
    per = 32 // bits
    words = np.zeros((N, W.packed_words_per_row(K, bits)), dtype=np.uint64)
    for k in range(K):
        wi, sh = k // per, (k % per) * bits
        if wi < words.shape[1]:
            words[:, wi] |= (c[:, k].astype(np.uint64) & np.uint64((1 << bits) - 1)) << np.uint64(sh)
    return words.astype(np.uint32)


def _unpack_word_aligned(packed, K, bits):
    w = np.asarray(packed, dtype=np.uint32).astype(np.uint64)
    per = 32 // bits
    codes = np.zeros((w.shape[0], K), dtype=np.int64)
    for k in range(K):
        wi, sh = k // per, (k % per) * bits
        if wi < w.shape[1]:
            codes[:, k] = ((w[:, wi] >> np.uint64(sh)) & np.uint64((1 << bits) - 1)).astype(np.int64)
    return codes


def _zero_point_minus_one(bits):
    return (1 << (int(bits) - 1)) - 1


def _zero_point_full_range(bits):
    """midpoint of [0, 2^b - 1] rounded down, taken as 2^b / 2 - 1/2 -> floor."""
    return ((1 << int(bits)) - 1) // 2


def _dequant_tiled_scales(codes, scales_bits, bits, group=W.GROUP):
    """scale of column k taken from group k mod G instead of k // 128."""
    q = np.asarray(codes).astype(np.float64)
    s = W.bf16_bits_to_f64(scales_bits)
    return np.tile(s, group) * (q - float(W.zero_point(bits)))


def _dequant_sign_flipped(codes, scales_bits, bits, group=W.GROUP):
    q = np.asarray(codes).astype(np.float64)
    s = np.repeat(W.bf16_bits_to_f64(scales_bits), group, axis=1)
    return s * (float(W.zero_point(bits)) - q)


def _dequant_abs_scales(codes, scales_bits, bits, group=W.GROUP):
    """the scale's sign bit dropped (bf16 read as unsigned magnitude)."""
    q = np.asarray(codes).astype(np.float64)
    s = np.repeat(np.abs(W.bf16_bits_to_f64(scales_bits)), group, axis=1)
    return s * (q - float(W.zero_point(bits)))


def _wna16_in_float32(x_bits, codes, scales_bits, bits, group=W.GROUP):
    x = W.bf16_bits_to_f32(x_bits)
    w = W.dequant(codes, scales_bits, bits, group).astype(np.float32)
    return (x @ w.T).astype(np.float64)


def _wna16_weights_rounded_to_bf16(x_bits, codes, scales_bits, bits, group=W.GROUP):
    """weights rounded to bf16 before the product (the dequant-then-bf16-GEMM
    shortcut), instead of the exact float64 weights."""
    x = W.bf16_bits_to_f64(x_bits)
    w = W.dequant(codes, scales_bits, bits, group).astype(np.float32)
    w = W.bf16_bits_to_f64(W.f32_to_bf16_bits_rne(w))
    return x @ w.T


def _act_quant_variant(ratio_fn=None, round_fn=np.rint, divisor=127.0, per_token=True):
    """act_quant_ref with one step swapped: the x / sx division, the rounding,
    the divisor of amax, or the per-token amax (per_token=False: one amax for
    the whole tensor)."""
    def act_quant(x_bits):
        x = W.bf16_bits_to_f32(x_bits)
        amax = np.max(np.abs(x), axis=1).astype(np.float32)
        if not per_token:
            amax = np.full_like(amax, amax.max())
        sx = (amax / np.float32(divisor)).astype(np.float32)
        xq = np.zeros(x.shape, dtype=np.int8)
        nz = sx > 0
        if nz.any():
            if ratio_fn is None:
                ratio = (x[nz] / sx[nz, None]).astype(np.float32)
            else:
                ratio = ratio_fn(x[nz], sx[nz, None])
            xq[nz] = np.clip(round_fn(ratio), -127, 127).astype(np.int8)
        return xq, np.where(nz, sx, np.float32(0.0)).astype(np.float32)
    return act_quant


def _reciprocal_multiply(x, sx):
    return (x * (np.float32(1.0) / sx)).astype(np.float32)


def _round_half_away(r):
    return np.sign(r) * np.floor(np.abs(r) + 0.5)


def _group_acc_zero_7(xq, codes4, group=W.GROUP):
    a = np.asarray(xq).astype(np.int64)
    w = np.asarray(codes4).astype(np.int64) - 7
    G = a.shape[1] // group
    return np.stack([a[:, g * group:(g + 1) * group] @ w[:, g * group:(g + 1) * group].T for g in range(G)],
                    axis=2)


def _group_acc_interleaved(xq, codes4, group=W.GROUP):
    """group g taken as the columns k with k mod G == g."""
    a = np.asarray(xq).astype(np.int64)
    w = np.asarray(codes4).astype(np.int64) - 8
    G = a.shape[1] // group
    return np.stack([a[:, g::G] @ w[:, g::G].T for g in range(G)], axis=2)


def _w4a8_no_token_scale(xq, sx, codes4, scales_bits, group=W.GROUP):
    acc = W.w4a8_group_acc(xq, codes4, group).astype(np.float64)
    return np.einsum("mng,ng->mn", acc, W.bf16_bits_to_f64(scales_bits))


def _rne_half_up(values):
    f = np.ascontiguousarray(np.asarray(values, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    return (((u + np.uint64(0x8000)) >> np.uint64(16)) & np.uint64(0xFFFF)).astype(np.uint16)


def _rne_truncate(values):
    f = np.ascontiguousarray(np.asarray(values, dtype=np.float32))
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _gather_variant(mode):
    def qembed(ids, codes_table, scales_bits, bits, group=W.GROUP):
        ids = np.asarray(ids).astype(np.int64)
        q = np.asarray(codes_table)
        V, D = q.shape
        s = W.bf16_bits_to_f32(scales_bits)
        out = np.zeros((ids.shape[0], D), dtype=np.uint16)
        bad = 0
        z = np.float32(W.zero_point(bits))
        for t, i in enumerate(ids):
            if i < 0 or (i > V if mode == "id_bound" else i >= V):
                bad += 1
                continue
            row_s = np.repeat(s[i], group).astype(np.float32)
            qf = q[i].astype(np.float32)
            if mode == "distributed":       # s*q - s*z: loses -0.0, rounds twice
                prod = (row_s * qf - row_s * z).astype(np.float32)
            else:
                prod = (row_s * (qf - z)).astype(np.float32)
            if mode == "truncate":
                out[t] = (np.ascontiguousarray(prod).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
            elif mode == "ties_away":       # round half away from zero
                u = np.ascontiguousarray(prod).view(np.uint32).astype(np.uint64)
                out[t] = ((u + np.uint64(0x8000)) >> np.uint64(16)).astype(np.uint16)
            else:
                out[t] = W.f32_to_bf16_bits_rne(prod)
        return out, bad
    return qembed


def _bytes_scale_per_row(rows, cols, bits, group=W.GROUP):
    return int(rows) * (W.packed_words_per_row(cols, bits) * 4 + 2)


def _dequant_zp_variant(kind):
    def f(codes, scales_bits, zeros, bits, group=W.GROUP):
        q = np.asarray(codes).astype(np.float64)
        N, K = q.shape
        s = np.repeat(W.bf16_bits_to_f64(scales_bits), group, axis=1)
        zp = W.zero_points_used(zeros, bits).astype(np.float64)
        if kind == "ignored":          # the symmetric zero point instead
            return s * (q - float(W.zero_point(bits)))
        if kind == "added":            # sign of the zero point flipped
            return s * (q + np.repeat(zp, group, axis=1))
        if kind == "tiled":            # group index k mod G instead of k // group
            G = K // group
            return s * (q - zp[:, np.arange(K) % G])
        if kind == "unmasked":         # every bit of the byte used
            return s * (q - np.repeat(np.asarray(zeros).astype(np.float64), group, axis=1))
        raise ValueError(kind)
    return f


def _zp_bits_masked_wrong(zeros, bits):
    return np.asarray(zeros).astype(np.int64) & ((1 << (int(bits) - 1)) - 1)


def _moe_variant(kind):
    def f(x_bits, offsets, codes, scales_bits, bits, group=W.GROUP):
        off = [int(v) for v in np.asarray(offsets).reshape(-1)]
        c = np.asarray(codes)
        E, N, K = c.shape
        M = np.asarray(x_bits).shape[0]
        y = np.zeros((M, N), dtype=np.float64)
        for e in range(E):
            we = (e + 1) % E if kind == "next expert" else e
            lo, hi = off[e], off[e + 1]
            if kind == "first token dropped":
                lo = min(lo + 1, hi)
            if hi > lo:
                y[lo:hi] = W.wna16_ref(np.asarray(x_bits)[lo:hi], c[we], np.asarray(scales_bits)[we], bits, group)
        return y
    return f


MUTANTS = {
    "MoE tokens use the next expert's weights": {"moe_ref": _moe_variant("next expert")},
    "MoE expert ranges start one token late": {"moe_ref": _moe_variant("first token dropped")},
    "zero point per group ignored": {"dequant_zp": _dequant_zp_variant("ignored")},
    "zero point added instead of subtracted": {"dequant_zp": _dequant_zp_variant("added")},
    "zero point indexed k mod G": {"dequant_zp": _dequant_zp_variant("tiled")},
    "zero point high bits used": {"dequant_zp": _dequant_zp_variant("unmasked")},
    "zero point masked to bits - 1": {"zero_points_used": _zp_bits_masked_wrong},
    "stream bits MSB-first in each word (pack and unpack)": {"pack": _pack_msb, "unpack": _unpack_msb},
    "each code's bits reversed (pack and unpack)": {"pack": _pack_codes_msb_first,
                                                   "unpack": _unpack_codes_msb_first},
    "word-aligned packing, straddling codes moved (pack and unpack)": {"pack": _pack_word_aligned,
                                                                      "unpack": _unpack_word_aligned},
    "zero point 2^(b-1) - 1": {"zero_point": _zero_point_minus_one},
    "zero point (2^b - 1) // 2": {"zero_point": _zero_point_full_range},
    "group scale indexed k mod G": {"dequant": _dequant_tiled_scales},
    "dequant sign flipped": {"dequant": _dequant_sign_flipped},
    "scale sign dropped": {"dequant": _dequant_abs_scales},
    "GEMM in float32": {"wna16_ref": _wna16_in_float32},
    "weights rounded to bf16 before the GEMM": {"wna16_ref": _wna16_weights_rounded_to_bf16},
    "act-quant reciprocal multiply": {"act_quant_ref": _act_quant_variant(ratio_fn=_reciprocal_multiply)},
    "act-quant round half away from zero": {"act_quant_ref": _act_quant_variant(round_fn=_round_half_away)},
    "act-quant truncation toward zero": {"act_quant_ref": _act_quant_variant(round_fn=np.trunc)},
    "act-quant scale amax / 128": {"act_quant_ref": _act_quant_variant(divisor=128.0)},
    "act-quant one scale for all tokens": {"act_quant_ref": _act_quant_variant(per_token=False)},
    "W4A8 zero point 7": {"w4a8_group_acc": _group_acc_zero_7},
    "W4A8 groups interleaved": {"w4a8_group_acc": _group_acc_interleaved},
    "W4A8 token scale dropped": {"w4a8_ref_from_quant": _w4a8_no_token_scale},
    "bf16 rounding half up": {"f32_to_bf16_bits_rne": _rne_half_up},
    "bf16 rounding by truncation": {"f32_to_bf16_bits_rne": _rne_truncate},
    "gather truncates to bf16": {"qembed_ref": _gather_variant("truncate")},
    "gather rounds ties away from zero": {"qembed_ref": _gather_variant("ties_away")},
    "gather computes s*q - s*z": {"qembed_ref": _gather_variant("distributed")},
    "gather accepts id == V": {"qembed_ref": _gather_variant("id_bound")},
    "one scale per table row in the byte count": {"quantized_matrix_bytes": _bytes_scale_per_row},
}


def test_pins_pass_on_the_oracle_as_written():
    assert _failing_pins() == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    for fn_name, repl in MUTANTS[name].items():
        assert hasattr(W, fn_name), fn_name
        monkeypatch.setattr(W, fn_name, repl)
        monkeypatch.setattr(oracle, fn_name, repl)
    failed = [p for p in _failing_pins() if p not in REPORTED_ONLY]
    assert failed, f"no pin catches: {name}"
