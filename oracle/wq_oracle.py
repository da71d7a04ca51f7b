"""CPU oracle for the weight-only quantized linear layer.

TEST INFRASTRUCTURE. This module exists to check the CUDA library. Only the
test suite, the smoke check of the entry module and the CPU-baseline leg of the
benchmark may import or run it. The product path (the CUDA library and its
Python binding) never calls it, and the two share no code: no kernels, helpers,
tables or constant generators.

Everything here is written for a reader who checks it against the source pages
by eye: plain loops over bits, float64 arithmetic, one library matmul per GEMM.
No blocking, fusion or reordering beyond what the definitions state.

Sources (cited by page title and section):

* "Qwen3.8-27B-INT6-Mixed-AutoRound" model card, section "Findings", first
  bullet: the compressed-tensors pack-quantized layout stores a row of
  ``in_features`` b-bit codes densely in ``ceil(in_features * bits / 32)``
  32-bit words, so codes may straddle a word boundary. The same bullet shows the
  older word-aligned formula ``shift = (col % (32 // bits)) * bits``, which puts
  the first code of a word in its least significant bits. Reading adopted here:
  the dense stream is LSB-first as well (stream bit j is bit j % 32 of word
  j // 32). The two layouts then coincide when bits divides 32 (pinned by test).
* Same card, "Findings", second bullet: groups above four bits are symmetric.
  Reading adopted: zero point 2^(bits-1), one bf16 scale per (output row,
  128-wide group along K); scales may be negative ("int8 activations (W4A8) ..."
  discussion, section "Under the hood": AutoRound emits about half negative
  group scales).
* "vLLM Can Run INT5-7", section 2: the pages' own reference evaluation
  dequantizes to a float weight and runs a plain F.linear. The oracle does the
  same, in float64.
* "int8 activations (W4A8) ..." discussion, section "Under the hood": per-token
  dynamic int8 activation quantization, int4 weights widened to int8
  losslessly, integer accumulation. The arithmetic details the page leaves open
  (float32, scale = amax/127 by IEEE division, x/scale by IEEE division,
  round-half-to-even, clamp to +-127, int32 accumulation per 128-wide group)
  are readings, stated on each function.
* "vLLM Can Run INT5-7", section 3 and the model card "Findings": the
  quantized embedding is a dequantize-and-gather of table rows.

Parity pins: every function here is pinned by the CPU tests (round trip,
big-integer construction, the word-aligned formula, exact rational brute
force, closed forms, sign symmetry, hand-computed rounding cases, the byte
counts printed on the pages). Float summation order in the GEMMs is the only
unpinned freedom, and the acceptance tolerance covers it.
"""

from __future__ import annotations

import numpy as np

GROUP = 128


# --------------------------------------------------------------------------
# bf16 <-> float conversions (the oracle's own, from the IEEE definitions)
# --------------------------------------------------------------------------

def bf16_bits_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32. Exact: bf16 is the top half of
    a float32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact)."""
    return bf16_bits_to_f32(bits).astype(np.float64)


def f32_to_bf16_bits_rne(values) -> np.ndarray:
    """float32 -> bf16 bits with round-to-nearest-even.

    Keeping the top 16 bits of the float32 pattern truncates; adding
    0x7FFF plus the lowest kept bit before truncating rounds half-way cases
    to the even neighbour and everything else to the nearest one. NaNs map to
    the quiet NaN 0x7FC0 (sign kept)."""
    f = np.ascontiguousarray(np.asarray(values, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    keep_lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + keep_lsb) >> np.uint64(16)) & np.uint64(0xFFFF)
    out = r.astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        sign = ((u >> np.uint64(16)) & np.uint64(0x8000)).astype(np.uint16)
        out = np.where(nan, sign | np.uint16(0x7FC0), out)
    return out


# --------------------------------------------------------------------------
# Packed layout (model card, "Findings": dense ceil(K*bits/32)-word rows)
# --------------------------------------------------------------------------

def packed_words_per_row(K: int, bits: int) -> int:
    """Number of 32-bit words a row of K b-bit codes takes in the dense
    layout: ceil(K * bits / 32)."""
    return (int(K) * int(bits) + 31) // 32


def zero_point(bits: int) -> int:
    """Symmetric zero point above four bits (and the W4A8 int4 case): 2^(b-1)."""
    return 1 << (int(bits) - 1)


def pack(codes, bits: int) -> np.ndarray:
    """Pack integer codes [N, K] into the dense LSB-first bitstream.

    Code k of a row occupies stream bits [k*bits, k*bits + bits); stream bit
    j is bit (j % 32) of word j // 32. Codes larger than 2^bits - 1 keep their
    low ``bits`` bits (the library counts them; see count_out_of_range)."""
    c = np.asarray(codes).astype(np.int64)
    if c.ndim != 2:
        raise ValueError("codes must be 2-D [N, K]")
    N, K = c.shape
    words = np.zeros((N, packed_words_per_row(K, bits)), dtype=np.uint64)
    for k in range(K):
        col = c[:, k].astype(np.uint64)
        for j in range(bits):
            p = k * bits + j
            bit = (col >> np.uint64(j)) & np.uint64(1)
            words[:, p // 32] |= bit << np.uint64(p % 32)
    return words.astype(np.uint32)


def unpack(packed, K: int, bits: int) -> np.ndarray:
    """Inverse of pack: read K codes of ``bits`` bits back from each row."""
    w = np.asarray(packed, dtype=np.uint32).astype(np.uint64)
    if w.ndim != 2 or w.shape[1] < packed_words_per_row(K, bits):
        raise ValueError("packed rows too short for K codes")
    N = w.shape[0]
    codes = np.zeros((N, K), dtype=np.uint64)
    for k in range(K):
        for j in range(bits):
            p = k * bits + j
            bit = (w[:, p // 32] >> np.uint64(p % 32)) & np.uint64(1)
            codes[:, k] |= bit << np.uint64(j)
    return codes.astype(np.int64)


def count_out_of_range(codes, bits: int) -> int:
    """How many codes lie outside [0, 2^bits - 1]."""
    c = np.asarray(codes).astype(np.int64)
    return int(np.count_nonzero((c < 0) | (c > (1 << bits) - 1)))


# --------------------------------------------------------------------------
# Dequantization and the WNA16 linear layer
# --------------------------------------------------------------------------

def dequant(codes, scales_bits, bits: int, group: int = GROUP) -> np.ndarray:
    """w[n, k] = s[n, k // group] * (q[n, k] - 2^(bits-1)) in float64.

    ``scales_bits`` are bf16 bit patterns [N, K // group]; bf16 -> float64 is
    exact, and so is every product here."""
    q = np.asarray(codes).astype(np.float64)
    N, K = q.shape
    if K % group:
        raise ValueError("K must be a multiple of the group size")
    s = bf16_bits_to_f64(scales_bits)
    if s.shape != (N, K // group):
        raise ValueError("scales must be [N, K // group]")
    s_per_k = np.repeat(s, group, axis=1)
    return s_per_k * (q - float(zero_point(bits)))


def wna16_ref(x_bits, codes, scales_bits, bits: int, group: int = GROUP) -> np.ndarray:
    """y = x . dequant(W)^T in float64 (x: bf16 bits [M, K]; codes [N, K])."""
    x = bf16_bits_to_f64(x_bits)
    w = dequant(codes, scales_bits, bits, group)
    return x @ w.T


# --------------------------------------------------------------------------
# Asymmetric groups: a zero point per (output row, group)
# --------------------------------------------------------------------------
# Model card "Qwen3.8-27B-INT6-Mixed-AutoRound", section "Findings", second
# bullet: asymmetric quantization (a zero point per group, not the symmetric
# 2^(b-1)) is what the four-bit tier of the previous build used, worth about a
# quarter of a bit; the serving path there offered it only at 4 and 8 bits.
# The page prints no layout. Readings adopted here: one integer zero point per
# (output row, 128-wide group), stored one byte each [N, K // group], of which
# the low ``bits`` bits are used (as for codes), and w = s * (q - zp).

def zero_points_used(zeros, bits: int) -> np.ndarray:
    """The zero points the layer uses: the low ``bits`` bits of each byte."""
    return np.asarray(zeros).astype(np.int64) & ((1 << int(bits)) - 1)


def dequant_zp(codes, scales_bits, zeros, bits: int, group: int = GROUP) -> np.ndarray:
    """w[n, k] = s[n, k // group] * (q[n, k] - zp[n, k // group]) in float64
    (every product exact)."""
    q = np.asarray(codes).astype(np.float64)
    N, K = q.shape
    if K % group:
        raise ValueError("K must be a multiple of the group size")
    s = bf16_bits_to_f64(scales_bits)
    zp = zero_points_used(zeros, bits).astype(np.float64)
    if s.shape != (N, K // group) or zp.shape != (N, K // group):
        raise ValueError("scales and zeros must be [N, K // group]")
    return np.repeat(s, group, axis=1) * (q - np.repeat(zp, group, axis=1))


def wna16_zp_ref(x_bits, codes, scales_bits, zeros, bits: int, group: int = GROUP) -> np.ndarray:
    """y = x . dequant_zp(W)^T in float64."""
    x = bf16_bits_to_f64(x_bits)
    return x @ dequant_zp(codes, scales_bits, zeros, bits, group).T


# --------------------------------------------------------------------------
# Mixture of experts: a WNA16 layer per expert over its own tokens
# --------------------------------------------------------------------------
# Model card "Qwen3.8-27B-INT6-Mixed-AutoRound", section "Findings", third
# bullet: the serving path of the pages has no fused mixture-of-experts
# WNA16 GEMM at 5/6/7 bits (its MoE method accepts only 4 and 8). The page
# does not describe the grouped layer; the reading adopted here is the plain
# one: the tokens come sorted by expert, expert e owns token rows
# [offsets[e], offsets[e+1]) and applies its own layer (codes [N, K], scales
# [N, K // 128]) to them.

def moe_ref(x_bits, offsets, codes, scales_bits, bits: int, group: int = GROUP) -> np.ndarray:
    """y[offsets[e]:offsets[e+1]] = wna16_ref(x[offsets[e]:offsets[e+1]], W_e)
    for each expert e; codes [E, N, K], scales [E, N, K // group]."""
    off = [int(v) for v in np.asarray(offsets).reshape(-1)]
    c = np.asarray(codes)
    E, N, K = c.shape
    if len(off) != E + 1 or off[0] != 0 or any(off[i] > off[i + 1] for i in range(E)):
        raise ValueError("offsets must be E + 1 nondecreasing values starting at 0")
    M = np.asarray(x_bits).shape[0]
    if off[E] != M:
        raise ValueError("offsets[E] must equal the number of token rows")
    y = np.zeros((M, N), dtype=np.float64)
    for e in range(E):
        if off[e + 1] > off[e]:
            y[off[e]:off[e + 1]] = wna16_ref(np.asarray(x_bits)[off[e]:off[e + 1]], c[e],
                                             np.asarray(scales_bits)[e], bits, group)
    return y


# --------------------------------------------------------------------------
# W4A8: per-token int8 activation quantization and integer accumulation
# --------------------------------------------------------------------------

def act_quant_ref(x_bits):
    """Per-token dynamic int8 quantization, all in IEEE float32.

    amax = max |x| over the row; sx = amax / 127 (IEEE division);
    xq = clamp(round_half_even(x / sx), -127, 127) with x / sx an IEEE
    division, not a reciprocal multiply. A row that is all zeros gets
    sx = 0 and xq = 0. Returns (xq int8 [M, K], sx float32 [M])."""
    x = bf16_bits_to_f32(x_bits)
    amax = np.max(np.abs(x), axis=1).astype(np.float32)
    sx = (amax / np.float32(127.0)).astype(np.float32)
    xq = np.zeros(x.shape, dtype=np.int8)
    nz = sx > 0
    if nz.any():
        ratio = (x[nz] / sx[nz, None]).astype(np.float32)
        r = np.rint(ratio)  # numpy rint rounds half to even
        xq[nz] = np.clip(r, -127, 127).astype(np.int8)
    sx = np.where(nz, sx, np.float32(0.0)).astype(np.float32)
    return xq, sx


def w4a8_group_acc(xq, codes4, group: int = GROUP) -> np.ndarray:
    """acc[m, n, g] = sum_{k in group g} xq[m, k] * (q[n, k] - 8), exact.

    int4 codes widen to int8 (q - 8 in [-8, 7]) without loss; the sum is
    taken in int64 and checked to fit the int32 accumulator the method uses."""
    a = np.asarray(xq).astype(np.int64)
    w = np.asarray(codes4).astype(np.int64) - 8
    M, K = a.shape
    N = w.shape[0]
    G = K // group
    acc = np.zeros((M, N, G), dtype=np.int64)
    for g in range(G):
        sl = slice(g * group, (g + 1) * group)
        acc[:, :, g] = a[:, sl] @ w[:, sl].T
    if acc.size and (acc.max() > 2**31 - 1 or acc.min() < -(2**31)):
        raise OverflowError("group accumulator exceeds int32")
    return acc


def w4a8_ref_from_quant(xq, sx, codes4, scales_bits, group: int = GROUP) -> np.ndarray:
    """y[m, n] = sum_g sx[m] * s[n, g] * acc[m, n, g] in float64."""
    acc = w4a8_group_acc(xq, codes4, group).astype(np.float64)
    s = bf16_bits_to_f64(scales_bits)                     # [N, G]
    sxd = np.asarray(sx, dtype=np.float32).astype(np.float64)
    return sxd[:, None] * np.einsum("mng,ng->mn", acc, s)


def w4a8_ref(x_bits, codes4, scales_bits, group: int = GROUP):
    """Full W4A8 layer: act_quant_ref then the integer path.
    Returns (y float64, xq, sx)."""
    xq, sx = act_quant_ref(x_bits)
    return w4a8_ref_from_quant(xq, sx, codes4, scales_bits, group), xq, sx


# --------------------------------------------------------------------------
# Quantized embedding gather
# --------------------------------------------------------------------------

def qembed_ref(ids, codes_table, scales_bits, bits: int, group: int = GROUP):
    """out[t, d] = bf16_RNE(float32(s[id, d // group]) * float32(q[id, d] - z)).

    ``codes_table`` holds the codes of the table rows [V, D] (or any row
    subset indexed consistently with ``ids``). The float32 product is exact
    (8 x at most 9 significant bits), so one rounding to bf16 remains. A code
    equal to the zero point times a negative scale is -0.0 (IEEE). Ids outside
    [0, V) give a +0.0 row and are counted. Returns (bf16 bits [T, D], bad)."""
    ids = np.asarray(ids).astype(np.int64)
    q = np.asarray(codes_table)
    V, D = q.shape
    s = bf16_bits_to_f32(scales_bits)
    out = np.zeros((ids.shape[0], D), dtype=np.uint16)
    bad = 0
    z = np.float32(zero_point(bits))
    for t, i in enumerate(ids):
        if i < 0 or i >= V:
            bad += 1
            continue
        row_q = q[i].astype(np.float32) - z
        row_s = np.repeat(s[i], group).astype(np.float32)
        out[t] = f32_to_bf16_bits_rne((row_s * row_q).astype(np.float32))
    return out, bad


# --------------------------------------------------------------------------
# Byte counts (vLLM Can Run INT5-7, section 3)
# --------------------------------------------------------------------------

def bf16_matrix_bytes(rows: int, cols: int) -> int:
    return int(rows) * int(cols) * 2


def quantized_matrix_bytes(rows: int, cols: int, bits: int, group: int = GROUP) -> int:
    """Packed codes plus one bf16 scale per (row, group)."""
    return int(rows) * (packed_words_per_row(cols, bits) * 4 + (int(cols) // group) * 2)
