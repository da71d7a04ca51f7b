"""GPU parity: every call of the C ABI against the CPU oracle on identical
seeded inputs. Integer and byte results must be bit-exact; bf16 GEMM outputs
must meet the acceptance tolerance (helpers.REL_FRO / REL_MAX)."""

import numpy as np
import pytest

import oracle as O
import wq_inputs as I
from helpers import (Guarded, assert_bf16_close, bf16_dev_to_bits, packed_dev_to_u32, to_dev,
                     to_dev_bf16)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import weight_only_int2_gb300 as wq  # noqa: E402


def _layer(N, K, bits, seed, sign="random"):
    q = I.make_codes(N, K, bits, seed)
    s = I.make_scales(N, K // 128, seed + 1, sign=sign)
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), bits)
    return q, s, packed, s_dev


# ------------------------------------------------------------------ repack

@pytest.mark.parametrize("bits", range(2, 9))
@pytest.mark.parametrize("N,K", [(1, 128), (37, 384), (130, 5120)])
def test_repack_bit_exact(bits, N, K):
    q = I.make_codes(N, K, bits, 100 + bits)
    q[0, :7] = (1 << bits) - 1       # extremes at the start of the first row
    q[-1, -5:] = 0
    bad = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = I.make_scales(N, K // 128, 7)
    gp = Guarded((N, wq.packed_words_per_row(K, bits)), torch.int32)
    gs = Guarded((N, K // 128), torch.bfloat16)
    packed, s_out = wq.wna16_repack(to_dev(q), to_dev_bf16(s), bits, packed=gp.t, scales_out=gs.t, bad_count=bad)
    gp.check("packed")
    gs.check("scales_out")
    assert np.array_equal(packed_dev_to_u32(packed), O.pack(q, bits))
    assert np.array_equal(bf16_dev_to_bits(s_out), s)
    assert int(bad.item()) == 0
    # inverse on the GPU
    assert np.array_equal(wq.debug_unpack(packed, N, K, bits).cpu().numpy(), q)


@pytest.mark.parametrize("bits", [3, 5, 6, 7])
def test_repack_counts_out_of_range_and_masks(bits):
    N, K = 3, 256
    q = I.make_codes(N, K, bits, 5)
    q[1, 10] = 200
    q[2, 255] = (1 << bits)
    bad = torch.zeros(1, dtype=torch.int32, device="cuda")
    packed, _ = wq.wna16_repack(to_dev(q), to_dev_bf16(I.make_scales(N, 2, 6)), bits, bad_count=bad)
    torch.cuda.synchronize()
    assert int(bad.item()) == O.count_out_of_range(q, bits) == 2
    assert np.array_equal(packed_dev_to_u32(packed), O.pack(q, bits))


def test_unpack_of_oracle_packed_data():
    for bits in range(2, 9):
        q = I.make_codes(9, 640, bits, 30 + bits)
        p = O.pack(q, bits)
        dev = to_dev(p.view(np.int32))
        assert np.array_equal(wq.debug_unpack(dev, 9, 640, bits).cpu().numpy(), q)


# ------------------------------------------------------------------ WNA16 GEMM

CASES = [
    # (M, N, K, bits)
    (1, 1024, 512, 6),      # the tiny configuration
    (1, 37, 128, 5),
    (2, 129, 384, 7),
    (3, 300, 640, 2),
    (5, 200, 1280, 3),
    (8, 257, 768, 4),
    (9, 131, 512, 8),
    (16, 128, 1024, 5),
    (17, 77, 384, 6),
    (33, 160, 256, 7),
    (63, 96, 896, 6),
    (64, 250, 512, 8),
    (65, 140, 384, 5),
    (130, 70, 256, 6),
    (200, 129, 640, 7),
    # persistent decode kernel (M <= 16, K a multiple of 1024)
    (1, 1000, 2048, 6),
    (4, 700, 5120, 7),
    (16, 300, 3072, 8),
    (3, 50, 1024, 3),
    (12, 2000, 5120, 5),
    (1, 17, 1024, 2),
    (9, 4096, 1024, 4),
    (2, 5120, 5120, 6),
]


@pytest.mark.parametrize("M,N,K,bits", CASES)
def test_wna16_gemm_matches_oracle(M, N, K, bits):
    seed = 10 * M + N + bits
    x = I.make_x(M, K, seed)
    q, s, packed, s_dev = _layer(N, K, bits, seed + 3)
    g = Guarded((M, N), torch.bfloat16)
    y = wq.wna16_gemm(to_dev_bf16(x), packed, s_dev, N, K, bits, y=g.t)
    g.check(f"y M={M} N={N} K={K} b={bits}")
    assert_bf16_close(y, O.wna16_ref(x, q, s, bits), f"M={M} N={N} K={K} b={bits}")


@pytest.mark.parametrize("bits", [5, 6, 7, 8])
def test_wna16_all_negative_scales_and_constant_codes(bits):
    M, N, K = 4, 150, 512
    x = I.make_x(M, K, 3)
    q, s, packed, s_dev = _layer(N, K, bits, 4, sign="negative")
    y = wq.wna16_gemm(to_dev_bf16(x), packed, s_dev, N, K, bits)
    assert_bf16_close(y, O.wna16_ref(x, q, s, bits), "negative scales")
    for c in (0, (1 << bits) - 1):
        qc = np.full((N, K), c, dtype=np.uint8)
        pc, _ = wq.wna16_repack(to_dev(qc), s_dev, bits)
        yc = wq.wna16_gemm(to_dev_bf16(x), pc, s_dev, N, K, bits)
        assert_bf16_close(yc, O.wna16_ref(x, qc, s, bits), f"constant code {c}")
    # codes equal to the zero point give zero up to float32 cancellation
    qz = np.full((N, K), 1 << (bits - 1), dtype=np.uint8)
    pz, _ = wq.wna16_repack(to_dev(qz), s_dev, bits)
    yz = wq.wna16_gemm(to_dev_bf16(x), pz, s_dev, N, K, bits).float()
    ref_scale = np.max(np.abs(O.wna16_ref(x, np.full((N, K), 0, dtype=np.uint8), s, bits)))
    assert float(yz.abs().max()) <= 1e-4 * ref_scale


@pytest.mark.parametrize("K", [2560, 5120])
def test_workspace_returns_to_zero(K):
    M, N, bits = 4, 1000, 6
    need = wq.wna16_workspace_bytes(M, N, K, bits)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    x = I.make_x(M, K, 1)
    q, s, packed, s_dev = _layer(N, K, bits, 2)
    ref = O.wna16_ref(x, q, s, bits)
    for _ in range(3):
        y = wq.wna16_gemm(to_dev_bf16(x), packed, s_dev, N, K, bits, ws=ws)
        torch.cuda.synchronize()
        assert_bf16_close(y, ref, "repeat")
        assert int(ws.count_nonzero()) == 0


# ------------------------------------------------------------------ act-quant

@pytest.mark.parametrize("M,K", [(1, 128), (7, 5120), (64, 1024), (300, 256)])
def test_act_quant_bit_exact(M, K):
    x = I.make_x_outliers(M, K, M + K)
    if M > 2:
        x[1] = 0
    gq, gs = Guarded((M, K), torch.int8), Guarded((M,), torch.float32)
    xq, sx = wq.act_quant_int8(to_dev_bf16(x), xq=gq.t, sx=gs.t)
    gq.check("xq")
    gs.check("sx")
    rq, rs = O.act_quant_ref(x)
    assert np.array_equal(xq.cpu().numpy(), rq)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), rs.view(np.uint32))


def test_act_quant_half_way_cases():
    row = np.array([[127.0, 2.5, 3.5, -2.5, 0.5, 1.5, -0.5, 126.5] + [0.0] * 120], dtype=np.float32)
    x = I._to_bf16_bits(row)
    xq, sx = wq.act_quant_int8(to_dev_bf16(x))
    assert xq.cpu().numpy()[0, :8].tolist() == [127, 2, 4, -2, 0, 2, 0, 126]
    assert float(sx.item()) == 1.0


# ------------------------------------------------------------------ W4A8

# (M, N, K, route): the debug entry runs the kernel w4a8_gemm launches for the
# shape, so every route's integer accumulators are checked bit for bit
W4A8_ACC_CASES = [
    (1, 100, 256, "chunked"), (5, 257, 640, "chunked"), (16, 128, 1280, "chunked"),
    (1, 300, 1024, "decode_pair"), (16, 200, 2048, "decode_pair"), (7, 64, 5120, "decode_pair"),
    (1, 1000, 5120, "decode_pair"), (16, 333, 2048, "decode_pair"),
    (16, 700, 14336, "decode_splitk"),
    (70, 90, 384, "tensor_core"), (100, 257, 640, "tensor_core"), (129, 300, 1024, "tensor_core"),
    (512, 640, 5120, "tensor_core"), (1000, 130, 256, "tensor_core"),
]


@pytest.mark.parametrize("M,N,K,route", W4A8_ACC_CASES)
def test_w4a8_group_accumulators_bit_exact(M, N, K, route):
    assert wq.debug_route(M, N, K, 4, torch.cuda.get_device_properties(0).multi_processor_count,
                          w4a8=True) == route
    x = I.make_x_outliers(M, K, 7 + M)
    q = I.make_codes(N, K, 4, 8 + M)
    xq_ref, _ = O.act_quant_ref(x)
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(I.make_scales(N, K // 128, 1)), 4)
    g = Guarded((M, N, K // 128), torch.int32)
    acc = wq.debug_w4a8_group_acc(to_dev_bf16(x), packed, s_dev, N, K, acc=g.t)
    g.check(f"acc M={M} N={N} K={K}")
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), O.w4a8_group_acc(xq_ref, q))


@pytest.mark.parametrize("M,N,K,sign", [(1, 300, 512, "random"), (4, 129, 1024, "negative"),
                                        (16, 200, 384, "random"), (100, 64, 256, "random"),
                                        (1, 1000, 5120, "random"), (16, 333, 2048, "negative")])
def test_w4a8_gemm_matches_oracle(M, N, K, sign):
    x = I.make_x_outliers(M, K, 20 + M)
    q, s, packed, s_dev = _layer(N, K, 4, 21 + M, sign=sign)
    g = Guarded((M, N), torch.bfloat16)
    y = wq.w4a8_gemm(to_dev_bf16(x), packed, s_dev, N, K, y=g.t)
    g.check(f"w4a8 y M={M}")
    y_ref, _, _ = O.w4a8_ref(x, q, s)
    assert_bf16_close(y, y_ref, f"w4a8 M={M}")


# ------------------------------------------------------------------ gather

@pytest.mark.parametrize("bits", range(2, 9))
def test_gather_bit_exact(bits):
    V, D, T = 50, 640, 33
    q = I.make_codes(V, D, bits, 60 + bits)
    q[3, :128] = 1 << (bits - 1)            # zero offsets -> +-0.0 by scale sign
    s = I.make_scales(V, D // 128, 61)
    s[3, 0] |= np.uint16(0x8000)            # make that group's scale negative
    ids = I.make_ids(T, V, 62)
    ids[0] = 3
    ids[5] = -4
    ids[6] = V
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), bits)
    bad = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = Guarded((T, D), torch.bfloat16)
    out = wq.qembed_gather(to_dev(ids), packed, s_dev, V, D, bits, out=g.t, bad_count=bad)
    g.check("gather out")
    ref, nbad = O.qembed_ref(ids, q, s, bits)
    assert np.array_equal(bf16_dev_to_bits(out), ref)
    assert int(bad.item()) == nbad == 2
    assert np.all(bf16_dev_to_bits(out)[0, :128] == 0x8000)


@pytest.mark.parametrize("bits", [5, 8])
def test_gather_long_rows(bits):
    """Rows longer than any shared-memory staging could hold (256 K codes,
    up to 256 KB packed): the gather reads them from global memory."""
    V, D, T = 5, 262144, 7
    q = I.make_codes(V, D, bits, 90 + bits)
    s = I.make_scales(V, D // 128, 91)
    ids = np.array([4, 0, 2, 2, -1, 3, 1], dtype=np.int32)
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), bits)
    bad = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = Guarded((T, D), torch.bfloat16)
    out = wq.qembed_gather(to_dev(ids), packed, s_dev, V, D, bits, out=g.t, bad_count=bad)
    g.check("gather out (long rows)")
    ref, nbad = O.qembed_ref(ids, q, s, bits)
    assert np.array_equal(bf16_dev_to_bits(out), ref)
    assert int(bad.item()) == nbad == 1


@pytest.mark.parametrize("bits", [5, 8])
def test_gather_tiny_and_huge_scales(bits):
    """Scales whose products with (q - z) fall in the bf16 subnormal range
    (2^-133 .. 2^-126), are subnormal themselves, or are very large: the
    gather still rounds the exact product once, as the definition says."""
    V, D = 6, 256
    q = I.make_codes(V, D, bits, 95 + bits)
    sv = np.array([2.0 ** -130, -(2.0 ** -133), 2.0 ** -125, 2.0 ** -120, 2.0 ** 100, -(2.0 ** 120)],
                  dtype=np.float32)
    s = np.repeat(O.f32_to_bf16_bits_rne(sv)[:, None], D // 128, axis=1).astype(np.uint16)
    ids = np.arange(V, dtype=np.int32)
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), bits)
    out = wq.qembed_gather(to_dev(ids), packed, s_dev, V, D, bits)
    torch.cuda.synchronize()
    ref, _ = O.qembed_ref(ids, q, s, bits)
    assert np.array_equal(bf16_dev_to_bits(out), ref)


def test_gather_empty():
    packed, s_dev = wq.wna16_repack(to_dev(I.make_codes(4, 128, 8, 1)),
                                    to_dev_bf16(I.make_scales(4, 1, 2)), 8)
    out = wq.qembed_gather(torch.zeros(0, dtype=torch.int32, device="cuda"), packed, s_dev, 4, 128, 8)
    assert out.shape == (0, 128)


def test_status_word_clear_after_runs():
    wq.check_status()


def test_w4a8_decode_quantizes_like_act_quant():
    """Few tokens: the decode kernel quantizes the activations itself. With
    half-way values (x / sx = k + 1/2), every code q - z = 1 and unit scales,
    y is the exact integer sum of the int8 codes, so any difference in
    rounding from the activation-quant definition shows up bit for bit."""
    M, N, K = 3, 64, 1024
    row = np.zeros((1, K), dtype=np.float32)
    row[0, :8] = [127.0, 2.5, 3.5, -2.5, 0.5, 1.5, -0.5, 126.5]
    row[0, 300:304] = [-4.5, 5.5, -6.5, 7.5]
    x = np.zeros((M, K), dtype=np.uint16)
    x[0] = I._to_bf16_bits(row)[0]
    x[2] = I._to_bf16_bits(row * np.float32(2.0))[0]   # sx = 2: the same codes
    q = np.full((N, K), 9, dtype=np.uint8)
    s = np.full((N, K // 128), 0x3F80, dtype=np.uint16)  # bf16 1.0
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), 4)
    y = wq.w4a8_gemm(to_dev_bf16(x), packed, s_dev, N, K)
    torch.cuda.synchronize()
    y_ref, _, _ = O.w4a8_ref(x, q, s)
    ref_bits = O.f32_to_bf16_bits_rne(y_ref.astype(np.float32))
    assert np.array_equal(bf16_dev_to_bits(y), ref_bits)
    assert np.all(bf16_dev_to_bits(y)[1] == 0)  # all-zero token


@pytest.mark.parametrize("M", [1, 5, 16])
def test_w4a8_decode_codes_bit_exact(M):
    """Every int8 code of the in-kernel quantization, checked one by one:
    row n of W is the zero point (8) except 9 at column n, unit scales, so
    y[m, n] = RN32(sx[m] * xq[m, n]) rounded to bf16. Outlier activations
    make the per-token scales differ widely."""
    N = K = 1024
    x = I.make_x_outliers(M, K, 500 + M)
    q = np.full((N, K), 8, dtype=np.uint8)
    q[np.arange(N), np.arange(N)] = 9
    s = np.full((N, K // 128), 0x3F80, dtype=np.uint16)
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), 4)
    y = wq.w4a8_gemm(to_dev_bf16(x), packed, s_dev, N, K)
    torch.cuda.synchronize()
    xq, sx = O.act_quant_ref(x)
    ref = O.f32_to_bf16_bits_rne((xq.astype(np.float32) * sx[:, None]).astype(np.float32))
    assert np.array_equal(bf16_dev_to_bits(y), ref)


@pytest.mark.parametrize("side", ["tiny", "huge"])
def test_w4a8_decode_codes_extreme_scales(side):
    """The in-kernel quantization at token scales far from 1: a subnormal sx
    (activations near 2^-130), sx near 2^-101, 2^99 and 2^119. The diagonal
    weight pattern with group scale 2^120 (tiny tokens) or 2^-120 (huge ones)
    keeps y = RN32(xq * sx * s) a normal number, so every int8 code shows in
    y bit for bit."""
    N = K = 1024
    exps = [-130, -124, -100] if side == "tiny" else [100, 120]
    base = O.bf16_bits_to_f32(I.make_x_outliers(len(exps), K, 700))
    rows = [base[i] * np.float32(2.0 ** e) for i, e in enumerate(exps)]
    x = I._to_bf16_bits(np.stack(rows).astype(np.float32))
    q = np.full((N, K), 8, dtype=np.uint8)
    q[np.arange(N), np.arange(N)] = 9
    s_val = 2.0 ** 120 if side == "tiny" else 2.0 ** -120
    s = np.full((N, K // 128), O.f32_to_bf16_bits_rne(np.array([s_val], dtype=np.float32))[0], dtype=np.uint16)
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), 4)
    y = wq.w4a8_gemm(to_dev_bf16(x), packed, s_dev, N, K)
    torch.cuda.synchronize()
    xq, sx = O.act_quant_ref(x)
    assert np.all(sx > 0)
    if side == "tiny":
        assert sx[0] < np.float32(2.0 ** -126)  # the subnormal case is exercised
    sxs = (sx.astype(np.float64) * s_val).astype(np.float32)  # exact: a power-of-two scaling
    ref = O.f32_to_bf16_bits_rne((xq.astype(np.float32) * sxs[:, None]).astype(np.float32))
    assert np.array_equal(bf16_dev_to_bits(y), ref)
