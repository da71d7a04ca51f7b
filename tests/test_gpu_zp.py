"""GPU parity of wna16_gemm_zp, the linear layer with asymmetric groups (a
zero point per output row and 128-wide group, model card "Findings", second
bullet), against the oracle's wna16_zp_ref: every route (CTA-pair decode,
chunked split-K, tensor-core prefill), widths 2..8, random and extreme zero
points, the zero point's high bits ignored, and the full-size decode sweep
(sampled rows). With every zero point at 2^(b-1) the layer is the symmetric
one, bit for bit."""

import numpy as np
import pytest

import oracle as O
import wq_inputs as I
from helpers import Guarded, assert_bf16_close, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import weight_only_int2_gb300 as wq  # noqa: E402


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _zeros(N, G, bits, seed):
    return np.random.default_rng(seed).integers(0, 1 << bits, size=(N, G)).astype(np.uint8)


def _layer(N, K, bits, seed):
    q = I.make_codes(N, K, bits, seed)
    s = I.make_scales(N, K // 128, seed + 1)
    zp = _zeros(N, K // 128, bits, seed + 2)
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), bits)
    return q, s, zp, packed, s_dev


CASES = [
    # (M, N, K, bits, route)
    (1, 1000, 2048, 6, "decode_pair"),
    (4, 700, 5120, 5, "decode_pair"),
    (16, 300, 3072, 8, "decode_pair"),
    (9, 257, 1024, 7, "decode_pair"),
    (3, 129, 1024, 4, "decode_pair"),
    (1, 37, 1024, 2, "decode_pair"),
    (2, 200, 1024, 3, "decode_pair"),
    (1, 300, 640, 6, "chunked"),
    (17, 77, 384, 5, "chunked"),
    (31, 129, 896, 8, "chunked"),
    (16, 700, 14336, 6, "chunked"),     # the symmetric call takes the split-K decode kernel
    (65, 140, 384, 5, "tensor_core"),
    (200, 129, 640, 7, "tensor_core"),
    (300, 257, 768, 8, "tensor_core"),
    (129, 130, 256, 4, "tensor_core"),
    (513, 640, 512, 6, "tensor_core"),
]


@pytest.mark.parametrize("M,N,K,bits,route", CASES)
def test_zp_matches_oracle(M, N, K, bits, route):
    assert wq.debug_route(M, N, K, bits, _sms(), zp=True) == route
    seed = 3 * M + N + bits
    x = I.make_x(M, K, seed)
    q, s, zp, packed, s_dev = _layer(N, K, bits, seed + 7)
    g = Guarded((M, N), torch.bfloat16)
    y = wq.wna16_gemm_zp(to_dev_bf16(x), packed, s_dev, to_dev(zp), N, K, bits, y=g.t)
    g.check(f"zp y M={M} N={N} K={K} b={bits}")
    assert_bf16_close(y, O.wna16_zp_ref(x, q, s, zp, bits), f"zp M={M} N={N} K={K} b={bits} ({route})")
    wq.check_status()


@pytest.mark.parametrize("M,N,K,bits", [(1, 500, 2048, 6), (16, 300, 1024, 8), (20, 200, 640, 5),
                                        (100, 257, 512, 7), (300, 129, 256, 8)])
def test_zp_at_half_range_equals_the_symmetric_layer_bit_for_bit(M, N, K, bits):
    x = I.make_x(M, K, 900 + M)
    q, s, _, packed, s_dev = _layer(N, K, bits, 901)
    zp = np.full((N, K // 128), 1 << (bits - 1), dtype=np.uint8)
    y_zp = wq.wna16_gemm_zp(to_dev_bf16(x), packed, s_dev, to_dev(zp), N, K, bits)
    y = wq.wna16_gemm(to_dev_bf16(x), packed, s_dev, N, K, bits)
    torch.cuda.synchronize()
    assert torch.equal(y_zp.view(torch.int16), y.view(torch.int16))


@pytest.mark.parametrize("M", [1, 16, 24, 300])
@pytest.mark.parametrize("bits", [5, 8])
def test_zp_extremes_and_high_bits(M, bits):
    """Zero points 0 and 2^b - 1 in alternate groups, high bits set on some
    bytes (only the low `bits` bits count), codes at both ends."""
    N, K = 160, 1024
    x = I.make_x(M, K, 950 + M)
    q = I.make_codes(N, K, bits, 951)
    q[:, :128] = 0
    q[:, 128:256] = (1 << bits) - 1
    s = I.make_scales(N, K // 128, 952)
    zp = np.zeros((N, K // 128), dtype=np.uint8)
    zp[:, 1::2] = (1 << bits) - 1
    zp_bytes = zp.copy()
    if bits < 8:
        zp_bytes[::3] |= np.uint8(0x80)
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), bits)
    y = wq.wna16_gemm_zp(to_dev_bf16(x), packed, s_dev, to_dev(zp_bytes), N, K, bits)
    assert_bf16_close(y, O.wna16_zp_ref(x, q, s, zp_bytes, bits), f"zp extremes M={M} b={bits}")
    wq.check_status()


@pytest.mark.parametrize("bits", [5, 6, 7])
@pytest.mark.parametrize("N", [5120, 17408])
def test_zp_decode_sweep_full_size(bits, N):
    """The decode sweep's shapes (K = 5120, M = 1/4/16/64) with random zero
    points, sampled output rows."""
    K = 5120
    q, s, zp, packed, s_dev = _layer(N, K, bits, 5000 + bits)
    zd = to_dev(zp)
    r = np.random.default_rng(N + bits)
    ns = np.unique(np.concatenate([r.choice(N, 64, replace=False), [0, N - 1]]).astype(np.int64))
    for M in (1, 4, 16, 64):
        x = I.make_x(M, K, 5100 + M)
        y = wq.wna16_gemm_zp(to_dev_bf16(x), packed, s_dev, zd, N, K, bits)
        torch.cuda.synchronize()
        got = y[:, torch.as_tensor(ns, device="cuda")]
        assert_bf16_close(got, O.wna16_zp_ref(x, q[ns], s[ns], zp[ns], bits), f"zp sweep b={bits} N={N} M={M}")
    wq.check_status()
