"""GPU parity of the routes that the benchmark shapes do not reach:

* the persistent split-K decode kernel, which few-token calls take when their
  K half does not fit the CTA-pair kernel's shared memory (K of 7168..16384
  by width and token count), in WNA16 and W4A8 modes;
* 17..31 tokens on a 17408-row layer (the chunked split-K kernel);
* the chunked kernel with K above 128 groups (its CTAs split over K), in
  WNA16, W4A8 and zero-point modes, up to K = 131072.

Each case first asserts the route it is meant to cover (so a routing change
cannot quietly turn it into coverage of another kernel), places its output
between sentinel bands, and checks sampled outputs against the oracle
(sampling rows and tokens is exact: each output depends only on its own
weight row and token)."""

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


def _rows(N, k, seed):
    r = np.random.default_rng(seed)
    return np.unique(np.concatenate([r.choice(N, min(k, N), replace=False), [0, N - 1]]).astype(np.int64))


SPLITK_WNA16 = [
    # (M, N, K, bits)
    (1, 17408, 14336, 8),
    (8, 17408, 16384, 6),
    (16, 5120, 14336, 5),
    (16, 700, 16384, 8),
    (16, 17408, 8192, 6),
]


@pytest.mark.parametrize("M,N,K,bits", SPLITK_WNA16)
def test_splitk_decode_wna16(M, N, K, bits):
    assert wq.debug_route(M, N, K, bits, _sms()) == "decode_splitk"
    ns = _rows(N, 96, M + N + K)
    x = I.make_x(M, K, 4000 + M)
    q = I.make_codes(N, K, bits, 4001 + bits)
    s = I.make_scales(N, K // 128, 4002 + bits)
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), bits)
    g = Guarded((M, N), torch.bfloat16)
    y = wq.wna16_gemm(to_dev_bf16(x), packed, s_dev, N, K, bits, y=g.t)
    g.check(f"split-K y M={M} N={N} K={K}")
    got = y[:, torch.as_tensor(ns, device="cuda")]
    assert_bf16_close(got, O.wna16_ref(x, q[ns], s[ns], bits), f"split-K decode M={M} N={N} K={K} b={bits}")
    wq.check_status()


SPLITK_W4A8 = [(1, 17408, 16384), (8, 17408, 16384), (16, 700, 14336)]


@pytest.mark.parametrize("M,N,K", SPLITK_W4A8)
def test_splitk_decode_w4a8(M, N, K):
    assert wq.debug_route(M, N, K, 4, _sms(), w4a8=True) == "decode_splitk"
    ns = _rows(N, 96, M + N + K + 1)
    x = I.make_x_outliers(M, K, 4100 + M)
    q = I.make_codes(N, K, 4, 4101)
    s = I.make_scales(N, K // 128, 4102)
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), 4)
    g = Guarded((M, N), torch.bfloat16)
    y = wq.w4a8_gemm(to_dev_bf16(x), packed, s_dev, N, K, y=g.t)
    g.check(f"split-K w4a8 y M={M} N={N} K={K}")
    got = y[:, torch.as_tensor(ns, device="cuda")]
    y_ref, _, _ = O.w4a8_ref(x, q[ns], s[ns])
    assert_bf16_close(got, y_ref, f"split-K w4a8 M={M} N={N} K={K}")
    wq.check_status()


@pytest.mark.parametrize("M", [17, 24, 31])
def test_chunked_17_to_31_tokens_full_size(M):
    N, K, bits = 17408, 5120, 6
    assert wq.debug_route(M, N, K, bits, _sms()) == "chunked"
    ns = _rows(N, 96, M)
    x = I.make_x(M, K, 4200 + M)
    q = I.make_codes(N, K, bits, 4201)
    s = I.make_scales(N, K // 128, 4202)
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), bits)
    g = Guarded((M, N), torch.bfloat16)
    y = wq.wna16_gemm(to_dev_bf16(x), packed, s_dev, N, K, bits, y=g.t)
    g.check(f"chunked y M={M}")
    got = y[:, torch.as_tensor(ns, device="cuda")]
    assert_bf16_close(got, O.wna16_ref(x, q[ns], s[ns], bits), f"chunked M={M}")
    wq.check_status()


LONGK_CHUNKED = [
    # (M, N, K, bits, kind): K above 128 groups splits the chunked kernel's
    # CTAs over K (at most 128 groups of scales per CTA)
    (1, 700, 16512, 6, "wna16"),     # not a multiple of 1024
    (24, 5120, 28672, 5, "wna16"),
    (17, 1000, 20480, 7, "wna16"),
    (20, 257, 131072, 2, "wna16"),   # 1024 groups: eight or more splits
    (24, 1536, 28672, 4, "w4a8"),
    (16, 700, 20480, 6, "zp"),
]


@pytest.mark.parametrize("M,N,K,bits,kind", LONGK_CHUNKED)
def test_chunked_kernel_long_k(M, N, K, bits, kind):
    sms = _sms()
    route = wq.debug_route(M, N, K, bits, sms, w4a8=kind == "w4a8", zp=kind == "zp")
    assert route == "chunked", route
    ns = _rows(N, 96, M + N + K + 11)
    x = (I.make_x_outliers if kind == "w4a8" else I.make_x)(M, K, 4400 + M)
    q = I.make_codes(N, K, bits, 4401 + bits)
    s = I.make_scales(N, K // 128, 4402 + bits)
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), bits)
    g = Guarded((M, N), torch.bfloat16)
    if kind == "w4a8":
        y = wq.w4a8_gemm(to_dev_bf16(x), packed, s_dev, N, K, y=g.t)
        y_ref, _, _ = O.w4a8_ref(x, q[ns], s[ns])
    elif kind == "zp":
        zp = np.random.default_rng(4403).integers(0, 1 << bits, size=(N, K // 128)).astype(np.uint8)
        y = wq.wna16_gemm_zp(to_dev_bf16(x), packed, s_dev, to_dev(zp), N, K, bits, y=g.t)
        y_ref = O.wna16_zp_ref(x, q[ns], s[ns], zp[ns], bits)
    else:
        y = wq.wna16_gemm(to_dev_bf16(x), packed, s_dev, N, K, bits, y=g.t)
        y_ref = O.wna16_ref(x, q[ns], s[ns], bits)
    g.check(f"chunked long K y M={M} N={N} K={K}")
    got = y[:, torch.as_tensor(ns, device="cuda")]
    assert_bf16_close(got, y_ref, f"chunked long K M={M} N={N} K={K} b={bits} {kind}")
    wq.check_status()
