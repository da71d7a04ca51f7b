"""GPU parity of the tensor-core (many-token) GEMM path against the oracle.

Shapes span several 128-row weight tiles and token tiles (128 and 256
tokens) with ragged tails in M and N, K from one group to 40 groups, every
code width, both scale signs, and the W4A8 variant. The full-size case
(8192 x 17408 x 5120, the prefill configuration) is checked on sampled
outputs that the oracle computes one by one."""

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


def _layer(N, K, bits, seed, sign="random"):
    q = I.make_codes(N, K, bits, seed)
    s = I.make_scales(N, K // 128, seed + 1, sign=sign)
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), bits)
    return q, s, packed, s_dev


PREFILL_CASES = [
    # (M, N, K, bits)
    (65, 128, 128, 6),       # smallest token count on this path, one group
    (128, 384, 1024, 7),     # exact 128-token tile, three row tiles
    (129, 130, 256, 2),      # first 256-token tile, ragged rows
    (256, 256, 2048, 8),
    (300, 257, 768, 3),
    (513, 640, 512, 4),
    (777, 1000, 1280, 5),
    (1024, 512, 5120, 6),    # four token tiles, 40 groups
    (300, 2112, 384, 6),     # 17 row tiles, last one ragged
    (4133, 2624, 256, 5),    # 357 tiles: several per CTA of the persistent grid
]


@pytest.mark.parametrize("M,N,K,bits", PREFILL_CASES)
def test_prefill_matches_oracle(M, N, K, bits):
    seed = 7 * M + N + bits
    x = I.make_x(M, K, seed)
    q, s, packed, s_dev = _layer(N, K, bits, seed + 5)
    g = Guarded((M, N), torch.bfloat16)
    y = wq.wna16_gemm(to_dev_bf16(x), packed, s_dev, N, K, bits, y=g.t)
    g.check(f"y M={M} N={N} K={K} b={bits}")
    assert_bf16_close(y, O.wna16_ref(x, q, s, bits), f"M={M} N={N} K={K} b={bits}")


@pytest.mark.parametrize("bits", range(2, 9))
def test_prefill_every_width(bits):
    M, N, K = 257, 200, 640
    x = I.make_x(M, K, 40 + bits)
    q, s, packed, s_dev = _layer(N, K, bits, 50 + bits)
    y = wq.wna16_gemm(to_dev_bf16(x), packed, s_dev, N, K, bits)
    assert_bf16_close(y, O.wna16_ref(x, q, s, bits), f"b={bits}")


@pytest.mark.parametrize("bits", [5, 6, 7, 8])
def test_prefill_negative_scales_and_extreme_codes(bits):
    M, N, K = 200, 150, 512
    x = I.make_x(M, K, 3)
    q, s, packed, s_dev = _layer(N, K, bits, 4, sign="negative")
    y = wq.wna16_gemm(to_dev_bf16(x), packed, s_dev, N, K, bits)
    assert_bf16_close(y, O.wna16_ref(x, q, s, bits), "negative scales")
    for c in (0, (1 << bits) - 1):
        qc = np.full((N, K), c, dtype=np.uint8)
        pc, _ = wq.wna16_repack(to_dev(qc), s_dev, bits)
        yc = wq.wna16_gemm(to_dev_bf16(x), pc, s_dev, N, K, bits)
        assert_bf16_close(yc, O.wna16_ref(x, qc, s, bits), f"constant code {c}")
    # codes at the zero point dequantize to (signed) zero: the output is zero
    qz = np.full((N, K), 1 << (bits - 1), dtype=np.uint8)
    pz, _ = wq.wna16_repack(to_dev(qz), s_dev, bits)
    yz = wq.wna16_gemm(to_dev_bf16(x), pz, s_dev, N, K, bits).float()
    assert float(yz.abs().max()) == 0.0


def test_prefill_needs_no_workspace():
    assert wq.wna16_workspace_bytes(4096, 17408, 5120, 6) == 0
    assert wq.wna16_workspace_bytes(65, 100, 256, 6) == 0


@pytest.mark.parametrize("M,N,K,sign", [(100, 64, 256, "random"), (300, 257, 1024, "negative"),
                                        (512, 640, 5120, "random")])
def test_w4a8_prefill_matches_oracle(M, N, K, sign):
    x = I.make_x_outliers(M, K, 90 + M)
    q, s, packed, s_dev = _layer(N, K, 4, 91 + M, sign=sign)
    g = Guarded((M, N), torch.bfloat16)
    y = wq.w4a8_gemm(to_dev_bf16(x), packed, s_dev, N, K, y=g.t)
    g.check(f"w4a8 y M={M}")
    y_ref, _, _ = O.w4a8_ref(x, q, s)
    assert_bf16_close(y, y_ref, f"w4a8 prefill M={M}")


@pytest.mark.parametrize("M,bits", [(8192, 5), (8192, 6), (8192, 7), (8192, 8), (2048, 5), (2048, 6),
                                    (2048, 7), (2048, 8)])
def test_prefill_full_size_sampled(M, bits):
    """N=17408, K=5120 at every width and both token counts of the prefill
    configuration. The oracle computes 48 token rows x 48 weight rows drawn
    over the whole output."""
    N, K = 17408, 5120
    x = I.make_x(M, K, 8192 + M)
    q = I.make_codes(N, K, bits, 8193 + bits)
    s = I.make_scales(N, K // 128, 8194 + bits)
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), bits)
    g = Guarded((M, N), torch.bfloat16)
    y = wq.wna16_gemm(to_dev_bf16(x), packed, s_dev, N, K, bits, y=g.t)
    g.check(f"full-size y M={M} b={bits}")
    r = np.random.default_rng(5 + bits)
    ms = np.unique(np.concatenate([r.choice(M, 46, replace=False), [0, M - 1]]))
    ns = np.unique(np.concatenate([r.choice(N, 46, replace=False), [0, N - 1]]))
    got = y[torch.as_tensor(ms, device="cuda")][:, torch.as_tensor(ns, device="cuda")]
    ref = O.wna16_ref(x[ms], q[ns], s[ns], bits)
    assert_bf16_close(got, ref, f"full-size sampled M={M} b={bits}")
