"""GPU parity of wna16_moe_gemm, the mixture-of-experts layer in one launch
(model card "Findings", third bullet), against the oracle's moe_ref: ragged
token counts with empty experts, one expert, many experts, every width,
decode-like and prefill-like token counts; outputs between sentinel bands;
and offsets that are out of order or out of range, which the kernel clamps
(no write outside y)."""

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


def _experts(E, N, K, bits, seed):
    q = np.stack([I.make_codes(N, K, bits, seed + e) for e in range(E)])
    s = np.stack([I.make_scales(N, K // 128, seed + 1000 + e) for e in range(E)])
    packed, s_dev = wq.wna16_repack(to_dev(q.reshape(E * N, K)), to_dev_bf16(s.reshape(E * N, K // 128)), bits)
    return q, s, packed, s_dev


CASES = [
    # (counts per expert, N, K, bits)
    ([3, 0, 5, 1], 300, 256, 6),
    ([1], 200, 512, 5),
    ([2, 2, 2, 2, 2, 2, 2, 2], 128, 1024, 7),       # decode-like: 16 tokens over 8 experts
    ([130, 0, 0, 257, 1], 260, 384, 8),
    ([600, 300, 100, 24], 192, 640, 5),              # prefill-like
    ([1, 0, 0, 0, 0, 0, 0, 3] * 8, 136, 256, 6),     # 64 experts, most empty
]


@pytest.mark.parametrize("counts,N,K,bits", CASES)
def test_moe_matches_oracle(counts, N, K, bits):
    E = len(counts)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M = int(off[-1])
    x = I.make_x(M, K, 700 + M)
    q, s, packed, s_dev = _experts(E, N, K, bits, 710 + E)
    g = Guarded((M, N), torch.bfloat16)
    y = wq.wna16_moe_gemm(to_dev_bf16(x), to_dev(off), packed, s_dev, E, N, K, bits, y=g.t)
    g.check(f"moe y E={E} M={M}")
    assert_bf16_close(y, O.moe_ref(x, off, q, s, bits), f"moe E={E} M={M} N={N} K={K} b={bits}")
    wq.check_status()


@pytest.mark.parametrize("bits", range(2, 9))
def test_moe_every_width(bits):
    counts = [5, 40, 0, 17]
    E, N, K = 4, 140, 256
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M = int(off[-1])
    x = I.make_x(M, K, 720 + bits)
    q, s, packed, s_dev = _experts(E, N, K, bits, 730 + bits)
    y = wq.wna16_moe_gemm(to_dev_bf16(x), to_dev(off), packed, s_dev, E, N, K, bits)
    assert_bf16_close(y, O.moe_ref(x, off, q, s, bits), f"moe b={bits}")


def test_moe_full_size_sampled():
    """Eight experts of 2048 x 5120 (6-bit) over 4096 tokens with a skewed
    split; sampled tokens and rows of every expert."""
    E, N, K, bits = 8, 2048, 5120, 6
    counts = [1024, 512, 0, 1536, 256, 255, 1, 512]
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M = int(off[-1])
    x = I.make_x(M, K, 740)
    q, s, packed, s_dev = _experts(E, N, K, bits, 750)
    y = wq.wna16_moe_gemm(to_dev_bf16(x), to_dev(off), packed, s_dev, E, N, K, bits)
    torch.cuda.synchronize()
    r = np.random.default_rng(3)
    ns = np.unique(np.concatenate([r.choice(N, 24, replace=False), [0, N - 1]]))
    for e in range(E):
        if counts[e] == 0:
            continue
        ms = np.unique(np.concatenate([r.choice(np.arange(off[e], off[e + 1]), min(6, counts[e]), replace=False),
                                       [off[e], off[e + 1] - 1]]))
        got = y[torch.as_tensor(ms, device="cuda")][:, torch.as_tensor(ns, device="cuda")]
        assert_bf16_close(got, O.wna16_ref(x[ms], q[e][ns], s[e][ns], bits), f"moe full size expert {e}")
    wq.check_status()


def test_moe_offsets_out_of_order_or_range_stay_inside_y():
    """The kernel clamps each offset into [0, M] and to at least the previous
    one: whatever the offsets, it reads and writes nothing outside x and y."""
    E, N, K, bits = 4, 130, 256, 5
    M = 40
    x = I.make_x(M, K, 760)
    _, _, packed, s_dev = _experts(E, N, K, bits, 770)
    for off in ([5, 2, 100000, -3, 7], [-8, 50, 10, 30, 40], [0, 0, 0, 0, 0], [40, 40, 40, 40, 1 << 30]):
        g = Guarded((M, N), torch.bfloat16)
        wq.wna16_moe_gemm(to_dev_bf16(x), to_dev(np.array(off, dtype=np.int32)), packed, s_dev, E, N, K, bits,
                          y=g.t)
        g.check(f"moe offsets {off}")
    wq.check_status()
