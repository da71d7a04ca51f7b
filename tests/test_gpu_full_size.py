"""GPU parity at the full sizes of the benchmark configurations, on sampled
outputs that the oracle computes one by one (sampling output rows and tokens is
exact: every output element depends only on its own weight row and token).

Covered: the decode sweep (bits 5/6/7 x N 5120/17408 x M 1/4/16/32/64), the 8-bit
lm_head (N = 248320, M = 1 and 4096), the quantized-embedding gather of 4096
ids from the 248320-row table (bit-exact), W4A8 at M = 1 / 16 / 32 / 512 / 8192, and the
64-layer mixed-bit stack (also replayed as one CUDA graph, which must give the
same bits as eager execution)."""

import numpy as np
import pytest

import oracle as O
import wq_inputs as I
from helpers import assert_bf16_close, bf16_dev_to_bits, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import weight_only_int2_gb300 as wq  # noqa: E402

K = 5120


def _sample(n, k, seed, must=()):
    r = np.random.default_rng(seed)
    pick = r.choice(n, min(k, n), replace=False)
    return np.unique(np.concatenate([pick, np.asarray(must, dtype=np.int64)]).astype(np.int64))


def _check_sampled(y_dev, x, q, s, bits, ms, ns, what):
    got = y_dev[torch.as_tensor(ms, device="cuda")][:, torch.as_tensor(ns, device="cuda")]
    ref = O.wna16_ref(x[ms], q[ns], s[ns], bits)
    assert_bf16_close(got, ref, what)


@pytest.mark.parametrize("bits", [5, 6, 7])
@pytest.mark.parametrize("N", [5120, 17408])
def test_decode_sweep_full_size(bits, N):
    q = I.make_codes(N, K, bits, 1000 + bits)
    s = I.make_scales(N, K // 128, 1100 + bits)
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), bits)
    ns = _sample(N, 64, bits + N, must=[0, N - 1])
    for M in (1, 4, 16, 32, 64):
        x = I.make_x(M, K, 1200 + M)
        y = wq.wna16_gemm(to_dev_bf16(x), packed, s_dev, N, K, bits)
        torch.cuda.synchronize()
        _check_sampled(y, x, q, s, bits, np.arange(M), ns, f"decode b={bits} N={N} M={M}")
    wq.check_status()


@pytest.fixture(scope="module")
def vocab_table():
    """The 8-bit 248320 x 5120 table (lm_head and embedding), repacked once."""
    V = 248320
    q = I.make_codes(V, K, 8, 2000)
    s = I.make_scales(V, K // 128, 2001)
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), 8)
    torch.cuda.synchronize()
    return V, q, s, packed, s_dev


@pytest.mark.parametrize("M", [1, 4096])
def test_lm_head_full_size(vocab_table, M):
    V, q, s, packed, s_dev = vocab_table
    x = I.make_x(M, K, 2100 + M)
    y = wq.wna16_gemm(to_dev_bf16(x), packed, s_dev, V, K, 8)
    torch.cuda.synchronize()
    ms = _sample(M, 24, 7, must=[0, M - 1])
    ns = _sample(V, 64, 8, must=[0, V - 1])
    _check_sampled(y, x, q, s, 8, ms, ns, f"lm_head M={M}")


def test_gather_full_size(vocab_table):
    V, q, s, packed, s_dev = vocab_table
    T = 4096
    ids = I.make_ids(T, V, 2200)
    out = wq.qembed_gather(to_dev(ids), packed, s_dev, V, K, 8)
    torch.cuda.synchronize()
    ts = _sample(T, 256, 9, must=[0, T - 1])
    ref, nbad = O.qembed_ref(ids[ts], q, s, 8)
    assert nbad == 0
    got = bf16_dev_to_bits(out[torch.as_tensor(ts, device="cuda")])
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("M", [1, 16, 32, 512, 8192])
def test_w4a8_full_size(M):
    N = 17408
    q = I.make_codes(N, K, 4, 2300)
    s = I.make_scales(N, K // 128, 2301)
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), 4)
    x = I.make_x_outliers(M, K, 2302 + M)
    y = wq.w4a8_gemm(to_dev_bf16(x), packed, s_dev, N, K)
    torch.cuda.synchronize()
    ms = _sample(M, 24, 10, must=[0, M - 1])
    ns = _sample(N, 64, 11, must=[0, N - 1])
    got = y[torch.as_tensor(ms, device="cuda")][:, torch.as_tensor(ns, device="cuda")]
    y_ref, _, _ = O.w4a8_ref(x[ms], q[ns], s[ns])
    assert_bf16_close(got, y_ref, f"w4a8 M={M}")


def test_w4a8_group_accumulators_full_size_sampled():
    """The exact int32 group accumulators at the full W4A8 prefill size
    (8192 x 17408 x 5120, the tensor-core route), sampled: every entry
    acc[m, n, g] depends only on token m and weight row n."""
    M, N = 8192, 17408
    G = K // 128
    assert wq.debug_route(M, N, K, 4, torch.cuda.get_device_properties(0).multi_processor_count,
                          w4a8=True) == "tensor_core"
    q = I.make_codes(N, K, 4, 2400)
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(I.make_scales(N, G, 2401)), 4)
    x = I.make_x_outliers(M, K, 2402)
    acc = wq.debug_w4a8_group_acc(to_dev_bf16(x), packed, s_dev, N, K)   # 22.8 GB of int32
    torch.cuda.synchronize()
    ms = _sample(M, 24, 12, must=[0, M - 1])
    ns = _sample(N, 64, 13, must=[0, N - 1])
    got = acc[torch.as_tensor(ms, device="cuda")][:, torch.as_tensor(ns, device="cuda")].cpu().numpy()
    del acc
    xq_ref, _ = O.act_quant_ref(x[ms])                                   # per token: rows are independent
    assert np.array_equal(got.astype(np.int64), O.w4a8_group_acc(xq_ref, q[ns]))
    wq.check_status()


def _stack_bits(layer):
    """Layers 0-9 and 54-63: 7 bits; 10-53 alternate 5 / 6, starting with 5."""
    if layer < 10 or layer >= 54:
        return 7
    return 5 if (layer - 10) % 2 == 0 else 6


def test_mixed_stack_full_size():
    N, L = 17408, 64
    layers = []
    for li in range(L):
        bits = _stack_bits(li)
        q = I.make_codes(N, K, bits, 3000 + li)
        s = I.make_scales(N, K // 128, 3100 + li)
        packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), bits)
        ns = _sample(N, 16, li, must=[li, N - 1 - li])
        layers.append((bits, packed, s_dev, q[ns], s[ns], ns))
        del q
    for M in (1, 4096):
        x = I.make_x(M, K, 3200 + M)
        xd = to_dev_bf16(x)
        ms = _sample(M, 8, M, must=[0, M - 1])
        ys = [torch.empty(M, N, dtype=torch.bfloat16, device="cuda") for _ in range(L)]
        for li, (bits, packed, s_dev, qs, ss, ns) in enumerate(layers):
            wq.wna16_gemm(xd, packed, s_dev, N, K, bits, y=ys[li])
        torch.cuda.synchronize()
        eager = [y.clone() for y in ys]
        for li, (bits, packed, s_dev, qs, ss, ns) in enumerate(layers):
            got = ys[li][torch.as_tensor(ms, device="cuda")][:, torch.as_tensor(ns, device="cuda")]
            assert_bf16_close(got, O.wna16_ref(x[ms], qs, ss, bits), f"stack layer {li} M={M}")
        # the same 64 layers as one CUDA graph: identical bits
        st = torch.cuda.Stream()
        with torch.cuda.stream(st):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                for li, (bits, packed, s_dev, _, _, _) in enumerate(layers):
                    wq.wna16_gemm(xd, packed, s_dev, N, K, bits, y=ys[li])
            for y in ys:
                y.zero_()
            g.replay()
            st.synchronize()
        for li in range(L):
            same = torch.equal(ys[li].view(torch.int16), eager[li].view(torch.int16))
            assert same, f"graph replay differs at layer {li} M={M}"
        del ys, eager
    wq.check_status()


@pytest.mark.parametrize("bits,N,M", [(5, 17408, 1), (6, 17408, 1), (7, 17408, 16), (6, 5120, 4), (8, 248320, 1)])
def test_decode_repeatable(bits, N, M):
    """A hundred launches of the same decode GEMM give the same bits (every
    output is reduced in a fixed order, so any difference is a race; the
    multi-chunk lm_head shape once showed a ring-slot race in about one
    launch in ten)."""
    codes = torch.randint(0, 1 << bits, (N, K), dtype=torch.uint8, device="cuda",
                          generator=torch.Generator(device="cuda").manual_seed(bits * N + M))
    scales = (torch.randn(N, K // 128, device="cuda") * 0.01).to(torch.bfloat16)
    packed, s_dev = wq.wna16_repack(codes, scales, bits)
    del codes
    x = torch.randn(M, K, device="cuda").to(torch.bfloat16)
    first = wq.wna16_gemm(x, packed, s_dev, N, K, bits).view(torch.int16).clone()
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    for rep in range(100):
        wq.wna16_gemm(x, packed, s_dev, N, K, bits, y=y)
        assert torch.equal(y.view(torch.int16), first), f"launch {rep} differs"
    wq.check_status()
