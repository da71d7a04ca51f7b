"""The library reuses encoded TMA descriptors across calls (a table keyed on
every encoding argument, the address included). These cases make sure that
reuse never changes a result: the same weight buffer read with different
shapes (distinct descriptors), new contents repacked into the same buffers
(the same descriptor), and more distinct layers than the table holds
(evictions)."""

import numpy as np
import pytest

import oracle as O
import wq_inputs as I
from helpers import assert_bf16_close, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import weight_only_int2_gb300 as wq  # noqa: E402

K = 2048


def _layer(N, bits, seed):
    q = I.make_codes(N, K, bits, seed)
    s = I.make_scales(N, K // 128, seed + 1)
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), bits)
    return q, s, packed, s_dev


def test_same_buffer_with_fewer_rows():
    """Rows 0..n-1 of a packed layer are a layer of n rows at the same
    address: each row count gets its own descriptor."""
    bits, N = 6, 1024
    q, s, packed, s_dev = _layer(N, bits, 7100)
    x = I.make_x(4, K, 7102)
    for n in (N, 512, 300, N):
        y = wq.wna16_gemm(to_dev_bf16(x), packed[:n], s_dev[:n], n, K, bits)
        torch.cuda.synchronize()
        assert_bf16_close(y, O.wna16_ref(x, q[:n], s[:n], bits), f"first {n} rows")
    wq.check_status()


def test_new_contents_at_the_same_address():
    """A second layer repacked into the very buffers of the first (same
    address, same shape, so the same descriptor): the call reads the new
    contents."""
    bits, N = 5, 768
    x = I.make_x(2, K, 7200)
    q1, s1, p1, sd1 = _layer(N, bits, 7201)
    y1 = wq.wna16_gemm(to_dev_bf16(x), p1, sd1, N, K, bits)
    torch.cuda.synchronize()
    assert_bf16_close(y1, O.wna16_ref(x, q1, s1, bits), "first layer")
    addr = (p1.data_ptr(), sd1.data_ptr())
    q2 = I.make_codes(N, K, bits, 7301)
    s2 = I.make_scales(N, K // 128, 7302)
    p2, sd2 = wq.wna16_repack(to_dev(q2), to_dev_bf16(s2), bits, packed=p1, scales_out=sd1)
    assert (p2.data_ptr(), sd2.data_ptr()) == addr
    y2 = wq.wna16_gemm(to_dev_bf16(x), p2, sd2, N, K, bits)
    torch.cuda.synchronize()
    assert_bf16_close(y2, O.wna16_ref(x, q2, s2, bits), "second layer, same buffers")
    wq.check_status()


def test_more_layers_than_the_table_holds():
    """300 distinct small layers (600 descriptors, more than the 256-entry
    table), then the first ones again: evicted entries are encoded anew."""
    bits, N = 7, 128
    rng = np.random.default_rng(7400)
    layers = []
    for i in range(300):
        q = rng.integers(0, 1 << bits, size=(N, K), dtype=np.uint8)
        s = I.make_scales(N, K // 128, 7401 + i)
        packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), bits)
        layers.append((q, s, packed, s_dev))
    x = I.make_x(1, K, 7399)
    xd = to_dev_bf16(x)
    ys = [wq.wna16_gemm(xd, p, sd, N, K, bits) for (_, _, p, sd) in layers]
    ys += [wq.wna16_gemm(xd, p, sd, N, K, bits) for (_, _, p, sd) in layers[:20]]
    torch.cuda.synchronize()
    for i in list(range(0, 300, 37)) + [299]:
        q, s, _, _ = layers[i]
        assert_bf16_close(ys[i], O.wna16_ref(x, q, s, bits), f"layer {i}")
    for i in range(20):
        assert torch.equal(ys[300 + i].view(torch.int16), ys[i].view(torch.int16))
    wq.check_status()
