"""The allocation-free entry point, wna16_gemm_noalloc, called through the C
ABI: for callers that cannot allocate device memory (for example a serving
engine whose memory is all reserved for its KV-cache pool), the split-K
scratch lives in a fixed array owned by the library. Its output must match the
regular wna16_gemm (which takes a caller workspace) within the acceptance
tolerance, on two calls in a row, since every call shares that array.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process."""

import ctypes

import numpy as np
import pytest

import oracle as O
import wq_inputs as I
from helpers import assert_bf16_close, bf16_dev_to_f64, errors, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import weight_only_int2_gb300 as wq  # noqa: E402


def _call_noalloc(lib, x, packed, s_dev, N, K, bits, y):
    st = lib.wna16_gemm_noalloc(ctypes.c_void_p(x.data_ptr()), x.shape[0], ctypes.c_void_p(packed.data_ptr()),
                                ctypes.c_void_p(s_dev.data_ptr()), N, K, bits, 128,
                                ctypes.c_void_p(y.data_ptr()),
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.wq_last_error().decode()


# (M, N, K, bits, uses_scratch): the pair-kernel shapes need no scratch; the
# split-K shapes do, the first near the 4 MiB cap (3,842,048 bytes).
CASES = [(16, 60000, 2560, 8, True), (4, 1000, 2560, 6, True), (3, 300, 640, 8, True),
         (4, 1000, 5120, 6, False), (1, 17408, 5120, 5, False), (16, 700, 2048, 7, False)]


@pytest.mark.parametrize("M,N,K,bits,uses_scratch", CASES)
def test_noalloc_matches_workspace_entry_point_twice(M, N, K, bits, uses_scratch):
    lib = wq.load()
    need = lib.wna16_workspace_bytes(M, N, K, bits)
    # a routing change must not quietly turn a scratch case into pair-kernel coverage
    assert (need > 0) == uses_scratch and need <= (4 << 20), need
    x = I.make_x(M, K, 500 + M)
    q = I.make_codes(N, K, bits, 501)
    s = I.make_scales(N, K // 128, 502)
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), bits)
    xd = to_dev_bf16(x)
    y_ref = wq.wna16_gemm(xd, packed, s_dev, N, K, bits)       # existing entry point
    ref64 = bf16_dev_to_f64(y_ref)
    for _ in range(2):                                         # two calls in a row
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        _call_noalloc(lib, xd, packed, s_dev, N, K, bits, y)
        torch.cuda.synchronize()
        fro, mx = errors(bf16_dev_to_f64(y), ref64)
        assert fro <= 5e-3 and mx <= 1e-2, (fro, mx)
        assert_bf16_close(y, O.wna16_ref(x, q, s, bits), "noalloc vs oracle")
    wq.check_status()


def _problem(M, N, K, bits, seed):
    x = I.make_x(M, K, seed)
    q = I.make_codes(N, K, bits, seed + 1)
    s = I.make_scales(N, K // 128, seed + 2)
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), bits)
    return x, q, s, to_dev_bf16(x), packed, s_dev


def test_two_split_k_shapes_back_to_back():
    """Two different split-K shapes share the array in one stream, twice over:
    each call must clear what the previous one left."""
    lib = wq.load()
    shapes = [(16, 60000, 2560, 8, 900), (4, 1000, 2560, 6, 910)]
    probs = [_problem(M, N, K, b, sd) for (M, N, K, b, sd) in shapes]
    for M, N, K, b, _ in shapes:
        assert lib.wna16_workspace_bytes(M, N, K, b) > 0
    refs = [O.wna16_ref(x, q, s, b) for (x, q, s, _, _, _), (_, _, _, b, _) in zip(probs, shapes)]
    for _ in range(2):
        ys = []
        for (M, N, K, b, _), (_, _, _, xd, packed, s_dev) in zip(shapes, probs):
            y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
            _call_noalloc(lib, xd, packed, s_dev, N, K, b, y)
            ys.append(y)
        torch.cuda.synchronize()
        for y, ref in zip(ys, refs):
            assert_bf16_close(y, ref, "back-to-back split-K shapes")
    wq.check_status()


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = wq.load()
    M, N, K = 16, 248320, 2560                                  # split-K shape: ~16 MB of scratch
    assert lib.wna16_workspace_bytes(M, N, K, 8) > (4 << 20)
    # real device buffers of the right sizes: the call is refused before any
    # launch, and a regression that launched would still touch valid memory
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((N, K * 8 // 32), dtype=torch.int32, device="cuda")
    s = torch.zeros((N, K // 128), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    st = lib.wna16_gemm_noalloc(ctypes.c_void_p(x.data_ptr()), M, ctypes.c_void_p(w.data_ptr()),
                                ctypes.c_void_p(s.data_ptr()), N, K, 8, 128, ctypes.c_void_p(y.data_ptr()), None)
    assert st == 1
    assert b"scratch" in lib.wq_last_error()


def test_bad_arguments_leave_the_scratch_untouched():
    """Argument checks come before anything is enqueued: a call with bad bits
    or a NULL pointer on a shape that uses the scratch returns WQ_EINVAL and
    leaves a sentinel planted in the array as it was."""
    lib = wq.load()
    M, N, K, bits = 4, 1000, 2560, 6
    need = lib.wna16_workspace_bytes(M, N, K, bits)
    assert 0 < need <= (4 << 20)
    x, q, s, xd, packed, s_dev = _problem(M, N, K, bits, 920)
    y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    sentinel = torch.arange(need, dtype=torch.int64, device="cuda").remainder(251).to(torch.uint8) + 3
    assert lib.wq_debug_noalloc_scratch(ctypes.c_void_p(sentinel.data_ptr()), need, 1, stream) == 0
    P = ctypes.c_void_p
    st = lib.wna16_gemm_noalloc(P(xd.data_ptr()), M, P(packed.data_ptr()), P(s_dev.data_ptr()), N, K, 9, 128,
                                P(y.data_ptr()), stream)
    assert st == 1 and b"bits" in lib.wq_last_error()
    st = lib.wna16_gemm_noalloc(P(xd.data_ptr()), M, None, P(s_dev.data_ptr()), N, K, bits, 128,
                                P(y.data_ptr()), stream)
    assert st == 1 and b"NULL" in lib.wq_last_error()
    back = torch.zeros(need, dtype=torch.uint8, device="cuda")
    assert lib.wq_debug_noalloc_scratch(ctypes.c_void_p(back.data_ptr()), need, 0, stream) == 0
    torch.cuda.synchronize()
    assert torch.equal(back, sentinel)
    # a valid call on the sentinel-filled array clears what it uses and is correct
    _call_noalloc(lib, xd, packed, s_dev, N, K, bits, y)
    torch.cuda.synchronize()
    assert_bf16_close(y, O.wna16_ref(x, q, s, bits), "after the sentinel")
    wq.check_status()


def test_tensor_core_shapes_need_no_scratch():
    """64 tokens on a 17408-row layer run on the tensor-core kernel, which
    needs no workspace: wna16_gemm accepts a NULL workspace and the
    allocation-free entry point accepts the shape although the workspace
    query (an upper bound) exceeds its 4 MiB array. Same kernel, same bits."""
    lib = wq.load()
    M, N, K, bits = 64, 17408, 5120, 6
    assert torch.cuda.get_device_properties(0).multi_processor_count <= 2 * ((N + 127) // 128)
    assert lib.wna16_workspace_bytes(M, N, K, bits) > (4 << 20)
    x = I.make_x(M, K, 510)
    q = I.make_codes(N, K, bits, 511)
    s = I.make_scales(N, K // 128, 512)
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), bits)
    xd = to_dev_bf16(x)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    y_ws = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = lib.wna16_gemm(ctypes.c_void_p(xd.data_ptr()), M, ctypes.c_void_p(packed.data_ptr()),
                        ctypes.c_void_p(s_dev.data_ptr()), N, K, bits, 128, ctypes.c_void_p(y_ws.data_ptr()),
                        None, 0, stream)
    assert st == 0, lib.wq_last_error().decode()
    y_na = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    _call_noalloc(lib, xd, packed, s_dev, N, K, bits, y_na)
    torch.cuda.synchronize()
    assert torch.equal(y_ws.view(torch.int16), y_na.view(torch.int16))
    ms = np.array([0, 17, 63])
    ns = np.array([0, 5000, N - 1])
    got = y_ws[torch.as_tensor(ms, device="cuda")][:, torch.as_tensor(ns, device="cuda")]
    assert_bf16_close(got, O.wna16_ref(x[ms], q[ns], s[ns], bits), "tensor-core route, no workspace")
    wq.check_status()
