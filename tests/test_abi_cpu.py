"""CPU checks of the C ABI surface: the library loads, exports every symbol
declared in include/wq.h, answers the host-only size queries, and rejects bad
arguments before touching any GPU."""

import ctypes
import os
import re

import pytest

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wq.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)
    skip = {"if", "sizeof", "defined"}
    return sorted({n for n in names if n not in skip})


@pytest.fixture(scope="module")
def lib():
    import weight_only_int2_gb300 as wq

    if not os.path.exists(wq.LIB_PATH):
        import __graft_entry__

        __graft_entry__.build()
    return wq.load()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ["wna16_repack", "wna16_gemm", "w4a8_gemm", "qembed_gather", "act_quant_int8",
              "wq_packed_words_per_row", "wq_check_status", "wq_last_error"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in _declared_functions():
        assert hasattr(lib, n), n


def test_binding_covers_every_declared_symbol():
    from weight_only_int2_gb300._lib import SIGNATURES

    assert sorted(SIGNATURES) == _declared_functions()


@pytest.mark.parametrize("bits", range(2, 9))
@pytest.mark.parametrize("K", [128, 5120, 248320])
def test_packed_words_match_oracle(lib, bits, K):
    assert lib.wq_packed_words_per_row(K, bits) == O.packed_words_per_row(K, bits)


def test_workspace_sizes(lib):
    # CTA-pair decode (M <= 16, K % 1024 == 0) and the tensor-core GEMM need
    # none; the split-K streaming kernels need fp32 partials
    assert lib.wna16_workspace_bytes(1, 17408, 5120, 6) == 0
    assert lib.wna16_workspace_bytes(16, 17408, 5120, 6) == 0
    assert lib.wna16_workspace_bytes(4, 1000, 2560, 6) >= 4 * 1000 * 4
    assert lib.wna16_workspace_bytes(32, 1000, 5120, 6) >= 32 * 1000 * 4
    assert lib.wna16_workspace_bytes(4096, 17408, 5120, 6) == 0
    assert lib.w4a8_workspace_bytes(8, 100, 256) >= 8 * 100 * 4
    assert lib.w4a8_scratch_bytes(8, 256) >= 8 * 256 + 8 * 4


@pytest.fixture(scope="module")
def fake():
    """A pointer that the checks below never let a kernel use. Without a GPU
    it is a plain address (no CUDA call can touch it); where a GPU is present
    it is a real 64 MiB device buffer, so that a regression that launched a
    kernel would still touch valid memory of the right sizes."""
    try:
        import torch

        if torch.cuda.is_available():
            buf = torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")
            yield ctypes.c_void_p(buf.data_ptr())
            torch.cuda.synchronize()
            return
    except ImportError:  # pragma: no cover
        pass
    yield ctypes.c_void_p(1 << 20)


def test_bad_arguments_rejected_before_any_cuda_call(lib, fake):
    addr = fake.value
    # bits out of range
    assert lib.wna16_gemm(fake, 1, fake, fake, 8, 128, 9, 128, fake, None, 0, None) == 1
    assert b"bits" in lib.wq_last_error()
    # group other than 128
    assert lib.wna16_gemm(fake, 1, fake, fake, 8, 128, 6, 64, fake, None, 0, None) == 2
    # K not a multiple of 128
    assert lib.wna16_repack(fake, fake, 4, 100, 6, 128, fake, fake, None, None) == 1
    # null pointers and misalignment
    assert lib.wna16_gemm(None, 1, fake, fake, 8, 128, 6, 128, fake, None, 0, None) == 1
    assert lib.wna16_gemm(ctypes.c_void_p(addr + 2), 1, fake, fake, 8, 128, 6, 128, fake, None, 0,
                          None) == 1
    assert b"aligned" in lib.wq_last_error()
    # M = 0
    assert lib.wna16_gemm(fake, 0, fake, fake, 8, 128, 6, 128, fake, None, 0, None) == 1
    # the mma.sync probe: kind, iteration and block bounds, NULL output
    assert lib.wq_debug_mma_peak(2, 10, 1, fake, None) == 1
    assert lib.wq_debug_mma_peak(0, 0, 1, fake, None) == 1
    assert lib.wq_debug_mma_peak(1, 1000001, 1, fake, None) == 1
    assert lib.wq_debug_mma_peak(0, 10, 0, fake, None) == 1
    assert lib.wq_debug_mma_peak(0, 10, 1, None, None) == 1
    assert b"wq_debug_mma_peak" in lib.wq_last_error()
    # workspace too small for a split-K decode shape
    assert lib.wna16_workspace_bytes(1, 5120, 2560, 6) > 16  # else the call below would launch
    assert lib.wna16_gemm(fake, 1, fake, fake, 5120, 2560, 6, 128, fake, fake, 16, None) == 1
    assert b"workspace" in lib.wq_last_error()
    # a decode-sized call whose K half does not fit the pair kernel's shared
    # memory streams through the split-K kernel: the query says so, and a
    # missing workspace is refused
    assert lib.wna16_workspace_bytes(1, 8, 65536, 2) > 0
    assert lib.wna16_gemm(fake, 1, fake, fake, 8, 65536, 2, 128, fake, None, 0, None) == 1
    assert b"workspace is NULL" in lib.wq_last_error()
    # sizes at or above 2^31 (grid dimensions, 32-bit TMA coordinates)
    big = 1 << 31
    assert lib.wna16_gemm(fake, big, fake, fake, 8, 128, 6, 128, fake, None, 0, None) == 1
    assert lib.wna16_gemm(fake, 1, fake, fake, big, 128, 6, 128, fake, None, 0, None) == 1
    assert lib.wna16_gemm(fake, 1, fake, fake, 8, big, 6, 128, fake, None, 0, None) == 1
    assert lib.act_quant_int8(fake, big, 128, fake, fake, None) == 1
    assert lib.qembed_gather(fake, big, fake, fake, 10, 128, 8, 128, fake, None, None) == 1
    assert lib.qembed_gather(fake, 4, fake, fake, big, 128, 8, 128, fake, None, None) == 1
    assert lib.wna16_repack(fake, fake, big, 128, 6, 128, fake, fake, None, None) == 1
    assert b"2^31" in lib.wq_last_error()
    # gather: T = 0 is a no-op that needs no GPU
    assert lib.qembed_gather(None, 0, fake, fake, 10, 128, 8, 128, fake, None, None) == 0


def test_header_is_plain_c(tmp_path):
    """include/wq.h is usable from C (not only C++): it compiles as C11 with
    warnings as errors, and every entry point is callable through a pointer
    of the declared type."""
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_wq.c"
    src.write_text('#include "wq.h"\n'
                   "int main(void) {\n"
                   "  wq_status (*g)(const wq_bf16*, int64_t, const uint32_t*, const wq_bf16*, int64_t, int64_t,\n"
                   "                 int, int, wq_bf16*, void*, size_t, void*) = wna16_gemm;\n"
                   "  size_t (*w)(int64_t, int) = wq_packed_words_per_row;\n"
                   "  return (g != 0 && w != 0) ? 0 : 1;\n"
                   "}\n")
    r = subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I",
                        os.path.join(ROOT, "include"), "-c", str(src), "-o", str(tmp_path / "use_wq.o")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_missing_library_fails_loudly(tmp_path):
    """There is no fallback path: without libwq.so the binding refuses to load."""
    import subprocess
    import sys

    code = ("import weight_only_int2_gb300._lib as L\n"
            "try:\n"
            "    L.load(%r)\n"
            "except RuntimeError as e:\n"
            "    print('refused:', e)\n" % str(tmp_path / "libwq.so"))
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert "refused: libwq.so not found" in r.stdout


def test_host_tensors_are_refused(lib):
    """The entry points take device tensors only; host tensors raise before
    any work instead of being computed somewhere else."""
    import torch

    import weight_only_int2_gb300 as wq

    bits, N, K = 6, 8, 128
    x = torch.zeros(1, K, dtype=torch.bfloat16)
    packed = torch.zeros(N, wq.packed_words_per_row(K, bits), dtype=torch.int32)
    scales = torch.zeros(N, K // 128, dtype=torch.bfloat16)
    codes = torch.zeros(N, K, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA tensor"):
        wq.wna16_gemm(x, packed, scales, N, K, bits)
    with pytest.raises(ValueError, match="CUDA tensor"):
        wq.wna16_repack(codes, scales, bits)
    with pytest.raises(ValueError, match="CUDA tensor"):
        wq.act_quant_int8(x)
    with pytest.raises(ValueError, match="CUDA tensor"):
        wq.w4a8_gemm(x, torch.zeros(N, wq.packed_words_per_row(K, 4), dtype=torch.int32), scales, N, K)
    with pytest.raises(ValueError, match="CUDA tensor"):
        wq.qembed_gather(torch.zeros(2, dtype=torch.int32), packed, scales, N, K, bits)


def test_device_failure_drops_cached_workspaces(lib):
    """A call that failed on the device (launch error, or a timeout read by
    check_status) may leave partial sums in a zero-at-rest workspace: the
    binding forgets its cached buffers then. Argument errors launch nothing
    and keep them."""
    from weight_only_int2_gb300 import _lib as L

    key = ("zero-at-rest", 0, 0)
    try:
        L._ws_cache[key] = object()
        with pytest.raises(L.WQError):
            L._check(L.WQ_ETIMEOUT, "wq_check_status")
        assert key not in L._ws_cache
        L._ws_cache[key] = object()
        with pytest.raises(L.WQError):
            L._check(L.WQ_ECUDA, "wna16_gemm")
        assert key not in L._ws_cache
        L._ws_cache[key] = object()
        with pytest.raises(L.WQError):
            L._check(L.WQ_EINVAL, "wna16_gemm")
        assert key in L._ws_cache
    finally:
        L._ws_cache.pop(key, None)
