"""ctypes binding over libwq.so: argument marshalling only.

Every call goes straight to the C ABI declared in include/wq.h; the kernels do
all of the work. PyTorch provides device memory and the current CUDA stream.
There is no fallback: if libwq.so is missing the import of a call fails.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG_DIR, "libwq.so")

WQ_OK, WQ_EINVAL, WQ_EUNSUPPORTED, WQ_ECUDA, WQ_ETIMEOUT = range(5)
_STATUS_NAMES = {0: "WQ_OK", 1: "WQ_EINVAL", 2: "WQ_EUNSUPPORTED", 3: "WQ_ECUDA", 4: "WQ_ETIMEOUT"}

_c_i64 = ctypes.c_int64
_c_int = ctypes.c_int
_c_size = ctypes.c_size_t
_c_ptr = ctypes.c_void_p

# name -> (restype, argtypes); mirrors include/wq.h
SIGNATURES = {
    "wq_packed_words_per_row": (_c_size, [_c_i64, _c_int]),
    "wna16_repack": (_c_int, [_c_ptr, _c_ptr, _c_i64, _c_i64, _c_int, _c_int, _c_ptr, _c_ptr, _c_ptr, _c_ptr]),
    "wna16_workspace_bytes": (_c_size, [_c_i64, _c_i64, _c_i64, _c_int]),
    "wna16_gemm": (_c_int, [_c_ptr, _c_i64, _c_ptr, _c_ptr, _c_i64, _c_i64, _c_int, _c_int, _c_ptr,
                            _c_ptr, _c_size, _c_ptr]),
    "wna16_gemm_zp": (_c_int, [_c_ptr, _c_i64, _c_ptr, _c_ptr, _c_ptr, _c_i64, _c_i64, _c_int, _c_int, _c_ptr,
                               _c_ptr, _c_size, _c_ptr]),
    "wna16_zp_workspace_bytes": (_c_size, [_c_i64, _c_i64, _c_i64, _c_int]),
    "wna16_moe_gemm": (_c_int, [_c_ptr, _c_i64, _c_ptr, _c_i64, _c_ptr, _c_ptr, _c_i64, _c_i64, _c_int, _c_int,
                                _c_ptr, _c_ptr]),
    "wna16_gemm_noalloc": (_c_int, [_c_ptr, _c_i64, _c_ptr, _c_ptr, _c_i64, _c_i64, _c_int, _c_int,
                                    _c_ptr, _c_ptr]),
    "act_quant_int8": (_c_int, [_c_ptr, _c_i64, _c_i64, _c_ptr, _c_ptr, _c_ptr]),
    "w4a8_workspace_bytes": (_c_size, [_c_i64, _c_i64, _c_i64]),
    "w4a8_scratch_bytes": (_c_size, [_c_i64, _c_i64]),
    "w4a8_gemm": (_c_int, [_c_ptr, _c_i64, _c_ptr, _c_ptr, _c_i64, _c_i64, _c_int, _c_ptr, _c_ptr,
                           _c_size, _c_ptr, _c_size, _c_ptr]),
    "qembed_gather": (_c_int, [_c_ptr, _c_i64, _c_ptr, _c_ptr, _c_i64, _c_i64, _c_int, _c_int, _c_ptr,
                               _c_ptr, _c_ptr]),
    "wq_debug_decode_plan": (_c_int, [_c_i64, _c_i64, _c_i64, _c_int, _c_int, _c_ptr]),
    "wq_debug_route": (_c_int, [_c_i64, _c_i64, _c_i64, _c_int, _c_int, _c_int, _c_ptr]),
    "wq_debug_unpack": (_c_int, [_c_ptr, _c_i64, _c_i64, _c_int, _c_ptr, _c_ptr]),
    "wq_debug_w4a8_group_acc": (_c_int, [_c_ptr, _c_i64, _c_ptr, _c_ptr, _c_i64, _c_i64, _c_ptr, _c_ptr,
                                         _c_size, _c_ptr]),
    "wq_debug_noalloc_scratch": (_c_int, [_c_ptr, _c_size, _c_int, _c_ptr]),
    "wq_debug_mma_peak": (_c_int, [_c_int, _c_i64, _c_int, _c_ptr, _c_ptr]),
    "wq_debug_decode_wait_fault": (_c_int, [_c_i64, ctypes.c_uint64]),
    "wq_check_status": (_c_int, []),
    "wq_last_error": (ctypes.c_char_p, []),
    "wq_version": (ctypes.c_char_p, []),
}

_lib = None
_lib_lock = threading.Lock()


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libwq.so (once) and attaches the C signatures."""
    global _lib
    with _lib_lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libwq.so not found at {path}; build it first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
        return _lib


class WQError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        super().__init__(f"{where}: {_STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def _check(status: int, where: str) -> None:
    if status != WQ_OK:
        msg = load().wq_last_error().decode()
        if status in (WQ_ECUDA, WQ_ETIMEOUT):
            # device work may have stopped part-way: a zero-at-rest workspace
            # can hold partial sums, so the cached buffers are dropped and the
            # next call gets a zero-filled one (argument errors launch nothing)
            drop_workspaces()
        raise WQError(status, where, msg)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _need(t: torch.Tensor, name: str, dtype, shape=None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype} (got {t.dtype})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)} (got {tuple(t.shape)})")


# ---------------------------------------------------------------- workspaces

_ws_cache: dict = {}
_ws_lock = threading.Lock()


def _cached(kind: str, nbytes: int, device=None) -> torch.Tensor | None:
    if nbytes == 0:
        return None
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    key = (kind, dev.index, _stream())
    with _ws_lock:
        buf = _ws_cache.get(key)
        if buf is None or buf.numel() < nbytes:
            buf = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device=dev)
            _ws_cache[key] = buf
        return buf


def drop_workspaces() -> None:
    """Forgets every cached workspace and scratch buffer; later calls allocate
    fresh zero-filled ones. Called after a device-side failure. The memory
    returns to PyTorch's allocator, which reuses it in stream order."""
    with _ws_lock:
        _ws_cache.clear()


def workspace(nbytes: int, device=None) -> torch.Tensor | None:
    """A zero-filled split-K workspace for the current stream, reused across
    calls. The library leaves it zero-filled after every successful call;
    calls that share it are serialised by the stream."""
    return _cached("zero-at-rest", nbytes, device)


def scratch(nbytes: int, device=None) -> torch.Tensor | None:
    """A scratch buffer (contents undefined between calls) for the current stream."""
    return _cached("scratch", nbytes, device)


# ---------------------------------------------------------------- host queries

def packed_words_per_row(K: int, bits: int) -> int:
    return int(load().wq_packed_words_per_row(K, bits))


def wna16_workspace_bytes(M: int, N: int, K: int, bits: int) -> int:
    return int(load().wna16_workspace_bytes(M, N, K, bits))


def wna16_zp_workspace_bytes(M: int, N: int, K: int, bits: int) -> int:
    return int(load().wna16_zp_workspace_bytes(M, N, K, bits))


def w4a8_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load().w4a8_workspace_bytes(M, N, K))


def w4a8_scratch_bytes(M: int, K: int) -> int:
    return int(load().w4a8_scratch_bytes(M, K))


def version() -> str:
    return load().wq_version().decode()


def check_status() -> None:
    _check(load().wq_check_status(), "wq_check_status")


# ---------------------------------------------------------------- entry points

def wna16_repack(codes: torch.Tensor, scales: torch.Tensor, bits: int, group: int = 128,
                 packed: torch.Tensor | None = None, scales_out: torch.Tensor | None = None,
                 bad_count: torch.Tensor | None = None):
    """codes uint8 [N, K], scales bf16 [N, K/128] -> (packed uint32-as-int32 [N, W], scales_out)."""
    N, K = codes.shape
    _need(codes, "codes", torch.uint8)
    _need(scales, "scales", torch.bfloat16, (N, K // group))
    W = packed_words_per_row(K, bits)
    if packed is None:
        packed = torch.empty((N, W), dtype=torch.int32, device=codes.device)
    _need(packed, "packed", torch.int32, (N, W))
    if scales_out is None:
        scales_out = torch.empty_like(scales)
    _need(scales_out, "scales_out", torch.bfloat16, (N, K // group))
    if bad_count is not None:
        _need(bad_count, "bad_count", torch.int32)
    _check(load().wna16_repack(_ptr(codes), _ptr(scales), N, K, bits, group, _ptr(packed),
                               _ptr(scales_out), _ptr(bad_count), _stream()), "wna16_repack")
    return packed, scales_out


def wna16_gemm(x: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor, N: int, K: int, bits: int,
               group: int = 128, y: torch.Tensor | None = None, ws: torch.Tensor | None = None):
    """y[M, N] = x[M, K] . dequant(W)^T, bf16 out."""
    M = x.shape[0]
    _need(x, "x", torch.bfloat16, (M, K))
    _need(packed, "packed", torch.int32, (N, packed_words_per_row(K, bits)))
    _need(scales, "scales", torch.bfloat16, (N, K // group))
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _need(y, "y", torch.bfloat16, (M, N))
    need = wna16_workspace_bytes(M, N, K, bits)
    if ws is None:
        ws = workspace(need)
    _check(load().wna16_gemm(_ptr(x), M, _ptr(packed), _ptr(scales), N, K, bits, group, _ptr(y),
                             _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(), _stream()),
           "wna16_gemm")
    return y


def wna16_gemm_zp(x: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor, N: int,
                  K: int, bits: int, group: int = 128, y: torch.Tensor | None = None,
                  ws: torch.Tensor | None = None):
    """y[M, N] = x[M, K] . dequant(W)^T with a zero point per (row, group):
    w = s * (q - zp); zeros uint8 [N, K/128]."""
    M = x.shape[0]
    _need(x, "x", torch.bfloat16, (M, K))
    _need(packed, "packed", torch.int32, (N, packed_words_per_row(K, bits)))
    _need(scales, "scales", torch.bfloat16, (N, K // group))
    _need(zeros, "zeros", torch.uint8, (N, K // group))
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _need(y, "y", torch.bfloat16, (M, N))
    need = wna16_zp_workspace_bytes(M, N, K, bits)
    if ws is None:
        ws = workspace(need)
    _check(load().wna16_gemm_zp(_ptr(x), M, _ptr(packed), _ptr(scales), _ptr(zeros), N, K, bits, group, _ptr(y),
                                _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(), _stream()),
           "wna16_gemm_zp")
    return y


def wna16_moe_gemm(x: torch.Tensor, expert_offsets: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor,
                   E: int, N: int, K: int, bits: int, group: int = 128, y: torch.Tensor | None = None):
    """Mixture of experts: x [M, K] sorted by expert, expert_offsets int32
    [E + 1] on the device, packed [E * N, words] and scales [E * N, K/128]
    stacked per expert; y [M, N]."""
    M = x.shape[0]
    _need(x, "x", torch.bfloat16, (M, K))
    _need(expert_offsets, "expert_offsets", torch.int32, (E + 1,))
    _need(packed, "packed", torch.int32, (E * N, packed_words_per_row(K, bits)))
    _need(scales, "scales", torch.bfloat16, (E * N, K // group))
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _need(y, "y", torch.bfloat16, (M, N))
    _check(load().wna16_moe_gemm(_ptr(x), M, _ptr(expert_offsets), E, _ptr(packed), _ptr(scales), N, K, bits, group,
                                 _ptr(y), _stream()), "wna16_moe_gemm")
    return y


def wna16_gemm_noalloc(x: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor, N: int, K: int,
                       bits: int, group: int = 128, y: torch.Tensor | None = None):
    """wna16_gemm without a workspace: the library's fixed scratch array is
    used instead (for callers that cannot allocate device memory)."""
    M = x.shape[0]
    _need(x, "x", torch.bfloat16, (M, K))
    _need(packed, "packed", torch.int32, (N, packed_words_per_row(K, bits)))
    _need(scales, "scales", torch.bfloat16, (N, K // group))
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _need(y, "y", torch.bfloat16, (M, N))
    _check(load().wna16_gemm_noalloc(_ptr(x), M, _ptr(packed), _ptr(scales), N, K, bits, group, _ptr(y),
                                     _stream()), "wna16_gemm_noalloc")
    return y


def act_quant_int8(x: torch.Tensor, xq: torch.Tensor | None = None, sx: torch.Tensor | None = None):
    M, K = x.shape
    _need(x, "x", torch.bfloat16)
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.int8, device=x.device)
    if sx is None:
        sx = torch.empty((M,), dtype=torch.float32, device=x.device)
    _need(xq, "xq", torch.int8, (M, K))
    _need(sx, "sx", torch.float32, (M,))
    _check(load().act_quant_int8(_ptr(x), M, K, _ptr(xq), _ptr(sx), _stream()), "act_quant_int8")
    return xq, sx


def w4a8_gemm(x: torch.Tensor, packed4: torch.Tensor, scales: torch.Tensor, N: int, K: int,
              group: int = 128, y: torch.Tensor | None = None, ws: torch.Tensor | None = None,
              scr: torch.Tensor | None = None):
    M = x.shape[0]
    _need(x, "x", torch.bfloat16, (M, K))
    _need(packed4, "packed4", torch.int32, (N, packed_words_per_row(K, 4)))
    _need(scales, "scales", torch.bfloat16, (N, K // group))
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _need(y, "y", torch.bfloat16, (M, N))
    need = w4a8_workspace_bytes(M, N, K)
    if ws is None:
        ws = workspace(need)
    if scr is None:
        scr = scratch(w4a8_scratch_bytes(M, K))
    _check(load().w4a8_gemm(_ptr(x), M, _ptr(packed4), _ptr(scales), N, K, group, _ptr(y), _ptr(ws),
                            0 if ws is None else ws.numel() * ws.element_size(), _ptr(scr),
                            scr.numel() * scr.element_size(), _stream()), "w4a8_gemm")
    return y


def qembed_gather(ids: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor, V: int, D: int,
                  bits: int, group: int = 128, out: torch.Tensor | None = None,
                  bad_count: torch.Tensor | None = None):
    T = ids.shape[0]
    _need(ids, "ids", torch.int32, (T,))
    _need(packed, "packed", torch.int32, (V, packed_words_per_row(D, bits)))
    _need(scales, "scales", torch.bfloat16, (V, D // group))
    if out is None:
        out = torch.empty((T, D), dtype=torch.bfloat16, device=ids.device)
    _need(out, "out", torch.bfloat16, (T, D))
    if bad_count is not None:
        _need(bad_count, "bad_count", torch.int32)
    _check(load().qembed_gather(_ptr(ids), T, _ptr(packed), _ptr(scales), V, D, bits, group, _ptr(out),
                                _ptr(bad_count), _stream()), "qembed_gather")
    return out


_PLAN_KEYS = ("ok", "C", "H", "nchunk", "T", "ksplit", "NS", "G", "Gh", "sbox", "sx0", "NT", "smem",
              "max_slots")


def debug_decode_plan(M: int, N: int, K: int, bits: int, sm_count: int) -> dict:
    """The CTA-pair decode kernel's launch plan for a shape (host only)."""
    out = (ctypes.c_int64 * len(_PLAN_KEYS))()
    _check(load().wq_debug_decode_plan(M, N, K, bits, sm_count, ctypes.addressof(out)), "wq_debug_decode_plan")
    return dict(zip(_PLAN_KEYS, (int(v) for v in out)))


ROUTES = {0: "none", 1: "decode_pair", 2: "decode_splitk", 3: "chunked", 4: "tensor_core"}


def debug_route(M: int, N: int, K: int, bits: int, sm_count: int, w4a8: bool = False, zp: bool = False) -> str:
    """Which kernel wna16_gemm (or w4a8_gemm, or with zp wna16_gemm_zp)
    launches for a shape on a device with sm_count SMs (host only): one of the
    ROUTES names."""
    out = ctypes.c_int(0)
    kind = 1 if w4a8 else (2 if zp else 0)
    _check(load().wq_debug_route(M, N, K, bits, kind, sm_count, ctypes.byref(out)), "wq_debug_route")
    return ROUTES[out.value]


def debug_unpack(packed: torch.Tensor, N: int, K: int, bits: int) -> torch.Tensor:
    _need(packed, "packed", torch.int32, (N, packed_words_per_row(K, bits)))
    codes = torch.empty((N, K), dtype=torch.uint8, device=packed.device)
    _check(load().wq_debug_unpack(_ptr(packed), N, K, bits, _ptr(codes), _stream()), "wq_debug_unpack")
    return codes


def debug_mma_peak(kind: int, iters: int, blocks: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """Launches the mma.sync throughput probe (kind 0: int8 m16n8k32, kind 1:
    bf16 m16n8k16) on the current stream; returns the per-thread checksums
    [blocks * 256] int32 (each 8 * 4 * K * iters)."""
    if out is None:
        out = torch.empty(blocks * 256, dtype=torch.int32, device="cuda")
    _need(out, "out", torch.int32, (blocks * 256,))
    _check(load().wq_debug_mma_peak(kind, iters, blocks, _ptr(out), _stream()), "wq_debug_mma_peak")
    return out


def debug_w4a8_group_acc(x: torch.Tensor, packed4: torch.Tensor, scales: torch.Tensor, N: int, K: int,
                         acc: torch.Tensor | None = None) -> torch.Tensor:
    """The exact int32 group accumulators [M, N, K/128] of W4A8, from the
    kernel w4a8_gemm launches for the same shape (x is the bf16 activation,
    quantized per token exactly as w4a8_gemm does)."""
    M = x.shape[0]
    _need(x, "x", torch.bfloat16, (M, K))
    _need(packed4, "packed4", torch.int32, (N, packed_words_per_row(K, 4)))
    _need(scales, "scales", torch.bfloat16, (N, K // 128))
    if acc is None:
        acc = torch.empty((M, N, K // 128), dtype=torch.int32, device=x.device)
    _need(acc, "acc", torch.int32, (M, N, K // 128))
    scr = scratch(w4a8_scratch_bytes(M, K))
    _check(load().wq_debug_w4a8_group_acc(_ptr(x), M, _ptr(packed4), _ptr(scales), N, K, _ptr(acc), _ptr(scr),
                                          scr.numel() * scr.element_size(), _stream()),
           "wq_debug_w4a8_group_acc")
    return acc
