"""Importer for pack-quantized checkpoints (safetensors files).

Model card "Qwen3.8-27B-INT6-Mixed-AutoRound", section "Findings", first
bullet: recent compressed-tensors releases store a layer's b-bit codes densely,
``ceil(in_features * bits / 32)`` 32-bit words per output row, codes
straddling word boundaries; older readers assumed the word-aligned layout
(``32 // bits`` codes per word, never straddling), which agrees with the dense
one only when bits divides 32. The dense layout is exactly this library's
packed layout, so a dense checkpoint tensor goes to the GPU unchanged; a
word-aligned one is converted to codes here and repacked on the GPU.

A layer ``<prefix>`` is read from these tensors:

* ``<prefix>.weight_packed``  int32 [N, words]: the codes (dense or word-aligned);
* ``<prefix>.weight_scale``   bf16 or fp16 [N, K / 128]: the group scales (an
  fp16 scale is converted to bf16, which rounds it; bf16 is kept bit for bit);
* ``<prefix>.weight_shape``   integer [2]: (N, K);
* ``<prefix>.weight_zero_point`` (optional) integer [N, K / 128]: per-group zero
  points of an asymmetric layer, one value per (row, group).

The safetensors container (a little-endian uint64 header length, a JSON header
naming each tensor's dtype, shape and byte range, then the raw bytes) is read
with numpy memory maps; nothing is copied until a tensor is used. This module
does host-side IO only: every dequantization and GEMM runs in the CUDA library
(``wna16_gemm`` / ``wna16_gemm_zp`` on the tensors returned by ``to_device``).
"""

from __future__ import annotations

import json
import os
import struct
from dataclasses import dataclass

import numpy as np

GROUP = 128

_DTYPES = {
    "BOOL": np.bool_, "U8": np.uint8, "I8": np.int8, "I16": np.int16, "U16": np.uint16,
    "I32": np.int32, "U32": np.uint32, "I64": np.int64, "U64": np.uint64,
    "F16": np.float16, "BF16": np.uint16, "F32": np.float32, "F64": np.float64,
}
_NAMES = {v: k for k, v in _DTYPES.items() if k != "BF16"}


class CheckpointError(ValueError):
    """A checkpoint tensor is missing or does not have the expected form."""


def read_safetensors(path: str) -> dict:
    """Maps every tensor of a safetensors file: name -> (dtype name, numpy
    array view). bf16 tensors come back as their raw uint16 bit patterns."""
    size = os.path.getsize(path)
    with open(path, "rb") as f:
        raw = f.read(8)
        if len(raw) != 8:
            raise CheckpointError(f"{path}: too short for a safetensors header")
        (hlen,) = struct.unpack("<Q", raw)
        if hlen <= 0 or 8 + hlen > size:
            raise CheckpointError(f"{path}: header length {hlen} does not fit the file")
        header = json.loads(f.read(hlen).decode("utf-8"))
    base = 8 + hlen
    mm = np.memmap(path, dtype=np.uint8, mode="r")
    out = {}
    for name, meta in header.items():
        if name == "__metadata__":
            continue
        dt = meta["dtype"]
        if dt not in _DTYPES:
            raise CheckpointError(f"{path}: tensor {name}: unsupported dtype {dt}")
        b0, b1 = meta["data_offsets"]
        shape = tuple(int(d) for d in meta["shape"])
        npdt = np.dtype(_DTYPES[dt])
        count = int(np.prod(shape, dtype=np.int64)) if shape else 1
        if b1 - b0 != count * npdt.itemsize or base + b1 > size:
            raise CheckpointError(f"{path}: tensor {name}: byte range [{b0}, {b1}) does not match {dt}{shape}")
        out[name] = (dt, mm[base + b0: base + b1].view(npdt).reshape(shape))
    return out


def write_safetensors(path: str, tensors: dict, metadata: dict | None = None) -> None:
    """Writes name -> (dtype name, numpy array) as a safetensors file ("BF16"
    arrays are given as uint16 bit patterns)."""
    header = {}
    blobs = []
    off = 0
    for name, (dt, arr) in tensors.items():
        a = np.ascontiguousarray(arr, dtype=_DTYPES[dt])
        header[name] = {"dtype": dt, "shape": list(a.shape), "data_offsets": [off, off + a.nbytes]}
        blobs.append(a.tobytes())
        off += a.nbytes
    if metadata:
        header["__metadata__"] = {str(k): str(v) for k, v in metadata.items()}
    h = json.dumps(header, separators=(",", ":")).encode("utf-8")
    h += b" " * ((8 - len(h) % 8) % 8)
    with open(path, "wb") as f:
        f.write(struct.pack("<Q", len(h)))
        f.write(h)
        for b in blobs:
            f.write(b)


def dense_words(K: int, bits: int) -> int:
    """Words per row of the dense layout: ceil(K * bits / 32)."""
    return (int(K) * int(bits) + 31) // 32


def word_aligned_words(K: int, bits: int) -> int:
    """Words per row of the word-aligned layout: ceil(K / (32 // bits))."""
    per = 32 // int(bits)
    return (int(K) + per - 1) // per


def codes_from_word_aligned(words: np.ndarray, K: int, bits: int) -> np.ndarray:
    """Codes [N, K] (uint8) of a word-aligned row: code k sits in word
    k // (32 // bits) at bit (k % (32 // bits)) * bits."""
    per = 32 // int(bits)
    w = np.asarray(words, dtype=np.uint32)
    k = np.arange(K)
    shifts = ((k % per) * bits).astype(np.uint32)
    vals = (w[:, k // per] >> shifts[None, :]) & np.uint32((1 << bits) - 1)
    return vals.astype(np.uint8)


@dataclass
class QuantLayer:
    """One pack-quantized linear layer on the host.

    packed: int32 [N, ceil(K * bits / 32)] in the dense layout, or None when
            the checkpoint was word-aligned (then ``codes`` holds the codes,
            which wna16_repack packs on the GPU);
    codes:  uint8 [N, K] or None;
    scales: bf16 bit patterns (uint16) [N, K / 128];
    zeros:  uint8 [N, K / 128] zero points, or None for the symmetric layer."""

    name: str
    N: int
    K: int
    bits: int
    packed: np.ndarray | None
    codes: np.ndarray | None
    scales: np.ndarray
    zeros: np.ndarray | None
    layout: str  # "dense" or "word-aligned"


def _f16_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    f = np.asarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)).astype(np.uint16)
    return r


def load_layer(tensors: dict, prefix: str, bits: int, group: int = GROUP) -> QuantLayer:
    """Reads layer ``prefix`` (see the module docstring) from the mapping
    returned by read_safetensors."""
    if group != GROUP:
        raise CheckpointError(f"{prefix}: group {group} is not supported (128)")
    if not 2 <= int(bits) <= 8:
        raise CheckpointError(f"{prefix}: bits {bits} outside 2..8")

    def get(suffix, required=True):
        key = f"{prefix}.{suffix}"
        if key not in tensors:
            if required:
                raise CheckpointError(f"missing tensor {key}")
            return None, None
        return tensors[key]

    _, shape = get("weight_shape")
    shape = np.asarray(shape).astype(np.int64).reshape(-1)
    if shape.size != 2:
        raise CheckpointError(f"{prefix}.weight_shape must hold (N, K)")
    N, K = int(shape[0]), int(shape[1])
    if K % group:
        raise CheckpointError(f"{prefix}: K = {K} is not a multiple of {group}")
    pdt, packed = get("weight_packed")
    if pdt not in ("I32", "U32") or packed.ndim != 2 or packed.shape[0] != N:
        raise CheckpointError(f"{prefix}.weight_packed must be int32 [N, words], got {pdt}{packed.shape}")
    words = packed.shape[1]
    sdt, scales = get("weight_scale")
    if scales.shape != (N, K // group):
        raise CheckpointError(f"{prefix}.weight_scale must be [{N}, {K // group}], got {scales.shape}")
    if sdt == "BF16":
        sbits = np.ascontiguousarray(scales, dtype=np.uint16)
    elif sdt in ("F16", "F32"):
        sbits = _f16_to_bf16_bits(scales)
    else:
        raise CheckpointError(f"{prefix}.weight_scale: unsupported dtype {sdt}")
    zdt, zp = get("weight_zero_point", required=False)
    zeros = None
    if zp is not None:
        if zp.shape != (N, K // group):
            raise CheckpointError(f"{prefix}.weight_zero_point must be [{N}, {K // group}] (one per row and group)")
        z = np.asarray(zp).astype(np.int64)
        if z.min(initial=0) < 0 or z.max(initial=0) > (1 << bits) - 1:
            raise CheckpointError(f"{prefix}.weight_zero_point: values outside [0, 2^{bits} - 1]")
        zeros = z.astype(np.uint8)
    dense, aligned = dense_words(K, bits), word_aligned_words(K, bits)
    if words == dense:
        return QuantLayer(prefix, N, K, bits, np.ascontiguousarray(packed).view(np.int32), None, sbits, zeros,
                          "dense")
    if words == aligned:
        codes = codes_from_word_aligned(np.asarray(packed).view(np.uint32), K, bits)
        return QuantLayer(prefix, N, K, bits, None, codes, sbits, zeros, "word-aligned")
    raise CheckpointError(f"{prefix}.weight_packed has {words} words per row: neither the dense layout "
                          f"({dense}) nor the word-aligned one ({aligned}) for K = {K}, bits = {bits}")


def to_device(layer: QuantLayer, device="cuda"):
    """Moves a layer to the GPU in the library's layout: returns (packed int32,
    scales bf16, zeros uint8 or None). A word-aligned layer is repacked on the
    GPU (wna16_repack)."""
    import torch

    from . import _lib

    s_dev = torch.from_numpy(np.array(layer.scales, dtype=np.uint16, order="C", copy=True).view(np.int16)).view(torch.bfloat16).to(device)
    z_dev = None if layer.zeros is None else torch.from_numpy(np.array(layer.zeros, dtype=np.uint8, order="C", copy=True)).to(device)
    if layer.packed is not None:
        p_dev = torch.from_numpy(np.array(layer.packed, dtype=np.int32, order="C", copy=True)).to(device)
    else:
        c_dev = torch.from_numpy(np.array(layer.codes, dtype=np.uint8, order="C", copy=True)).to(device)
        p_dev, _ = _lib.wna16_repack(c_dev, s_dev, layer.bits)
    return p_dev, s_dev, z_dev


def linear(layer_dev, x, layer: QuantLayer):
    """y = x . dequant(W)^T for a layer moved with to_device."""
    from . import _lib

    p_dev, s_dev, z_dev = layer_dev
    if z_dev is None:
        return _lib.wna16_gemm(x, p_dev, s_dev, layer.N, layer.K, layer.bits)
    return _lib.wna16_gemm_zp(x, p_dev, s_dev, z_dev, layer.N, layer.K, layer.bits)
