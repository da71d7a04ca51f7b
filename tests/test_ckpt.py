"""CPU checks of the checkpoint importer (weight_only_int2_gb300.ckpt): the
safetensors container read from a file built byte by byte after its published
definition, the dense layout taken over bit for bit (it is the library's
packed layout; compared with the oracle's packing), the word-aligned layout
converted to codes, fp16 scales rounded to bf16, zero points, and clear
errors for malformed layers. No GPU."""

import json
import struct

import numpy as np
import pytest

import oracle as O
import wq_inputs as I
from weight_only_int2_gb300 import ckpt


def test_reader_on_a_hand_built_file(tmp_path):
    a = np.arange(6, dtype=np.int32).reshape(2, 3)
    b = np.array([0x3F80, 0xC000], dtype=np.uint16)          # bf16 1.0, -2.0
    header = {"a": {"dtype": "I32", "shape": [2, 3], "data_offsets": [0, 24]},
              "b": {"dtype": "BF16", "shape": [2], "data_offsets": [24, 28]},
              "__metadata__": {"format": "pt"}}
    h = json.dumps(header).encode()
    path = tmp_path / "hand.safetensors"
    path.write_bytes(struct.pack("<Q", len(h)) + h + a.tobytes() + b.tobytes())
    t = ckpt.read_safetensors(str(path))
    assert sorted(t) == ["a", "b"]
    assert t["a"][0] == "I32" and np.array_equal(t["a"][1], a)
    assert t["b"][0] == "BF16" and np.array_equal(t["b"][1], b)


def test_writer_round_trip(tmp_path):
    arrs = {"x": ("F32", np.linspace(-1, 1, 12, dtype=np.float32).reshape(3, 4)),
            "y": ("U8", np.arange(7, dtype=np.uint8)),
            "z": ("I64", np.array([5, -6], dtype=np.int64))}
    path = str(tmp_path / "rt.safetensors")
    ckpt.write_safetensors(path, arrs, {"k": "v"})
    t = ckpt.read_safetensors(path)
    for k, (dt, a) in arrs.items():
        assert t[k][0] == dt and np.array_equal(t[k][1], a)


def _word_aligned(q, bits):
    per = 32 // bits
    N, K = q.shape
    w = np.zeros((N, (K + per - 1) // per), dtype=np.uint64)
    for k in range(K):
        w[:, k // per] |= q[:, k].astype(np.uint64) << np.uint64((k % per) * bits)
    return w.astype(np.uint32)


def _layer_tensors(prefix, q, s_bits, bits, layout="dense", zeros=None, scale_dtype="BF16"):
    N, K = q.shape
    packed = O.pack(q, bits) if layout == "dense" else _word_aligned(q, bits)
    t = {f"{prefix}.weight_packed": ("I32", packed.view(np.int32)),
         f"{prefix}.weight_shape": ("I64", np.array([N, K], dtype=np.int64))}
    if scale_dtype == "BF16":
        t[f"{prefix}.weight_scale"] = ("BF16", s_bits)
    else:
        t[f"{prefix}.weight_scale"] = ("F16", O.bf16_bits_to_f32(s_bits).astype(np.float16))
    if zeros is not None:
        t[f"{prefix}.weight_zero_point"] = ("I32", zeros.astype(np.int32))
    return t


@pytest.mark.parametrize("bits", [3, 5, 6, 7, 8])
def test_dense_layer_is_taken_over_bit_for_bit(tmp_path, bits):
    N, K = 9, 640
    q = I.make_codes(N, K, bits, 70 + bits)
    s = I.make_scales(N, K // 128, 71)
    path = str(tmp_path / "d.safetensors")
    ckpt.write_safetensors(path, _layer_tensors("model.layers.0.mlp.up_proj", q, s, bits))
    lay = ckpt.load_layer(ckpt.read_safetensors(path), "model.layers.0.mlp.up_proj", bits)
    assert lay.layout == "dense" and (lay.N, lay.K) == (N, K)
    assert np.array_equal(lay.packed.view(np.uint32), O.pack(q, bits))
    assert np.array_equal(lay.scales, s) and lay.zeros is None


@pytest.mark.parametrize("bits", [3, 5, 6, 7])
def test_word_aligned_layer_becomes_codes(tmp_path, bits):
    """Widths that do not divide 32: the word-aligned layout has more words
    than the dense one (1024 against 960 at 6 bits, K = 5120)."""
    N, K = 5, 5120
    q = I.make_codes(N, K, bits, 80 + bits)
    s = I.make_scales(N, K // 128, 81)
    assert ckpt.word_aligned_words(K, bits) != ckpt.dense_words(K, bits)
    path = str(tmp_path / "w.safetensors")
    ckpt.write_safetensors(path, _layer_tensors("l", q, s, bits, layout="word-aligned"))
    lay = ckpt.load_layer(ckpt.read_safetensors(path), "l", bits)
    assert lay.layout == "word-aligned" and lay.packed is None
    assert np.array_equal(lay.codes, q)


def test_fp16_scales_and_zero_points(tmp_path):
    bits, N, K = 5, 4, 256
    q = I.make_codes(N, K, bits, 90)
    s = I.make_scales(N, K // 128, 91)
    zp = np.random.default_rng(92).integers(0, 1 << bits, size=(N, K // 128))
    path = str(tmp_path / "z.safetensors")
    ckpt.write_safetensors(path, _layer_tensors("l", q, s, bits, zeros=zp, scale_dtype="F16"))
    lay = ckpt.load_layer(ckpt.read_safetensors(path), "l", bits)
    f16_then_bf16 = O.f32_to_bf16_bits_rne(O.bf16_bits_to_f32(s).astype(np.float16).astype(np.float32))
    assert np.array_equal(lay.scales, f16_then_bf16)
    assert np.array_equal(lay.zeros, zp.astype(np.uint8))


def test_malformed_layers_are_refused(tmp_path):
    bits, N, K = 6, 3, 256
    q = I.make_codes(N, K, bits, 1)
    s = I.make_scales(N, K // 128, 2)
    t = _layer_tensors("l", q, s, bits)
    path = str(tmp_path / "m.safetensors")
    bad = dict(t)
    bad["l.weight_packed"] = ("I32", np.zeros((N, 7), dtype=np.int32))
    ckpt.write_safetensors(path, bad)
    with pytest.raises(ckpt.CheckpointError, match="words per row"):
        ckpt.load_layer(ckpt.read_safetensors(path), "l", bits)
    with pytest.raises(ckpt.CheckpointError, match="missing tensor"):
        ckpt.load_layer(ckpt.read_safetensors(path), "other", bits)
    bad = dict(t)
    bad["l.weight_zero_point"] = ("I32", np.full((N, K // 128), 64, dtype=np.int32))
    ckpt.write_safetensors(path, bad)
    with pytest.raises(ckpt.CheckpointError, match="zero_point"):
        ckpt.load_layer(ckpt.read_safetensors(path), "l", bits)
    (tmp_path / "short.safetensors").write_bytes(b"\x01")
    with pytest.raises(ckpt.CheckpointError):
        ckpt.read_safetensors(str(tmp_path / "short.safetensors"))
