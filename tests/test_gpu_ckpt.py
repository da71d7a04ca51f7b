"""Layers imported from a pack-quantized safetensors checkpoint (dense,
word-aligned and asymmetric) run through the library and match the oracle."""

import numpy as np
import pytest

import oracle as O
import wq_inputs as I
from helpers import assert_bf16_close, to_dev_bf16
from test_ckpt import _layer_tensors

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from weight_only_int2_gb300 import ckpt  # noqa: E402


def test_imported_layers_match_the_oracle(tmp_path):
    K = 1024
    specs = [("dense6", 6, 300, "dense", False), ("aligned6", 6, 200, "word-aligned", False),
             ("dense5zp", 5, 260, "dense", True)]
    tensors, ref = {}, {}
    for name, bits, N, layout, asym in specs:
        q = I.make_codes(N, K, bits, 300 + N)
        s = I.make_scales(N, K // 128, 301 + N)
        zp = np.random.default_rng(N).integers(0, 1 << bits, size=(N, K // 128)) if asym else None
        tensors.update(_layer_tensors(name, q, s, bits, layout=layout, zeros=zp))
        ref[name] = (q, s, zp, bits)
    path = str(tmp_path / "model.safetensors")
    ckpt.write_safetensors(path, tensors)
    t = ckpt.read_safetensors(path)
    for M in (1, 16, 100):
        x = I.make_x(M, K, 310 + M)
        for name, bits, N, layout, asym in specs:
            lay = ckpt.load_layer(t, name, bits)
            assert lay.layout == layout
            y = ckpt.linear(ckpt.to_device(lay), to_dev_bf16(x), lay)
            q, s, zp, _ = ref[name]
            y_ref = O.wna16_zp_ref(x, q, s, zp, bits) if asym else O.wna16_ref(x, q, s, bits)
            assert_bf16_close(y, y_ref, f"{name} M={M}")
