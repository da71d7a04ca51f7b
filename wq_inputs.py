"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no packing, dequantization or quantization). Both the CPU
oracle and the CUDA library receive the identical arrays produced here.

Recipe (numpy PCG64, one generator per call, seeded explicitly):

* activations x: N(0, 1) rounded to bf16 (round-to-nearest-even, done by
  torch's dtype conversion);
* W4A8 activations: the same, with 1% of the K channels (chosen by the seed,
  shared by every token) multiplied by 20 before rounding;
* codes: integers uniform in [0, 2^bits - 1], stored one per byte;
* scales: 0.01 * |N(0, 1)| with an independent random sign per (row, group),
  rounded to bf16, so about half of the scales are negative;
* token ids: uniform in [0, V).

Every array that stands for bf16 data is returned as raw uint16 bit patterns.
"""

from __future__ import annotations

import numpy as np

GROUP = 128


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(int(seed)))


def _to_bf16_bits(a: np.ndarray) -> np.ndarray:
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def make_x(M: int, K: int, seed: int) -> np.ndarray:
    """bf16 bits [M, K] of N(0, 1) activations."""
    return _to_bf16_bits(rng(seed).standard_normal((M, K), dtype=np.float32))


def make_x_outliers(M: int, K: int, seed: int, frac: float = 0.01,
                    factor: float = 20.0) -> np.ndarray:
    """bf16 bits [M, K]: N(0, 1) with round(frac*K) outlier channels x factor."""
    g = rng(seed)
    x = g.standard_normal((M, K), dtype=np.float32)
    n_out = max(1, int(round(frac * K)))
    cols = g.choice(K, size=n_out, replace=False)
    x[:, cols] *= np.float32(factor)
    return _to_bf16_bits(x)


def make_codes(N: int, K: int, bits: int, seed: int) -> np.ndarray:
    """uint8 [N, K] codes uniform in [0, 2^bits - 1]."""
    return rng(seed).integers(0, 1 << bits, size=(N, K), dtype=np.uint8)


def make_scales(N: int, G: int, seed: int, sign: str = "random") -> np.ndarray:
    """bf16 bits [N, G] of 0.01*|N(0,1)| with a sign per entry.

    sign: "random" (independent +-1, p = 1/2), "negative" or "positive"."""
    g = rng(seed)
    mag = np.float32(0.01) * np.abs(g.standard_normal((N, G), dtype=np.float32))
    if sign == "random":
        sgn = np.where(g.integers(0, 2, size=(N, G)) == 1, -1.0, 1.0).astype(np.float32)
    elif sign == "negative":
        sgn = np.float32(-1.0)
    elif sign == "positive":
        sgn = np.float32(1.0)
    else:
        raise ValueError(sign)
    return _to_bf16_bits(mag * sgn)


def make_ids(T: int, V: int, seed: int) -> np.ndarray:
    """int32 [T] token ids uniform in [0, V)."""
    return rng(seed).integers(0, V, size=(T,), dtype=np.int64).astype(np.int32)


def stack_layer_bits(layer: int) -> int:
    """Bit width of layer 0..63 of the synthetic mixed-bit stack: edge layers
    0-9 and 54-63 use 7 bits; the 44 middle layers alternate 5 and 6 bits,
    starting with 5 at layer 10."""
    if layer < 0 or layer > 63:
        raise ValueError("layer out of range")
    if layer <= 9 or layer >= 54:
        return 7
    return 5 if (layer - 10) % 2 == 0 else 6


def seed_for(config_index: int, salt: int = 0) -> int:
    """Seed convention: 1000 + configuration index, plus a per-array salt."""
    return 1000 + int(config_index) + 7919 * int(salt)
