"""CPU checks of the bit-unpacking tables the weight-streaming kernels use
(`pair_spec<B>` in weight_only_int2_gb300/csrc/wq_unpack.cuh), parsed from the
header and replayed in Python on random words: every table pairs the 32 codes
of a b-word slice exactly once, and its 32-bit window holds both codes of a
pair, at offsets the 16-bit float mantissa keeps exact, for every width 2..8.
The layout being read is the dense LSB-first stream of the
"Qwen3.8-27B-INT6-Mixed-AutoRound" model card, section "Findings"."""

import os
import re

import numpy as np
import pytest

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "weight_only_int2_gb300", "csrc", "wq_unpack.cuh")


def _tables():
    src = open(HEADER).read()
    out = {2: [(16 * (p >> 3) + (p & 7), 16 * (p >> 3) + (p & 7) + 8, 32 * (p >> 3) + 2 * (p & 7), 0, 0)
               for p in range(16)],
           4: [(8 * (p >> 2) + (p & 3), 8 * (p >> 2) + (p & 3) + 4, 32 * (p >> 2) + 4 * (p & 3), 0, 0)
               for p in range(16)]}
    for b in (3, 5, 6, 7):
        m = re.search(r"B == %d\) \{\s*constexpr PairSpec t\[16\] = \{(.*?)\};" % b, src, re.S)
        out[b] = [tuple(int(v) for v in e.split(",")) for e in re.findall(r"\{([-\d,\s]+)\}", m.group(1))]
    m = re.search(r"\} else \{\s*constexpr PairSpec t\[16\] = \{(.*?)\};", src, re.S)
    out[8] = [tuple(int(v) for v in e.split(",")) for e in re.findall(r"\{([-\d,\s]+)\}", m.group(1))]
    # the closed forms of b = 2 and 4 are written in the header, not a table
    assert "16 * (p >> 3) + (p & 7)" in src and "8 * (p >> 2) + (p & 3)" in src
    return out


def _window(words, s):
    """32 bits of the slice starting at bit s (bits below the slice read as 0)."""
    stream = 0
    for i, w in enumerate(words):
        stream |= int(w) << (32 * i)
    return (stream << -s) & 0xFFFFFFFF if s < 0 else (stream >> s) & 0xFFFFFFFF


@pytest.mark.parametrize("bits", range(2, 9))
def test_pair_table_covers_each_code_once(bits):
    t = _tables()[bits]
    assert len(t) == 16
    codes = sorted([lo for lo, _, _, _, _ in t] + [hi for _, hi, _, _, _ in t])
    assert codes == list(range(32))


@pytest.mark.parametrize("bits", range(2, 9))
def test_pair_windows_hold_the_codes(bits):
    """Window W = slice >> s keeps code lo at bit olo and code hi at bit
    16 + ohi, with the code's top bit below the mantissa's (7 bits for the
    bf16 widths 2 and 4, 10 for the fp16 ones), so magic | code is exact."""
    mant = 7 if bits in (2, 4) else 10
    rng = np.random.default_rng(bits)
    t = _tables()[bits]
    for _ in range(64):
        codes = rng.integers(0, 1 << bits, size=(1, 32), dtype=np.uint8)
        words = O.pack(codes, bits)[0]            # the oracle's packing of one slice
        assert len(words) == bits
        for lo, hi, s, olo, ohi in t:
            assert olo + bits <= mant and ohi + bits <= mant
            w = _window(words, s)
            assert (w >> olo) & ((1 << bits) - 1) == codes[0, lo]
            assert (w >> (16 + ohi)) & ((1 << bits) - 1) == codes[0, hi]
