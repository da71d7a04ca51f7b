"""The division recipe of the in-kernel W4A8 activation quantization, checked
with exact rational arithmetic (no GPU). For a token scale sx = m 2^e
(m in [0.5, 1)) the kernel takes f = 2^k, k = clamp(1 - e, -126, 127), and
computes sx' = sx f, x' = x f, y = RN(1 / sx'), q0 = RN(x' y),
r = fma(-q0, sx', x'), q = RN(q0 + r y) (Markstein's correction, IBM J. Res.
Dev. 34(1), 1990), then rint(q) clamped to +-127. This must equal
clamp(rint(RN(x / sx))), the activation-quant definition, for every binary32
x with |x| <= 127 sx (up to rounding), whatever the scale: a normal, a huge or
a subnormal one."""

from fractions import Fraction

import numpy as np
import pytest

F32 = np.float32


def rn32(v: Fraction) -> np.float32:
    """Round an exact rational to the nearest binary32 (ties to even)."""
    if v == 0:
        return F32(0.0)
    f = F32(float(v))  # float() rounds to nearest double; refine to binary32 exactly
    cands = [f, np.nextafter(f, F32(np.inf)), np.nextafter(f, F32(-np.inf))]
    best = None
    for c in cands:
        if not np.isfinite(c):
            continue
        d = abs(Fraction(float(c)) - v)
        if best is None or d < best[0] or (d == best[0] and (int(c.view(np.uint32)) & 1) == 0):
            best = (d, c)
    return best[1]


def fma32(a, b, c) -> np.float32:
    return rn32(Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c)))


def quant_reference(x, sx) -> int:
    if sx == 0:
        return 0
    q = rn32(Fraction(float(x)) / Fraction(float(sx)))
    return int(max(-127, min(127, np.rint(q))))


def quant_recipe(x, sx) -> int:
    if sx == 0:
        return 0
    _, e = np.frexp(np.float64(sx))              # sx = m 2^e, m in [0.5, 1)
    k = min(127, max(-126, 1 - int(e)))
    f = F32(2.0 ** k)
    sxn = F32(sx * f)                             # exact (a power-of-two scaling)
    xs = F32(x * f)                               # exact unless it underflows
    y = rn32(Fraction(1) / Fraction(float(sxn)))
    q0 = F32(xs * y)
    r = fma32(-q0, sxn, xs)
    q = fma32(r, y, q0)
    return int(max(-127, min(127, np.rint(q))))


def _cases(rng, n):
    out = []
    for _ in range(n):
        sx = F32(rng.choice([1e-44, 1e-40, 1e-38, 1e-30, 3e-5, 0.013, 1.0, 7.9, 2.0 ** 60, 2.0 ** 120])
                 * F32(rng.uniform(0.5, 2.0)))
        kind = rng.integers(0, 3)
        if kind == 0:   # uniform in the row's range
            x = F32(rng.uniform(-127.0, 127.0)) * sx
        elif kind == 1:  # exactly at a half-way point, or one ulp off it
            h = F32(rng.integers(-127, 127) + 0.5)
            x = F32(h * sx)
            x = [x, np.nextafter(x, F32(np.inf)), np.nextafter(x, F32(-np.inf))][rng.integers(0, 3)]
        else:            # tiny against the scale
            x = F32(rng.uniform(-1, 1)) * F32(sx) * F32(2.0 ** -int(rng.integers(1, 60)))
        out.append((F32(x), sx))
    return out


@pytest.mark.parametrize("seed", [0, 1])
def test_recipe_equals_rounded_division(seed):
    rng = np.random.default_rng(seed)
    for x, sx in _cases(rng, 1500):
        assert quant_recipe(x, sx) == quant_reference(x, sx), (float(x), float(sx))
