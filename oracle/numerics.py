"""Exact number-format helpers for the oracle (float64 throughout).

TEST INFRASTRUCTURE ONLY (see the package docstring).

bf16 is carried as its raw 16-bit pattern in ``numpy.uint16`` arrays because
numpy has no bf16 type.  A bf16 value is the upper half of an IEEE binary32
pattern, so widening is exact.  Rounding goes straight from float64 to the bf16
grid with ties to even; it never passes through float32, which would round
twice.
"""

import numpy as np

BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def bf16_bits_to_f64(bits):
    """Widen bf16 bit patterns (uint16) to float64 exactly."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):   # signalling-NaN patterns widen to NaN
        return u.view(np.float32).astype(np.float64)


def round_bf16(x):
    """Round float64 values to the nearest bf16 value, ties to even.

    bf16 keeps 8 significant bits (1 implicit + 7 stored) and float32's exponent
    range.  A normal value x = m * 2**e with 0.5 <= |m| < 1 lands on the grid of
    spacing 2**(e-8); below 2**-126 the grid spacing is fixed at 2**-133.
    ``np.rint`` rounds half to even, and the scaled values are exact in float64.
    Results above the largest finite bf16 become +-inf.  Returns float64.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    normal = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
    tiny = np.ldexp(np.rint(np.ldexp(x, 133)), -133)
    r = np.where(e >= -125, normal, tiny)
    return np.where(np.abs(r) > BF16_MAX, np.copysign(np.inf, x), r)


def f64_to_bf16_bits(x):
    """Round float64 values to bf16 (ties to even) and return the bit patterns."""
    r = round_bf16(x).astype(np.float32)  # exact: r is already on the bf16 grid
    return (r.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def round_f32(x):
    """Round float64 values to float32 (numpy rounds to nearest even), as float64."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def as_f64(w):
    """A weight given either as bf16 bits (uint16) or as real numbers, as float64."""
    w = np.asarray(w)
    if w.dtype == np.uint16:
        return bf16_bits_to_f64(w)
    return w.astype(np.float64)
