"""Pins for the oracle's number formats and sampling primitives.

Each check compares against something other than the oracle's own formula: a
library routine the oracle does not use, a closed form, or an exact integral.
"""

import numpy as np
import pytest
import scipy.special
import torch

from oracle.numerics import bf16_bits_to_f64, f64_to_bf16_bits, round_bf16, round_f32
from oracle.sampling import argmax_lowest, inverse_cdf, softmax_T


# ---------------------------------------------------------------- bf16

def test_bf16_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * np.float32(3.0),
        (rng.standard_normal(20000) * 1e-30).astype(np.float32),     # near the bottom of the range
        (rng.standard_normal(20000) * 1e37).astype(np.float32),      # near the top
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38], dtype=np.float32),
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = round_bf16(x.astype(np.float64))
    np.testing.assert_array_equal(got, ref)


def test_bf16_ties_to_even_and_no_double_rounding():
    one = 1.0
    # exact ties between two bf16 neighbours go to the even mantissa
    assert round_bf16(one + 2.0 ** -8) == one
    assert round_bf16(one + 3 * 2.0 ** -8) == one + 2 * 2.0 ** -7
    # just above a tie rounds up; rounding via float32 first would lose the 2^-30 and give 1.0
    assert round_bf16(one + 2.0 ** -8 + 2.0 ** -30) == one + 2.0 ** -7
    assert round_f32(one + 2.0 ** -8 + 2.0 ** -30) == one + 2.0 ** -8
    # overflow
    assert np.isinf(round_bf16(3.4e38))
    assert round_bf16(-(2 - 2 ** -7) * 2.0 ** 127) == -(2 - 2 ** -7) * 2.0 ** 127


def test_bf16_bits_roundtrip():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = bf16_bits_to_f64(bits)
    finite = np.isfinite(vals)
    back = f64_to_bf16_bits(vals[finite])
    np.testing.assert_array_equal(back, bits[finite])
    # widening agrees with torch's bf16 -> float conversion
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(vals[finite], t[finite])


# ---------------------------------------------------------------- softmax / argmax

@pytest.mark.parametrize("T", [1.0, 0.7, 2.5])
def test_softmax_matches_scipy(T):
    rng = np.random.default_rng(1)
    z = rng.standard_normal(5000) * 4.0
    p = softmax_T(z, T)
    np.testing.assert_allclose(p, scipy.special.softmax(z / T), rtol=1e-12, atol=0)
    assert abs(p.sum() - 1.0) < 1e-12


def test_softmax_extreme_logits():
    z = np.array([1000.0, 0.0, -np.inf, 999.0])
    p = softmax_T(z, 1.0)
    assert p[2] == 0.0 and abs(p.sum() - 1.0) < 1e-15
    assert p[0] == pytest.approx(1.0 / (1.0 + np.exp(-1.0)), rel=1e-14)


def test_argmax_lowest_index_on_ties():
    assert argmax_lowest([0.0, 3.0, 1.0, 3.0]) == 1
    assert argmax_lowest([5.0, 5.0, 5.0]) == 0
    assert argmax_lowest([-np.inf, -1.0, -1.0]) == 1
    rng = np.random.default_rng(2)
    for _ in range(200):
        z = rng.integers(0, 4, size=13).astype(float)
        m = max(z)
        assert argmax_lowest(z) == min(i for i, v in enumerate(z) if v == m)


# ---------------------------------------------------------------- inverse CDF

def _grid(n):
    return (np.arange(n) + 0.5) / n


def test_inverse_cdf_exact_selection_probabilities():
    """Over u ~ U[0,1) index i must be chosen with probability exactly w_i / S.

    With weights that are integer multiples of S/n, every CDF boundary sits on a
    multiple of 1/n, so the n-point midpoint grid integrates the selection
    exactly (no grid cell straddles a boundary)."""
    rng = np.random.default_rng(4)
    n = 64
    for _ in range(50):
        V = int(rng.integers(1, 12))
        units = rng.multinomial(n, rng.dirichlet(np.ones(V)))
        scale = float(rng.choice([1.0, 3.0, 1e-3]))
        w = units * scale
        counts = np.zeros(V)
        for u in _grid(n):
            counts[inverse_cdf(w, u)] += 1
        np.testing.assert_array_equal(counts, units)


def test_inverse_cdf_edges():
    w = np.array([0.0, 0.0, 2.0, 0.0, 1.0, 0.0])
    assert inverse_cdf(w, 0.0) == 2                     # first positive weight
    assert inverse_cdf(w, np.nextafter(1.0, 0.0)) == 4  # never a zero-weight index
    assert inverse_cdf(w, 2.0 / 3.0) == 4               # C_i > u*S is strict
    assert inverse_cdf(w, 0.6666) == 2
    # u = 1 is outside U[0,1): the fallback still returns the last positive index
    assert inverse_cdf(w, 1.0) == 4


def test_inverse_cdf_against_sorted_search():
    """Brute force: the chosen index is the first whose running sum passes u*S."""
    rng = np.random.default_rng(5)
    w = rng.random(1000) ** 3
    total = 0.0
    for x in w:                          # explicit running total, index order
        total += x
    for u in rng.random(200):
        run = 0.0
        for j, x in enumerate(w):
            run += x
            if run > u * total:
                break
        assert inverse_cdf(w, u) == j
