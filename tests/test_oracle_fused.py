"""Pins of the oracle's verification from hidden states (target_logits_from_hidden,
spec_verify_fused) against things other than itself: a one-hot hidden state
picks one column of the head exactly, the map is linear, an element-by-element
loop gives the same logits, and the verification equals spec_verify on logits
formed independently."""

import math

import numpy as np
import pytest

from mtp_speculative_decoding_draft_gb300 import workloads as W
from oracle.numerics import bf16_bits_to_f64
from oracle.sampling import softmax_T
from oracle.verify import spec_verify, spec_verify_fused, target_logits_from_hidden

GREEDY, STOCH = 0, 1


def _bf16(x):
    return W.to_bf16_bits(np.asarray(x, np.float32))


def test_one_hot_hidden_gives_one_column_of_the_head():
    rng = np.random.default_rng(11)
    V, d = 37, 12                     # V != d: a transposed head would not even fit
    head = _bf16(rng.standard_normal((V, d)) * 0.02)
    hf = bf16_bits_to_f64(head)
    for i in (0, 5, d - 1):
        for c in (1.0, -0.375, 3.5):  # products of bf16 values are exact in float64
            h = np.zeros((1, d))
            h[0, i] = c
            t = target_logits_from_hidden(head, h)
            assert t.shape == (1, V)
            assert np.array_equal(t[0], c * hf[:, i])


def test_linear_in_the_hidden_state():
    rng = np.random.default_rng(12)
    V, d = 101, 24
    head = _bf16(rng.standard_normal((V, d)) * 0.02)
    h1 = rng.standard_normal((3, d))
    h2 = rng.standard_normal((3, d))
    a = target_logits_from_hidden(head, h1 + 2.0 * h2)
    b = target_logits_from_hidden(head, h1) + 2.0 * target_logits_from_hidden(head, h2)
    assert np.max(np.abs(a - b)) <= 1e-12 * np.max(np.abs(a))


def test_matches_an_element_by_element_loop():
    rng = np.random.default_rng(13)
    V, d = 9, 7
    head = _bf16(rng.standard_normal((V, d)) * 0.02)
    hidden = _bf16(rng.standard_normal((2, 2, d)))
    hf, xf = bf16_bits_to_f64(head), bf16_bits_to_f64(hidden)
    t = target_logits_from_hidden(head, hidden)
    assert t.shape == (2, 2, V)
    for b in range(2):
        for j in range(2):
            for v in range(V):
                want = math.fsum(float(hf[v, i]) * float(xf[b, j, i]) for i in range(d))
                assert abs(t[b, j, v] - want) <= 1e-15 * max(1.0, abs(want))


@pytest.mark.parametrize("mode", [GREEDY, STOCH])
def test_fused_verification_equals_the_logits_path(mode):
    rng = np.random.default_rng(14)
    B, k, V, d, T = 6, 3, 211, 40, 0.8
    head = _bf16(rng.standard_normal((V, d)) * 0.3)
    hidden = _bf16(rng.standard_normal((B, k + 1, d)))
    # logits formed without the oracle's matmul: explicit sums per entry
    hf, xf = bf16_bits_to_f64(head), bf16_bits_to_f64(hidden)
    t = np.zeros((B, k + 1, V))
    for b in range(B):
        for j in range(k + 1):
            t[b, j] = [math.fsum(hf[v] * xf[b, j]) for v in range(V)]
    draft = t[:, :k] + rng.standard_normal((B, k, V)) * 0.7
    ua = rng.random((B, k))
    uf = rng.random(B)
    d = np.zeros((B, k), np.int64)
    for b in range(B):
        for j in range(k):
            d[b, j] = rng.choice(V, p=softmax_T(draft[b, j], T))
    got = spec_verify_fused(head, hidden, draft, d, mode, T, ua, uf)
    want = spec_verify(t, draft, d, mode, T, ua, uf)
    for g, w in zip(got, want):
        assert np.array_equal(g, w)
    # a subset of sequences gives those sequences' rows
    sub = spec_verify_fused(head, hidden, draft, d, mode, T, ua, uf, seqs=[4, 1])
    for g, w in zip(sub, want):
        assert np.array_equal(g, w[[4, 1]])
