"""Pins for the oracle's verification rule.

* Greedy: the emitted tokens equal plain greedy decoding of the same target
  ("The Tiny Draft Model Hidden Inside Qwen", section "How the draft becomes real
  output").
* Stochastic: the distribution of what one speculative step emits, completed by
  the target itself, equals the target's own autoregressive distribution exactly
  ("Speculative Decoding and MTP: Why Guessing Is Free", section "It's exact, not
  approximate").  The check integrates the oracle's uniform-driven functions
  exactly: all probabilities are dyadic, so every decision boundary falls on the
  midpoint grid's cell edges and the grid sum is the exact integral.
"""

import itertools

import numpy as np
import pytest

from oracle.block import GREEDY, STOCHASTIC, select_token
from oracle.sampling import softmax_T
from oracle.verify import (residual, spec_verify, verify_greedy_one,
                           verify_stochastic_one)


def _grid(n):
    return (np.arange(n) + 0.5) / n


# ---------------------------------------------------------------- greedy

def _plain_greedy(table, k):
    """Ordinary greedy decoding of a target given as prefix -> logits."""
    seq = []
    for _ in range(k + 1):
        z = table[tuple(seq)]
        best = 0
        for i in range(1, len(z)):          # explicit scan, lowest index on ties
            if z[i] > z[best]:
                best = i
        seq.append(best)
    return seq


def test_greedy_equals_plain_greedy():
    rng = np.random.default_rng(11)
    V, k = 5, 3
    for trial in range(300):
        table = {}
        for n in range(k + 1):
            for pre in itertools.product(range(V), repeat=n):
                z = rng.integers(0, 4, size=V).astype(float) if trial % 3 == 0 else rng.standard_normal(V)
                table[pre] = z                 # trial % 3 == 0 has many exact ties
        plain = _plain_greedy(table, k)
        # drafts: mostly right guesses, sometimes wrong
        d = [plain[j] if rng.random() < 0.7 else int(rng.integers(0, V)) for j in range(k)]
        rows = np.stack([table[tuple(d[:j])] for j in range(k + 1)])
        out, a = verify_greedy_one(rows, d)
        expect_a = 0
        while expect_a < k and d[expect_a] == plain[expect_a]:
            expect_a += 1
        assert a == expect_a
        assert out == plain[:a + 1]


# ---------------------------------------------------------------- stochastic exactness

def _dyadic_pair(rng, V, unit_q, n_units):
    """Target p (multiples of 1/n_units, all positive) and draft q (a permutation
    of unit_q / n_units) such that the residual mass sum max(0, p - q) is a power
    of two in units (or zero): then p/q and every residual CDF point are dyadic."""
    while True:
        p = rng.multinomial(n_units - V, rng.dirichlet(np.ones(V))) + 1
        q = rng.permutation(np.asarray(unit_q))
        s = int(np.maximum(p - q, 0).sum())
        if s == 0 or (s & (s - 1)) == 0:
            return p / n_units, q / n_units


def _exactness_check(V, k, unit_q, n_units, grid_n, T, seed, verify_fn=None):
    verify_fn = verify_fn or verify_stochastic_one
    rng = np.random.default_rng(seed)
    P, Q = {}, {}
    for n in range(k + 1):
        for pre in itertools.product(range(V), repeat=n):
            p, q = _dyadic_pair(rng, V, unit_q, n_units)
            P[pre] = p
            if n < k:
                Q[pre] = q
    # emitted-sequence distribution of one speculative step
    spec = {}
    g = _grid(grid_n)
    cell = 1.0 / grid_n ** (k + 1)
    for d in itertools.product(range(V), repeat=k):
        wq = np.prod([Q[d[:j]][d[j]] for j in range(k)])
        target = np.stack([T * np.log(P[d[:j]]) for j in range(k + 1)])
        draft = np.stack([T * np.log(Q[d[:j]]) for j in range(k)])
        for us in itertools.product(g, repeat=k + 1):
            out, a = verify_fn(target, draft, d, us[:k], us[k], T)
            assert len(out) == a + 1 and 0 <= a <= k
            key = tuple(out)
            spec[key] = spec.get(key, 0.0) + wq * cell
    assert abs(sum(spec.values()) - 1.0) < 1e-12
    # complete each emission with the target's own continuation and compare joints
    for x in itertools.product(range(V), repeat=k + 1):
        p_target = np.prod([P[x[:j]][x[j]] for j in range(k + 1)])
        p_spec = 0.0
        for L in range(1, k + 2):
            e = x[:L]
            if e in spec:
                cont = np.prod([P[x[:j]][x[j]] for j in range(L, k + 1)]) if L <= k else 1.0
                p_spec += spec[e] * cont
        assert abs(p_spec - p_target) < 1e-12, (x, p_spec, p_target)
    return spec


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_stochastic_rule_is_exact_V4_k2(T):
    # q in {1/2, 1/4, 1/8, 1/8}, p in multiples of 1/16: boundaries on multiples of 1/16
    _exactness_check(V=4, k=2, unit_q=[8, 4, 2, 2], n_units=16, grid_n=16, T=T, seed=21)


def test_stochastic_rule_is_exact_V8_k1():
    # q in {1/4,1/4,1/8,1/8,1/16 x4}, p in multiples of 1/32: boundaries on multiples of 1/32
    _exactness_check(V=8, k=1, unit_q=[8, 8, 4, 4, 2, 2, 2, 2], n_units=32, grid_n=32, T=1.0, seed=22)


def test_exactness_check_detects_a_planted_mistake(monkeypatch):
    """The exactness check must fail if the residual is replaced by max(0, q - p)."""
    import oracle.verify as ov
    monkeypatch.setattr(ov, "residual", lambda p, q: np.maximum(np.asarray(q) - np.asarray(p), 0.0))
    with pytest.raises(AssertionError):
        _exactness_check(V=4, k=1, unit_q=[8, 4, 2, 2], n_units=16, grid_n=16, T=1.0, seed=23)


def test_exactness_check_detects_wrong_bonus_row():
    """... and if the bonus token were drawn from the previous position's row."""
    def wrong(target, draft, draft_tok, u_accept, u_final, T):
        t = np.array(target, copy=True)
        t[-1] = t[-2]
        return verify_stochastic_one(t, draft, draft_tok, u_accept, u_final, T)

    with pytest.raises(AssertionError):
        _exactness_check(V=4, k=1, unit_q=[8, 4, 2, 2], n_units=16, grid_n=16, T=1.0, seed=24,
                         verify_fn=wrong)


def test_exactness_check_detects_swapped_p_and_q():
    """... and if the roles of target and draft were swapped."""
    def wrong(target, draft, draft_tok, u_accept, u_final, T):
        return verify_stochastic_one(draft.tolist() + [target[-1]], target[:-1], draft_tok,
                                     u_accept, u_final, T)

    with pytest.raises(AssertionError):
        _exactness_check(V=4, k=1, unit_q=[8, 4, 2, 2], n_units=16, grid_n=16, T=1.0, seed=25,
                         verify_fn=wrong)


# ---------------------------------------------------------------- special cases

def test_draft_sampling_selects_with_draft_probabilities():
    """select_token over u ~ U[0,1) picks i with probability exactly q_i."""
    q = np.array([8, 4, 2, 1, 1]) / 16.0
    for T in (1.0, 0.7):
        z = T * np.log(q)
        counts = np.zeros(5)
        for u in _grid(16):
            counts[select_token(z, STOCHASTIC, T, u)] += 1
        np.testing.assert_array_equal(counts / 16.0, q)


def test_identical_distributions_always_accept():
    rng = np.random.default_rng(31)
    V, k = 50, 3
    for _ in range(50):
        t = rng.standard_normal((k + 1, V)) * 4
        d = rng.integers(0, V, size=k)
        u = rng.random(k)
        out, a = verify_stochastic_one(t, t[:k], d, u, 0.3, 1.0)
        assert a == k and out[:k] == list(d)


def test_one_hot_draft_accepts_with_target_probability():
    """q concentrated on the draft token d: acceptance probability is p(d)."""
    p = np.array([3, 5, 7, 1]) / 16.0
    t = np.log(p)[None, :].repeat(2, axis=0)
    for d in range(4):
        l = np.full((1, 4), -1e4)
        l[0, d] = 0.0
        acc = 0
        for u in _grid(16):
            _, a = verify_stochastic_one(t, l, [d], [u], 0.5, 1.0)
            acc += a
        assert acc / 16.0 == p[d]


def test_zero_residual_falls_back_to_target():
    """If p == q the residual is identically zero; a forced rejection draws from p."""
    p = np.array([1, 2, 5]) / 8.0
    t = np.log(p)[None, :].repeat(2, axis=0)
    counts = np.zeros(3)
    for uf in _grid(8):
        out, a = verify_stochastic_one(t, t[:1], [0], [1.0], uf, 1.0)  # u = 1 forces the reject
        assert a == 0
        counts[out[0]] += 1
    np.testing.assert_array_equal(counts / 8.0, p)


def test_residual_mass_is_total_variation():
    rng = np.random.default_rng(41)
    for _ in range(100):
        p = softmax_T(rng.standard_normal(300) * 3, 1.0)
        q = softmax_T(rng.standard_normal(300) * 3, 1.0)
        R = residual(p, q)
        assert abs(R.sum() - (1.0 - np.minimum(p, q).sum())) < 1e-12
        assert abs((R / R.sum()).sum() - 1.0) < 1e-12
        np.testing.assert_array_equal(R > 0, p > q)


def test_low_temperature_reduces_to_greedy():
    rng = np.random.default_rng(51)
    V, k, T = 40, 3, 1e-3
    for _ in range(100):
        t = rng.permutation(V)[None, :].repeat(k + 1, 0) * 0.1 + rng.standard_normal((k + 1, V)) * 0.01
        for j in range(k + 1):
            t[j] = rng.permutation(V) * 0.1
        l = np.stack([rng.permutation(V) * 0.1 for _ in range(k)])
        d = [int(np.argmax(l[j])) for j in range(k)]
        # make some drafts agree with the target's argmax
        for j in range(k):
            if rng.random() < 0.6:
                l[j, d[j]], l[j, int(np.argmax(t[j]))] = l[j, int(np.argmax(t[j]))], l[j, d[j]]
                d[j] = int(np.argmax(l[j]))
        g_out, g_a = verify_greedy_one(t, d)
        s_out, s_a = verify_stochastic_one(t, l, d, rng.random(k), float(rng.random()), T)
        assert (g_out, g_a) == (s_out, s_a)


def test_high_temperature_reduces_to_uniform():
    """As T grows, p_j and q_j both tend to 1/V, so p(d)/q(d) -> 1: every draft
    with u < 1 - O(1/T) is accepted and the bonus token is the uniform draw
    floor(u V) of the inverse CDF."""
    rng = np.random.default_rng(52)
    V, k, T = 257, 4, 1e9
    for _ in range(100):
        t = rng.standard_normal((k + 1, V)) * 5
        l = rng.standard_normal((k, V)) * 5
        d = [int(x) for x in rng.integers(0, V, size=k)]
        ua = rng.random(k) * 0.999
        uf = float(rng.random())
        if abs(uf * V - round(uf * V)) < 1e-6:
            continue
        out, a = verify_stochastic_one(t, l, d, ua, uf, T)
        assert a == k and out[:k] == d
        assert out[k] == int(np.floor(uf * V))


def test_batched_outputs_bounds_and_padding():
    rng = np.random.default_rng(61)
    B, k, V = 40, 4, 300
    t = rng.standard_normal((B, k + 1, V)).astype(np.float32) * 4
    l = (t[:, :k] + rng.standard_normal((B, k, V)).astype(np.float32) * 1.5)
    d = rng.integers(0, V, size=(B, k))
    for mode in (GREEDY, STOCHASTIC):
        out, L, a = spec_verify(t, l, d, mode, 1.0, rng.random((B, k)), rng.random(B))
        assert np.all((L >= 1) & (L <= k + 1)) and np.all(a == L - 1)
        for b in range(B):
            assert np.all(out[b, :L[b]] >= 0) and np.all(out[b, L[b]:] == -1)
            assert list(out[b, :a[b]]) == list(d[b, :a[b]])


def test_accept_threshold_bisection_recovers_p_over_q():
    """The bisection the GPU test reads the verifier's probabilities with:
    on the oracle's own decisions it finds V * p(d) for a constant draft row."""
    from parity_helpers import accept_threshold_bisection, constant_draft_ratio_case
    B, V, T = 6, 997, 0.8
    t, draft, d, ratio = constant_draft_ratio_case(B, V, T, seed=4402)
    uf = np.full(B, 0.5, np.float32)
    lo, hi = accept_threshold_bisection(
        lambda u: spec_verify(t, draft, d, STOCHASTIC, T, u[:, None], uf)[2] >= 1, B)
    assert np.all(ratio < 1.0)
    assert np.all((lo <= ratio * (1 + 1e-7)) & (ratio <= hi * (1 + 1e-7)))
    assert np.all((hi - lo) <= 1e-8 + 2e-7 * ratio)
