"""Pins of the oracle's dynamic draft length: each sequence keeps the drafts
before its first depth whose draft confidence (the draft distribution's largest
probability) is below stop_p, and is verified over those drafts only, the bonus
row being the row after them.  ("Faster Rollouts with MTP Speculative
Decoding", section "What's Next", names dynamic draft length; the stopping rule
is this build's reading.)

The exactness pin: the stop decision depends on the draft distribution only, so
the emitted tokens must still follow the target's own distribution exactly.
That is checked by enumeration, as for the fixed-length rule.
"""

import itertools

import numpy as np
import pytest
import scipy.special

from oracle.block import GREEDY, STOCHASTIC, draft_confidence, dynamic_depths
from oracle.sampling import argmax_lowest, inverse_cdf, softmax_T
from oracle.verify import spec_verify, verify_stochastic_one


def test_confidence_is_the_largest_draft_probability():
    rng = np.random.default_rng(31)
    for _ in range(20):
        z = rng.standard_normal(50) * 3
        T = float(rng.uniform(0.3, 2.0))
        assert abs(draft_confidence(z, STOCHASTIC, T) - scipy.special.softmax(z / T).max()) < 1e-14
        assert abs(draft_confidence(z, GREEDY, T) - scipy.special.softmax(z).max()) < 1e-14
    assert draft_confidence(np.zeros(8), GREEDY, 1.0) == 1.0 / 8
    assert draft_confidence(np.array([0.0, -np.inf, -np.inf]), GREEDY, 1.0) == 1.0


def _rows_with_confidence(confs, V):
    """Logit rows whose largest softmax probability is confs[j]: one entry a,
    the other V - 1 at zero, e^a / (e^a + V - 1) = c."""
    rows = np.zeros((len(confs), V))
    for j, c in enumerate(confs):
        rows[j, j % V] = np.log(c * (V - 1) / (1 - c))
    return rows


def test_dynamic_depths_first_depth_below_the_threshold():
    V = 10
    dl = np.stack([_rows_with_confidence([0.9, 0.5, 0.8], V),     # stops at depth 1
                   _rows_with_confidence([0.2, 0.9, 0.9], V),     # stops at depth 0
                   _rows_with_confidence([0.9, 0.7, 0.61], V),    # keeps all three
                   _rows_with_confidence([0.9, 0.9, 0.55], V)])   # stops at depth 2
    assert list(dynamic_depths(dl, GREEDY, 1.0, 0.6)) == [1, 0, 3, 2]
    assert list(dynamic_depths(dl, GREEDY, 1.0, 0.0)) == [3, 3, 3, 3]   # never stops
    assert list(dynamic_depths(dl, GREEDY, 1.0, 1.01)) == [0, 0, 0, 0]  # always stops at once
    # stochastic: the confidence is taken at the temperature
    hot = dynamic_depths(dl, STOCHASTIC, 4.0, 0.6)
    assert list(hot) == [0, 0, 0, 0]


def test_verify_with_k_eff():
    rng = np.random.default_rng(32)
    B, k, V = 6, 3, 12
    target = rng.standard_normal((B, k + 1, V)) * 2
    draft = target[:, :k] + rng.standard_normal((B, k, V))
    d = np.array([[argmax_lowest(target[b, j]) for j in range(k)] for b in range(B)])
    ua = rng.random((B, k))
    uf = rng.random(B)
    for mode in (GREEDY, STOCHASTIC):
        full = spec_verify(target, draft, d, mode, 0.9, ua, uf)
        same = spec_verify(target, draft, d, mode, 0.9, ua, uf, k_eff=np.full(B, k))
        for x, y in zip(full, same):
            np.testing.assert_array_equal(x, y)
        out, alen, nacc = spec_verify(target, draft, d, mode, 0.9, ua, uf, k_eff=np.zeros(B, int))
        assert np.all(alen == 1) and np.all(nacc == 0) and np.all(out[:, 1:] == -1)
        for b in range(B):   # no draft kept: one ordinary decoding step on target row 0
            expect = argmax_lowest(target[b, 0]) if mode == GREEDY else \
                inverse_cdf(softmax_T(target[b, 0], 0.9), float(uf[b]))
            assert out[b, 0] == expect
    # greedy with matching drafts: every kept draft is accepted, the bonus is row k_eff
    ke = np.array([0, 1, 2, 3, 1, 2])
    out, alen, _ = spec_verify(target, draft, d, GREEDY, 1.0, k_eff=ke)
    for b in range(B):
        assert alen[b] == ke[b] + 1
        assert list(out[b, :ke[b]]) == list(d[b, :ke[b]])
        assert out[b, ke[b]] == argmax_lowest(target[b, ke[b]])


# ---------------------------------------------------------------- exactness by enumeration

def _dyadic(rng, V, unit_q, n_units):
    """As in test_oracle_verify: p on a 1/n_units grid, q a permutation of unit_q,
    residual mass a power of two in units (or zero)."""
    while True:
        p = rng.multinomial(n_units - V, rng.dirichlet(np.ones(V))) + 1
        q = rng.permutation(np.asarray(unit_q))
        s = int(np.maximum(p - q, 0).sum())
        if s == 0 or (s & (s - 1)) == 0:
            return p / n_units, q / n_units


def _exactness_dynamic(V, k, unit_qs, n_units, grid_n, T, stop_p, seed, bonus_row=None):
    """Emitted-sequence distribution of one speculative step with the dynamic
    stop, summed over every draft sequence and a midpoint grid of uniforms;
    its joint with the target's own continuation must equal the target's."""
    rng = np.random.default_rng(seed)
    P, Q = {}, {}
    for n in range(k + 1):
        for pre in itertools.product(range(V), repeat=n):
            # the first depth never stops, the later ones vary
            uq = unit_qs[0] if n == 0 else unit_qs[int(rng.integers(len(unit_qs)))]
            p, q = _dyadic(rng, V, uq, n_units)
            P[pre] = p
            if n < k:
                Q[pre] = q
    g = (np.arange(grid_n) + 0.5) / grid_n
    cell = 1.0 / grid_n ** (k + 1)
    spec, kept = {}, set()
    for d in itertools.product(range(V), repeat=k):
        wq = np.prod([Q[d[:j]][d[j]] for j in range(k)])
        target = np.stack([T * np.log(P[d[:j]]) for j in range(k + 1)])
        draft = np.stack([T * np.log(Q[d[:j]]) for j in range(k)])
        kb = int(dynamic_depths(draft[None], STOCHASTIC, T, stop_p)[0])
        kept.add(kb)
        tb = target[:kb + 1] if bonus_row is None else np.concatenate([target[:kb], target[bonus_row(kb):][:1]])
        for us in itertools.product(g, repeat=k + 1):
            out, a = verify_stochastic_one(tb, draft[:kb], d[:kb], us[:kb], us[k], T)
            assert len(out) == a + 1 and 0 <= a <= kb
            spec[tuple(out)] = spec.get(tuple(out), 0.0) + wq * cell
    assert abs(sum(spec.values()) - 1.0) < 1e-12
    for x in itertools.product(range(V), repeat=k + 1):
        p_target = np.prod([P[x[:j]][x[j]] for j in range(k + 1)])
        p_spec = 0.0
        for L in range(1, k + 2):
            e = x[:L]
            if e in spec:
                cont = np.prod([P[x[:j]][x[j]] for j in range(L, k + 1)]) if L <= k else 1.0
                p_spec += spec[e] * cont
        assert abs(p_spec - p_target) < 1e-12, (x, p_spec, p_target)
    return kept


# Draft rows with largest probability 1/2, 1/4 or 1 (every q dyadic, so every
# acceptance and CDF boundary falls on the 1/16 grid): stop_p = 0.3 stops at the
# 1/4 rows.  The first row decides whether depth 0 stops.
UNIT_QS = [[8, 4, 2, 2], [4, 4, 4, 4], [16, 0, 0, 0]]


@pytest.mark.parametrize("T", [1.0, 0.8])
def test_dynamic_stop_keeps_the_rule_exact(T):
    with np.errstate(divide="ignore"):
        kept = _exactness_dynamic(V=4, k=2, unit_qs=UNIT_QS, n_units=16, grid_n=16, T=T, stop_p=0.3,
                                  seed=41)
        assert kept == {1, 2}     # some draft paths stop after one draft, others keep two
        kept = _exactness_dynamic(V=4, k=2, unit_qs=[UNIT_QS[1]] + UNIT_QS, n_units=16, grid_n=16, T=T,
                                  stop_p=0.3, seed=43)
        assert kept == {0}        # the first depth already stops: a plain decoding step


def test_dynamic_exactness_check_detects_a_wrong_bonus_row():
    """Drawing the bonus token from row k instead of row k_eff breaks exactness."""
    with np.errstate(divide="ignore"), pytest.raises(AssertionError):
        _exactness_dynamic(V=4, k=2, unit_qs=UNIT_QS, n_units=16, grid_n=16, T=1.0, stop_p=0.3, seed=42,
                           bonus_row=lambda kb: 2)
