"""GPU parity of stochastic verification on both of its kernels.

Stochastic spec_verify runs on the streaming kernel (one CTA per chunk of
32768 logits; the CTA that completes a sequence decides and draws) unless
MTP_VERIFY_SPLIT=0 selects the cluster kernel.  The main verify tests run the
default; here the cluster kernel gets the same stochastic checks, and both
get vocabularies that span several 32768-element chunks with ragged tails,
unaligned rows and a one-element last chunk."""

import numpy as np
import pytest

from mtp_speculative_decoding_draft_gb300 import workloads as W
from oracle.sampling import softmax_T
from oracle.verify import spec_verify as oracle_verify
from parity_helpers import SAMPLE_BAND, cdf_margin, check_excused
from test_gpu_verify import STOCH, _case, _check, _draft_tokens_from_q, _run

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["split", "cluster"])
def kernel(request, monkeypatch):
    monkeypatch.setenv("MTP_VERIFY_SPLIT", "1" if request.param == "split" else "0")  # read at every call
    return request.param


@pytest.mark.parametrize("B,k,V,T", [(7, 3, 2 * 32768 + 5, 0.9),   # odd V: unaligned rows, ragged tail
                                     (3, 2, 3 * 32768, 1.0),       # whole chunks only
                                     (5, 4, 32768 + 1, 1.2),       # a one-element last chunk
                                     (6, 3, 3 * 8192 + 4, 1.1),    # a 4-logit tail
                                     (37, 3, 5003, 1.0),           # one ragged chunk
                                     (40, 2, 5004, 0.8),           # aligned rows below one chunk
                                     (3, 8, 777, 1.0)])            # the deepest draft
def test_stochastic_multi_chunk(kernel, B, k, V, T):
    t, l, d, ua, uf = _case(B, k, V, T, seed=7700 + B * 10 + k)
    exc, L = _check(t, l, d, ua, uf, STOCH, T)
    assert L.min() >= 1


def test_stochastic_everything_accepted(kernel):
    """draft == target: every draft is accepted, so the bonus draw (from the
    chunk statistics, then one chunk's sub-chunks) makes every emitted token."""
    rng = np.random.default_rng(77)
    B, k, V = 12, 3, 2 * 32768 + 1000
    t = (rng.standard_normal((B, k + 1, V)) * 3).astype(np.float32)
    d = rng.integers(0, V, size=(B, k)).astype(np.int32)
    ua = rng.random((B, k)).astype(np.float32)
    uf = rng.random(B).astype(np.float32)
    exc, L = _check(t, t[:, :k].copy(), d, ua, uf, STOCH, 1.0)
    assert np.all(L == k + 1)


def test_stochastic_sweep_k3_full_size(kernel):
    w = W.with_k(W.VERIFY_SWEEP, 3)
    inp = W.verify_inputs(w)
    d = _draft_tokens_from_q(inp["draft_logits"], inp["u_draft"], w.T)
    exc, L = _check(inp["target_logits"], inp["draft_logits"], d, inp["u_accept"], inp["u_final"], STOCH, w.T)
    print("%s kernel: mean accepted length %.3f, excused %d" % (kernel, L.mean(), exc))


def test_stochastic_residual_zero_draws_from_p(kernel):
    """Identical target and draft rows, with the same masked (-inf) entries,
    and a draft token at a masked position: p(d) = q(d) = 0, so u q(d) < p(d)
    fails and the position rejects, while max(0, p - q) is zero everywhere.
    The rule then draws from p itself, as the oracle does."""
    rng = np.random.default_rng(78)
    B, k, V = 6, 2, 3 * 8192 + 4
    t = (rng.standard_normal((B, k + 1, V)) * 3).astype(np.float32)
    mask = rng.random(V) < 0.05
    t[:, :, mask] = -np.inf
    masked = np.nonzero(mask)[0]
    l = t[:, :k].copy()
    d = np.array([[int(rng.choice(masked)) if j == 0 else int(rng.integers(0, V)) for j in range(k)]
                  for _ in range(B)], np.int32)
    ua = rng.random((B, k)).astype(np.float32)
    uf = rng.random(B).astype(np.float32)
    exc, L = _check(t, l, d, ua, uf, STOCH, 1.0)
    assert np.all(L == 1)   # every sequence rejects its first draft


@pytest.mark.parametrize("T", [0.05, 20.0])
def test_stochastic_temperature_extremes(kernel, T):
    """Near one-hot (T = 0.05: scaled logits spread over hundreds, most exp2
    terms underflow) and near uniform (T = 20: p and q differ by a few percent,
    so the residual max(0, p - q) is a small difference of close values) over
    a vocabulary of three sub-chunk groups and a 4-logit tail."""
    t, l, d, ua, uf = _case(24, 3, 3 * 8192 + 4, T, seed=7800 + int(T * 10))
    exc, L = _check(t, l, d, ua, uf, STOCH, T)
    print("%s kernel T=%g: mean accepted length %.3f, excused %d" % (kernel, T, L.mean(), exc))


def _equal_rows_case(B, k, V, seed):
    """Draft rows equal to the target rows: p = q at every position, so that
    u q(d) < p(d) holds exactly when u < 1."""
    rng = np.random.default_rng(seed)
    t = (rng.standard_normal((B, k + 1, V)) * 3).astype(np.float32)
    d = rng.integers(0, V, size=(B, k)).astype(np.int32)
    ua = np.full((B, k), 0.5, np.float32)
    uf = rng.random(B).astype(np.float32)
    return t, t[:, :k].copy(), d, ua, uf


def _check_draws_from_p(g, o, t, uf):
    """Outputs equal to the oracle's, the last emitted token (every draw here is
    from p of row L - 1: a bonus draw, or a residual that is zero) allowed to
    differ only within the CDF band."""
    g_out, g_len, g_acc = g
    o_out, o_len, o_acc = o
    assert np.array_equal(g_len, o_len) and np.array_equal(g_acc, o_acc)
    exc = 0
    for b in range(len(g_len)):
        L = int(g_len[b])
        assert list(g_out[b, :L - 1]) == list(o_out[b, :L - 1]) and np.all(g_out[b, L:] == -1)
        if g_out[b, L - 1] != o_out[b, L - 1]:
            margin = cdf_margin(softmax_T(t[b, L - 1].astype(np.float64), 1.0), float(uf[b]))
            assert margin < SAMPLE_BAND, "sequence %d: draw differs, CDF margin %.3g" % (b, margin)
            exc += 1
    check_excused(exc, len(g_len), "draws from p")


def test_stochastic_out_of_range_tokens(kernel):
    """A draft token outside [0, V) is never accepted: the position is rejected
    and its replacement drawn as after any rejection -- here, with p = q, from p
    itself.  The oracle defines no such token, so the expected outputs are the
    oracle's on the same rows with a valid token there and u_accept = 1, which
    rejects when p = q."""
    from mtp_speculative_decoding_draft_gb300 import binding as bd
    B, k, V = 5, 3, 3 * 8192 + 4
    t, l, d, ua, uf = _equal_rows_case(B, k, V, seed=7900)
    bad = {(0, 1): V + 5, (1, 0): -3, (3, 2): V}
    for (b, j), v in bad.items():
        d[b, j] = v
    g, st = _run(t, l, d, ua, uf, STOCH, 1.0)
    assert st & bd.STATUS_BAD_TOKEN and not st & bd.STATUS_NONFINITE
    d2, ua2 = d.copy(), ua.copy()
    for (b, j) in bad:
        d2[b, j] = 0
        ua2[b, j] = 1.0
    o = oracle_verify(t, l, d2, STOCH, 1.0, ua2, uf)
    _check_draws_from_p(g, o, t, uf)
    assert list(g[1]) == [2, 1, 4, 3, 4]


def test_stochastic_nonfinite_row_sets_status(kernel):
    """A target row with no finite logit: p is undefined there, the position is
    rejected with a token in range and the status word says so; the other
    sequences are unaffected."""
    from mtp_speculative_decoding_draft_gb300 import binding as bd
    B, k, V = 4, 3, 2 * 8192 + 100
    t, l, d, ua, uf = _equal_rows_case(B, k, V, seed=7901)
    t[0, 1, :] = -np.inf
    (g_out, g_len, g_acc), st = _run(t, l, d, ua, uf, STOCH, 1.0)
    assert st & bd.STATUS_NONFINITE
    assert g_len[0] == 2 and g_acc[0] == 1 and 0 <= g_out[0, 1] < V and g_out[0, 0] == d[0, 0]
    o = oracle_verify(t[1:], l[1:], d[1:], STOCH, 1.0, ua[1:], uf[1:])
    _check_draws_from_p((g_out[1:], g_len[1:], g_acc[1:]), o, t[1:], uf[1:])
