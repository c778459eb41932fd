"""GPU parity of spec_verify against the oracle (called through the C ABI)."""

import numpy as np
import pytest
import torch

from mtp_speculative_decoding_draft_gb300 import workloads as W
from mtp_speculative_decoding_draft_gb300.model import Verifier, to_device
from oracle.block import select_token
from oracle.verify import spec_verify as oracle_verify
from parity_helpers import accept_threshold_bisection, check_excused, compare_verify, constant_draft_ratio_case

pytestmark = pytest.mark.gpu

GREEDY, STOCH = 0, 1


def _draft_tokens_from_q(draft, u, T):
    """Drafts drawn from q = softmax(draft / T) with the oracle's sampler."""
    B, k, _ = draft.shape
    return np.array([[select_token(draft[b, j], STOCH, T, float(u[b, j])) for j in range(k)]
                     for b in range(B)], dtype=np.int32)


def _run(target, draft, d, ua, uf, mode, T):
    B, k1, V = target.shape
    k = k1 - 1
    ver = Verifier(B, k, V)
    ver(T, mode, to_device(target), to_device(draft) if draft is not None else None, to_device(d),
        to_device(ua) if ua is not None else None, to_device(uf) if uf is not None else None)
    res = ver.results()
    ver.check_canaries()
    from mtp_speculative_decoding_draft_gb300 import binding as bd
    st = bd.get_status(ver.ws)
    return res, st


def _case(B, k, V, T, seed, target_std=4.0, noise=1.5):
    w = W.Workload("verify_case", B=B, k=k, V=V, T=T, target_std=target_std, draft_noise_std0=noise,
                   verify_only=True, seed=seed)
    inp = W.verify_inputs(w)
    d = _draft_tokens_from_q(inp["draft_logits"], inp["u_draft"], T)
    return inp["target_logits"], inp["draft_logits"], d, inp["u_accept"], inp["u_final"]


def _check(target, draft, d, ua, uf, mode, T):
    (g_out, g_len, g_acc), st = _run(target, draft if mode == STOCH else None, d, ua, uf, mode, T)
    assert st == 0, "status word %d" % st
    o = oracle_verify(target, draft, d, mode, T, ua, uf)
    exc = compare_verify((g_out, g_len, g_acc), o, mode, target, draft, d, ua, uf, T)
    check_excused(exc, target.shape[0], "verify outputs")
    assert np.all((g_len >= 1) & (g_len <= d.shape[1] + 1)) and np.all(g_acc == g_len - 1)
    return exc, g_len


@pytest.mark.parametrize("mode", [GREEDY, STOCH])
def test_tiny_vocab_1000(mode):
    t, l, d, ua, uf = _case(B=1, k=3, V=1000, T=1.0, seed=1001, noise=1.0)
    _check(t, l, d, ua, uf, mode, 1.0)


@pytest.mark.parametrize("mode", [GREEDY, STOCH])
@pytest.mark.parametrize("B,k,V,T", [(37, 3, 5003, 1.0), (5, 1, 20011, 0.7), (64, 5, 4099, 1.3),
                                     (3, 8, 777, 1.0), (300, 2, 1024, 1.0)])
def test_ragged_shapes(mode, B, k, V, T):
    t, l, d, ua, uf = _case(B, k, V, T, seed=7000 + B * 10 + k)
    _check(t, l, d, ua, uf, mode, T)


@pytest.mark.parametrize("k", [1, 2, 3, 4, 5])
def test_verify_sweep_full_size(k):
    w = W.with_k(W.VERIFY_SWEEP, k)
    inp = W.verify_inputs(w)
    d = _draft_tokens_from_q(inp["draft_logits"][:, :, :], inp["u_draft"], w.T)
    exc_s, L = _check(inp["target_logits"], inp["draft_logits"], d, inp["u_accept"], inp["u_final"], STOCH, w.T)
    _check(inp["target_logits"], inp["draft_logits"], d, inp["u_accept"], inp["u_final"], GREEDY, w.T)
    print("k=%d stochastic: mean accepted length %.3f, excused %d" % (k, L.mean(), exc_s))


def test_degenerate_cases():
    rng = np.random.default_rng(5)
    # V = 1: every token is 0, everything is accepted
    t = np.zeros((4, 3, 1), np.float32)
    d = np.zeros((4, 2), np.int32)
    ua = rng.random((4, 2)).astype(np.float32)
    uf = rng.random(4).astype(np.float32)
    for mode in (GREEDY, STOCH):
        _check(t, t[:, :2].copy(), d, ua, uf, mode, 1.0)
    # V smaller than the cluster's slices: most CTAs own nothing
    t, l, d, ua, uf = _case(B=2, k=3, V=3, T=1.0, seed=5)
    for mode in (GREEDY, STOCH):
        _check(t, l, d, ua, uf, mode, 1.0)


def test_ties_lowest_index_and_identical_draft():
    rng = np.random.default_rng(6)
    B, k, V = 16, 4, 3001
    t = rng.integers(0, 3, size=(B, k + 1, V)).astype(np.float32)    # many exact ties at the max
    d = np.array([[int(np.argmax(t[b, j])) if rng.random() < 0.7 else int(rng.integers(0, V))
                   for j in range(k)] for b in range(B)], np.int32)
    ua = rng.random((B, k)).astype(np.float32)
    uf = rng.random(B).astype(np.float32)
    _check(t, None, d, ua, uf, GREEDY, 1.0)
    # draft == target: every draft accepted, the bonus comes from the last row
    t2 = (rng.standard_normal((B, k + 1, V)) * 4).astype(np.float32)
    d2 = rng.integers(0, V, size=(B, k)).astype(np.int32)
    exc, L = _check(t2, t2[:, :k].copy(), d2, ua, uf, STOCH, 1.0)
    assert np.all(L == k + 1)


def test_minus_infinity_logits():
    rng = np.random.default_rng(8)
    B, k, V = 8, 3, 2050
    t = (rng.standard_normal((B, k + 1, V)) * 3).astype(np.float32)
    l = (t[:, :k] + rng.standard_normal((B, k, V)).astype(np.float32))
    t[rng.random(t.shape) < 0.3] = -np.inf          # masked vocabulary entries
    l[rng.random(l.shape) < 0.3] = -np.inf
    for b in range(B):
        for j in range(k + 1):
            t[b, j, rng.integers(0, V)] = 1.0       # at least one finite entry per row
        for j in range(k):
            l[b, j, rng.integers(0, V)] = 1.0
    u = rng.random((B, k)).astype(np.float32)
    d = _draft_tokens_from_q(l, u, 1.0)
    ua = rng.random((B, k)).astype(np.float32)
    uf = rng.random(B).astype(np.float32)
    for mode in (GREEDY, STOCH):
        _check(t, l, d, ua, uf, mode, 1.0)


def test_invalid_arguments_are_rejected():
    from mtp_speculative_decoding_draft_gb300 import binding as bd
    L = bd.library()
    ws = bd.alloc_workspace(256)
    buf = torch.zeros(1024, dtype=torch.float32, device="cuda")
    ib = torch.zeros(1024, dtype=torch.int32, device="cuda")
    p = buf.data_ptr()
    ip = ib.data_ptr()
    # k = 0, k = 9, T <= 0 in stochastic mode, null target, misaligned pointer
    assert L.spec_verify(2, 0, 10, 1.0, 0, p, p, ip, p, p, ip, ip, ip, ws.data_ptr(), 256, None) == -1
    assert L.spec_verify(2, 9, 10, 1.0, 0, p, p, ip, p, p, ip, ip, ip, ws.data_ptr(), 256, None) == -1
    assert L.spec_verify(2, 2, 10, 0.0, 1, p, p, ip, p, p, ip, ip, ip, ws.data_ptr(), 256, None) == -1
    assert L.spec_verify(2, 2, 10, 1.0, 0, None, p, ip, p, p, ip, ip, ip, ws.data_ptr(), 256, None) == -1
    assert L.spec_verify(2, 2, 10, 1.0, 0, p + 4, p, ip, p, p, ip, ip, ip, ws.data_ptr(), 256, None) == -1
    assert L.spec_verify(2, 2, 10, 1.0, 0, p, p, ip, p, p, ip, ip, ip, ws.data_ptr(), 16, None) == -3


def test_bad_draft_token_sets_status():
    from mtp_speculative_decoding_draft_gb300 import binding as bd
    rng = np.random.default_rng(9)
    B, k, V = 2, 2, 500
    t = rng.standard_normal((B, k + 1, V)).astype(np.float32)
    d = np.array([[V + 5, 1], [-3, 0]], np.int32)
    (g_out, g_len, _), st = _run(t, None, d, None, None, GREEDY, 1.0)
    assert st & bd.STATUS_BAD_TOKEN
    assert list(g_len) == [1, 1]                    # an invalid draft is never accepted


@pytest.mark.parametrize("V,T", [(151936, 1.0), (20011, 0.7)])
def test_acceptance_probabilities_within_1e5_relative(V, T):
    """The softmax probabilities the verifier decides with, read off its
    decisions: with a constant draft row q(d) = 1/V, so u * q(d) < p(d) flips
    at V * p(d) as the kernel computes it.  Bisection on u_accept finds that
    point to float precision; it must lie within 1e-5 relative of the float64
    softmax."""
    from mtp_speculative_decoding_draft_gb300 import binding as bd
    B = 48
    t, draft, d, ratio = constant_draft_ratio_case(B, V, T, seed=4401)
    ver = Verifier(B, 1, V)
    t_d, l_d, d_d = to_device(t), to_device(draft), to_device(d)
    uf_d = to_device(np.full(B, 0.5, np.float32))

    def decide(u):
        ver(T, STOCH, t_d, l_d, d_d, to_device(u[:, None].copy()), uf_d)
        _, _, acc = ver.results()
        assert bd.get_status(ver.ws) == 0
        return acc >= 1

    lo, hi = accept_threshold_bisection(decide, B)
    got = (lo.astype(np.float64) + hi) / 2
    rel = np.abs(got - ratio) / ratio
    print("V=%d T=%g: V*p(d) from the decisions, max relative error %.3g (bracket %.3g)"
          % (V, T, rel.max(), float(np.max((hi - lo) / ratio))))
    assert np.all(rel <= 1e-5), "sequence %d: %r vs %r" % (int(np.argmax(rel)), got[np.argmax(rel)],
                                                           ratio[np.argmax(rel)])
