"""Pins of the oracle's reduced draft vocabulary ("Optimize vLLM speculative
decoding with FastMTP heads", sections "How FastMTP-style fine-tuning works in
Speculators" and "What's next?", name FR-Spec-style reduction; the rule is this
build's reading): the draft head is N rows of E, the draft distribution the
softmax over their logits, the draft token the vocabulary id of the chosen row,
and q = 0 at every other id.
"""

import itertools

import numpy as np

from oracle.block import GREEDY, STOCHASTIC, Dims, mtp_draft
from oracle.sampling import argmax_lowest
from oracle.verify import verify_stochastic_one
from mtp_speculative_decoding_draft_gb300 import workloads as W


def _tiny():
    w = W.TINY
    dims = Dims(w.B, w.d, w.Hq, w.Hkv, w.Dh, w.F, w.V, w.Lmax, w.eps)
    return w, dims, W.make_weights(w), W.make_context(w), W.make_uniforms(w)["u_draft"]


def _run(wts, dims, ctx, w, mode, u, vmap=None):
    return mtp_draft(wts, dims, ctx["h"], ctx["last_tok"], ctx["k_cache"], ctx["v_cache"], ctx["ctx_len"],
                     w.k, 0.9, mode, u, vocab_map=vmap)


def test_draft_vocab_generator():
    w = W.TINY
    vmap, head = W.make_draft_vocab(w, 300)
    assert len(set(vmap.tolist())) == 300 and vmap.min() >= 0 and vmap.max() < w.V
    assert np.array_equal(head, W.make_weights(w)["E"][vmap])


def test_identity_map_is_the_full_vocabulary():
    w, dims, wts, ctx, u = _tiny()
    for mode in (GREEDY, STOCHASTIC):
        full = _run(wts, dims, ctx, w, mode, u)
        ident = _run(dict(wts, head=wts["E"]), dims, ctx, w, mode, u, vmap=np.arange(w.V))
        np.testing.assert_array_equal(full["draft_logits"], ident["draft_logits"])
        np.testing.assert_array_equal(full["draft_tok"], ident["draft_tok"])


def test_reduced_head_logits_are_the_full_logits_at_their_ids():
    w, dims, wts, ctx, u = _tiny()
    vmap, head = W.make_draft_vocab(w, 250)
    full = _run(wts, dims, ctx, w, GREEDY, u)
    red = _run(dict(wts, head=head), dims, ctx, w, GREEDY, u, vmap=vmap)
    row = red["draft_logits"][0, 0]
    outside = np.ones(w.V, bool)
    outside[vmap] = False
    assert np.all(row[outside] == -np.inf)
    np.testing.assert_allclose(row[vmap], full["draft_logits"][0, 0][vmap], rtol=1e-6, atol=1e-9)
    # greedy: the best id of the subset, found by scanning the subset in head-row order
    sub = full["draft_logits"][0, 0][vmap]
    assert red["draft_tok"][0, 0] == vmap[argmax_lowest(sub)]
    assert red["draft_tok"][0, 0] in set(vmap.tolist())
    # stochastic: every draft comes from the subset
    reds = _run(dict(wts, head=head), dims, ctx, w, STOCHASTIC, u, vmap=vmap)
    assert set(reds["draft_tok"].ravel().tolist()) <= set(vmap.tolist())


def test_verification_stays_exact_with_q_zero_outside_the_subset():
    """Enumeration as in test_oracle_verify, with every draft row supported on
    ids {0, 2} of V = 4 only (dyadic q), the target on all four."""
    rng = np.random.default_rng(51)
    V, k, n_units, grid_n, T = 4, 2, 16, 16, 1.0
    P, Q = {}, {}
    for n in range(k + 1):
        for pre in itertools.product(range(V), repeat=n):
            while True:
                p = rng.multinomial(n_units - V, rng.dirichlet(np.ones(V))) + 1
                q = np.zeros(V, int)
                q[[0, 2]] = 8                  # q = 1/2 on ids 0 and 2: p / q on the 1/8 grid
                s = int(np.maximum(p - q, 0).sum())
                if s == 0 or (s & (s - 1)) == 0:
                    break
            P[pre] = p / n_units
            if n < k:
                Q[pre] = q / n_units
    g = (np.arange(grid_n) + 0.5) / grid_n
    cell = 1.0 / grid_n ** (k + 1)
    spec = {}
    with np.errstate(divide="ignore"):
        for d in itertools.product([0, 2], repeat=k):
            wq = np.prod([Q[d[:j]][d[j]] for j in range(k)])
            target = np.stack([T * np.log(P[d[:j]]) for j in range(k + 1)])
            draft = np.stack([T * np.log(Q[d[:j]]) for j in range(k)])
            for us in itertools.product(g, repeat=k + 1):
                out, a = verify_stochastic_one(target, draft, d, us[:k], us[k], T)
                spec[tuple(out)] = spec.get(tuple(out), 0.0) + wq * cell
    assert abs(sum(spec.values()) - 1.0) < 1e-12
    outside_emitted = 0.0
    for x in itertools.product(range(V), repeat=k + 1):
        p_target = np.prod([P[x[:j]][x[j]] for j in range(k + 1)])
        p_spec = 0.0
        for L in range(1, k + 2):
            e = x[:L]
            if e in spec:
                cont = np.prod([P[x[:j]][x[j]] for j in range(L, k + 1)]) if L <= k else 1.0
                p_spec += spec[e] * cont
        assert abs(p_spec - p_target) < 1e-12, (x, p_spec, p_target)
        if x[0] in (1, 3):
            outside_emitted += p_spec
    assert outside_emitted > 0.1   # ids outside the draft vocabulary are still emitted, through the residual
