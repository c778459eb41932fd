"""Verification of k drafted tokens against the target model's distributions.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The target scores all draft positions in one pass and produces, for each
sequence, k+1 rows of logits: row j is the target's distribution for the token
after the context and the first j drafts ("The Tiny Draft Model Hidden Inside
Qwen", section "How the draft becomes real output").  The verifier accepts the
longest prefix the target agrees with and, at the first rejection, drops the
rest of the draft and emits a token from the corrected replacement distribution.
If every draft is accepted, one more token comes from row k: "guess three tokens
correctly and you've produced four" ("Speculative Decoding and MTP: Why Guessing
Is Free", section "Speculative decoding: draft, then verify").

Greedy mode: draft j+1 is accepted while it equals argmax of target row j; the
emitted tokens then equal ordinary greedy decoding.

Stochastic mode: the pages require a "proper rejection sampler" that leaves the
output distributed exactly as the target's ("Speculative Decoding and MTP: Why
Guessing Is Free", section "It's exact, not approximate").  The plainest rule
with that property, taken here: with p = softmax(t_j / T), q = softmax(l_j / T)
and d the draft, accept iff u_accept * q(d) < p(d) (accept with probability
min(1, p/q)); at the first rejection r, draw from R proportional to
max(0, p_r - q_r) with u_final (from p_r itself if R is identically zero); if all
k are accepted, draw the bonus token from p_k with u_final.

Parity: greedy is pinned against plain greedy decoding; the stochastic rule is
pinned by exact enumeration of the emitted-sequence distribution on small
vocabularies (it must equal the target's own autoregressive distribution).
"""

import numpy as np

from .sampling import argmax_lowest, inverse_cdf, softmax_T

GREEDY = 0
STOCHASTIC = 1


def residual(p, q):
    """Unnormalised corrected distribution max(0, p - q)."""
    return np.maximum(np.asarray(p, np.float64) - np.asarray(q, np.float64), 0.0)


def verify_greedy_one(target, draft_tok):
    """target [k+1, V] logits, draft_tok [k].  Returns (emitted tokens, a)."""
    k = len(draft_tok)
    a = 0
    while a < k and argmax_lowest(target[a]) == int(draft_tok[a]):
        a += 1
    return [int(t) for t in draft_tok[:a]] + [argmax_lowest(target[a])], a


def verify_stochastic_one(target, draft, draft_tok, u_accept, u_final, T):
    """target [k+1, V] and draft [k, V] logits, draft_tok [k], u_accept [k].

    Returns (emitted tokens, a) where a is the number of accepted drafts.
    """
    k = len(draft_tok)
    for j in range(k):
        p = softmax_T(target[j], T)
        q = softmax_T(draft[j], T)
        d = int(draft_tok[j])
        if u_accept[j] * q[d] < p[d]:
            continue
        R = residual(p, q)
        c = inverse_cdf(R, u_final) if np.any(R > 0) else inverse_cdf(p, u_final)
        return [int(t) for t in draft_tok[:j]] + [c], j
    c = inverse_cdf(softmax_T(target[k], T), u_final)
    return [int(t) for t in draft_tok] + [c], k


def spec_verify(target_logits, draft_logits, draft_tok, mode, T=1.0,
                u_accept=None, u_final=None, seqs=None, k_eff=None):
    """Batched verification.

    target_logits [B, k+1, V]; draft_logits [B, k, V] (unused when greedy);
    draft_tok [B, k]; u_accept [B, k]; u_final [B]; k_eff [B] (optional): the
    drafts sequence b keeps (a dynamic draft length, ``block.dynamic_depths``);
    its verification then sees only drafts 0..k_eff-1 and target rows
    0..k_eff, the bonus row being row k_eff.
    Returns out_tok [n, k+1] (padded with -1), accept_len [n] (= a + 1) and
    num_accepted [n] (= a) for the sequences in ``seqs`` (all by default).
    """
    target_logits = np.asarray(target_logits)
    B, k1, _ = target_logits.shape
    k = k1 - 1
    seqs = list(range(B)) if seqs is None else list(seqs)
    out_tok = np.full((len(seqs), k + 1), -1, dtype=np.int64)
    accept_len = np.zeros(len(seqs), dtype=np.int64)
    num_accepted = np.zeros(len(seqs), dtype=np.int64)
    for i, b in enumerate(seqs):
        kb = k if k_eff is None else int(k_eff[b])
        t = target_logits[b, :kb + 1].astype(np.float64)
        if mode == GREEDY:
            toks, a = verify_greedy_one(t, draft_tok[b][:kb])
        else:
            toks, a = verify_stochastic_one(t, np.asarray(draft_logits[b][:kb], np.float64),
                                            draft_tok[b][:kb], u_accept[b][:kb], float(u_final[b]), T)
        out_tok[i, :len(toks)] = toks
        accept_len[i] = a + 1
        num_accepted[i] = a
    return out_tok, accept_len, num_accepted


def target_logits_from_hidden(head, hidden):
    """The target's logits at every verified position, formed from its final
    hidden states: t[..., v] = sum_i head[v, i] * hidden[..., i], in float64.

    "The Tiny Draft Model Hidden Inside Qwen", section "How the draft becomes
    real output": the target runs once over all candidate positions and its
    vocabulary head gives its own distribution at each of them.  head [V, d] is
    that head (the shared embedding matrix), hidden [..., d] what the head
    consumes at each position (the target's final hidden state after its final
    norm); both bf16 bits or reals, widened exactly.

    Parity: pinned by one-hot hidden states (a single column of the head
    comes out, which a transposed operand would not give), by linearity, and
    by an element-by-element loop on a small case.
    """
    from .block import linear
    from .numerics import as_f64
    return linear(head, as_f64(hidden))


def spec_verify_fused(head, hidden, draft_logits, draft_tok, mode, T=1.0, u_accept=None, u_final=None,
                      seqs=None):
    """Verification from the target's hidden states instead of its logits: the
    logits come from ``target_logits_from_hidden`` (never stored as float32)
    and the rule is ``spec_verify``'s, unchanged.

    hidden [B, k+1, d]; other arguments and the result as ``spec_verify``.
    """
    hidden = np.asarray(hidden)
    B = hidden.shape[0]
    seqs = list(range(B)) if seqs is None else list(seqs)
    t = target_logits_from_hidden(head, hidden[seqs])
    dl = None if draft_logits is None else np.asarray(draft_logits)[seqs]
    ua = None if u_accept is None else np.asarray(u_accept)[seqs]
    uf = None if u_final is None else np.asarray(u_final)[seqs]
    return spec_verify(t, dl, np.asarray(draft_tok)[seqs], mode, T, ua, uf)


def spec_step(W, dims, h, last_tok, k_cache, v_cache, ctx_len, k, T, mode,
              target_logits, u_draft=None, u_accept=None, u_final=None, seqs=None, stop_p=None,
              vocab_map=None):
    """Draft k tokens with the chained module, then verify them.  With stop_p,
    each sequence keeps the drafts before its first depth of confidence below
    stop_p (``block.dynamic_depths``; the result dict then holds k_eff).

    Returns (draft result dict from ``block.mtp_draft``, out_tok, accept_len,
    num_accepted) for the sequences in ``seqs``.
    """
    return spec_step_modules([(W, k_cache, v_cache)], dims, h, last_tok, ctx_len, k, T, mode,
                             target_logits, u_draft, u_accept, u_final, seqs, stop_p, vocab_map)


def spec_step_modules(modules, dims, h, last_tok, ctx_len, k, T, mode, target_logits,
                      u_draft=None, u_accept=None, u_final=None, seqs=None, stop_p=None, vocab_map=None):
    """``spec_step`` over a chain of distinct modules (``block.mtp_draft_modules``)."""
    from .block import dynamic_depths, mtp_draft_modules
    seqs = list(range(np.asarray(last_tok).shape[0])) if seqs is None else list(seqs)
    dr = mtp_draft_modules(modules, dims, h, last_tok, ctx_len, k, T, mode, u_draft, seqs, vocab_map)
    tl = np.asarray(target_logits)[seqs]
    ua = None if u_accept is None else np.asarray(u_accept)[seqs]
    uf = None if u_final is None else np.asarray(u_final)[seqs]
    k_eff = None
    if stop_p is not None:
        k_eff = dynamic_depths(dr["draft_logits"], mode, T, stop_p)
        dr["k_eff"] = k_eff
    out_tok, accept_len, num_acc = spec_verify(tl, dr["draft_logits"], dr["draft_tok"], mode, T, ua, uf,
                                               k_eff=k_eff)
    return dr, out_tok, accept_len, num_acc
