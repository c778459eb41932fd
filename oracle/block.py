"""The MTP draft module (one transformer block with an input projection) and its
k-deep autoregressive chain, in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Dataflow of one application, for each sequence b ("The Tiny Draft Model Hidden
Inside Qwen", sections "One step deeper than the main model" and "What vLLM and
SGLang do with the weights"; module inventory in the opening section: one
``mtp.fc`` projection, one full-attention block ``mtp.layers.0``, three
normalisation weights, no embedding table of its own):

  a1  e  = E[tok]                            shared embedding row
      u  = [rms(e) * g_emb ; rms(x) * g_hid]  normalise both, concatenate (2d)
      x0 = W_fc u                             project 2d -> d
  a2  n  = rms(x0) * g_attn
      q = Wq n,  k = Wk n,  v = Wv n          k, v rounded to bf16 and appended
                                              to the cache at position L_b + j
  a3  o_h = sum_t softmax_t(q_h . K_t / sqrt(Dh)) V_t  over t = 0 .. L_b + j,
      head h reads kv head h // (Hq / Hkv)
  a4  x1 = x0 + Wo o
  a5  n' = rms(x1) * g_mlp
      x2 = x1 + Wdown (silu(Wgate n') * (Wup n'))
  a6  logits = E (rms(x2) * g_final)          the shared vocabulary head

The chain ("Optimize vLLM speculative decoding with FastMTP heads", section "Why
fine-tune a single MTP head"; "The Tiny Draft Model Hidden Inside Qwen", section
"One step deeper than the main model"): depth 0 takes the trunk hidden state h
and the last token; every later depth takes the module's own output hidden state
x2 and the token it just drafted.

Readings where the pages are silent (each listed in the design notes):
concatenation order embedding first; rms(v) = v / sqrt(mean(v^2) + eps) with a
plain multiplicative gain; no positional rotation inside the block; no QK-norm,
gate or bias; SiLU(z) = z / (1 + exp(-z)); the attention scale 1/sqrt(Dh); the
embedding matrix doubles as the LM head; the hidden state fed back is the block
output x2 before the final norm; the logits are stored as float32.

Parity: structural pins only (see the tests); the GPU comparison of the block's
numerics is "parity unpinned" beyond the stated tolerance, since the pages print
no worked example.
"""

import numpy as np

from .numerics import as_f64, round_bf16, round_f32
from .sampling import argmax_lowest, inverse_cdf

GREEDY = 0
STOCHASTIC = 1


def rmsnorm(v, g, eps):
    """v / sqrt(mean(v^2) + eps) * g over the last axis."""
    v = np.asarray(v, dtype=np.float64)
    return v / np.sqrt(np.mean(v * v, axis=-1, keepdims=True) + eps) * as_f64(g)


def silu(z):
    """SiLU(z) = z / (1 + exp(-z))."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def linear(W, a, rows_per_chunk=8192):
    """y = a W^T for W [out, in] (bf16 bits or reals) and a [..., in].

    The weight is widened to float64 one row block at a time so that a large
    matrix never needs a full float64 copy.
    """
    W = np.asarray(W)
    a = np.asarray(a, dtype=np.float64)
    out = W.shape[0]
    y = np.empty(a.shape[:-1] + (out,), dtype=np.float64)
    for r0 in range(0, out, rows_per_chunk):
        Wc = as_f64(W[r0:r0 + rows_per_chunk])
        y[..., r0:r0 + Wc.shape[0]] = a @ Wc.T
    return y


def gqa_attention(q, K, V):
    """Single-query softmax attention with grouped KV heads.

    q [Hq, Dh]; K, V [Hkv, T, Dh]; query head h reads kv head h // (Hq / Hkv).
    Full softmax over all T keys with the maximum subtracted; scale 1/sqrt(Dh).
    """
    q = np.asarray(q, dtype=np.float64)
    Hq, Dh = q.shape
    Hkv = K.shape[0]
    group = Hq // Hkv
    o = np.empty((Hq, Dh), dtype=np.float64)
    for h in range(Hq):
        g = h // group
        s = (K[g] @ q[h]) / np.sqrt(Dh)
        w = np.exp(s - np.max(s))
        o[h] = (w / np.sum(w)) @ V[g]
    return o


class Dims:
    """Block shape: batch B, hidden d, heads Hq / Hkv of size Dh, FFN F, vocab V,
    cache capacity Lmax, RMSNorm epsilon."""

    def __init__(self, B, d, Hq, Hkv, Dh, F, V, Lmax, eps=1e-6):
        self.B, self.d, self.Hq, self.Hkv, self.Dh = B, d, Hq, Hkv, Dh
        self.F, self.V, self.Lmax, self.eps = F, V, Lmax, eps


def draft_depth(W, dims, x, tok, keys, values, trace=None):
    """One application of the MTP module to a group of sequences (steps a1-a6).

    W       dict of weights: E [V,d], fc [d,2d], wq [Hq*Dh,d], wk/wv [Hkv*Dh,d],
            wo [d,Hq*Dh], wgate/wup [F,d], wdown [d,F] and gains g_emb, g_hid,
            g_attn, g_mlp, g_final [d]; bf16 bits or reals.
    x       [n, d] input hidden state (trunk h at depth 0, previous x2 later).
    tok     [n] input token ids.
    keys    list of n arrays [Hkv, T_b, Dh]: the visible cache of each sequence
            before this depth; values likewise.
    trace   optional dict: receives "attn_in" [n, d], the attention input n
            (the vector the Q/K/V projections multiply), for error estimates.
    Returns (x2 [n,d], logits [n,V] float64, k_new [n,Hkv,Dh], v_new [n,Hkv,Dh]);
    k_new / v_new are already rounded to bf16 (they are stored in a bf16 cache
    and the current position attends to the stored values).
    """
    eps = dims.eps
    n = x.shape[0]
    x = np.asarray(x, dtype=np.float64)
    e = as_f64(np.asarray(W["E"])[np.asarray(tok)])
    u = np.concatenate([rmsnorm(e, W["g_emb"], eps), rmsnorm(x, W["g_hid"], eps)], axis=-1)
    x0 = linear(W["fc"], u)

    nrm = rmsnorm(x0, W["g_attn"], eps)
    if trace is not None:
        trace["attn_in"] = nrm
    q = linear(W["wq"], nrm).reshape(n, dims.Hq, dims.Dh)
    k_new = round_bf16(linear(W["wk"], nrm)).reshape(n, dims.Hkv, dims.Dh)
    v_new = round_bf16(linear(W["wv"], nrm)).reshape(n, dims.Hkv, dims.Dh)

    o = np.empty((n, dims.Hq * dims.Dh), dtype=np.float64)
    for b in range(n):
        Kb = np.concatenate([keys[b], k_new[b][:, None, :]], axis=1)
        Vb = np.concatenate([values[b], v_new[b][:, None, :]], axis=1)
        o[b] = gqa_attention(q[b], Kb, Vb).reshape(-1)
    x1 = x0 + linear(W["wo"], o)

    nrm2 = rmsnorm(x1, W["g_mlp"], eps)
    act = silu(linear(W["wgate"], nrm2)) * linear(W["wup"], nrm2)
    x2 = x1 + linear(W["wdown"], act)

    # the vocabulary head: E, or the rows of a reduced draft vocabulary
    logits = linear(W.get("head", W["E"]), rmsnorm(x2, W["g_final"], eps))
    return x2, logits, k_new, v_new


def select_token(logits, mode, T, u):
    """Pick the next draft token from one row of (float32-valued) logits.

    Greedy: the argmax, lowest index on ties.  Stochastic: the inverse-CDF draw
    at u from q = softmax(logits / T) (SGLang's recommended topk=1 chain, "The
    Tiny Draft Model Hidden Inside Qwen", section "What vLLM and SGLang do with
    the weights").
    """
    if mode == GREEDY:
        return argmax_lowest(logits)
    z = np.asarray(logits, dtype=np.float64)
    return inverse_cdf(np.exp((z - np.max(z)) / T), u)


def draft_confidence(logits, mode, T):
    """The draft's largest probability at one depth: max_i q(i), with q the
    distribution the draft token is taken from -- softmax(logits / T) when
    stochastic, softmax(logits) when greedy.  Written as 1 / sum_i exp((l_i -
    max) / T), in float64."""
    z = np.asarray(logits, dtype=np.float64)
    t = T if mode == STOCHASTIC else 1.0
    return 1.0 / float(np.sum(np.exp((z - np.max(z)) / t)))


def dynamic_depths(draft_logits, mode, T, stop_p):
    """Drafts each sequence keeps under a dynamic draft length ("Faster
    Rollouts with MTP Speculative Decoding", section "What's Next", names
    dynamic draft length without a rule; the reading taken here): the chain of
    sequence b stops at the first depth j whose draft confidence is below
    stop_p, keeping the j drafts before it; k if no depth falls below.

    draft_logits [n, k, V] (float32 values).  Returns k_eff [n] in 0..k.
    """
    dl = np.asarray(draft_logits)
    n, k = dl.shape[0], dl.shape[1]
    out = np.full(n, k, dtype=np.int64)
    for i in range(n):
        for j in range(k):
            if draft_confidence(dl[i, j], mode, T) < stop_p:
                out[i] = j
                break
    return out


def mtp_draft(W, dims, h, last_tok, k_cache, v_cache, ctx_len, k, T, mode,
              u_draft=None, seqs=None, vocab_map=None, forced_tok=None):
    """Run the module k times in a chain and return the drafts.

    h        [B, d] trunk hidden states (bf16 bits or reals).
    last_tok [B] the token the trunk just produced.
    k_cache, v_cache  [B, Hkv, Lmax, Dh] bf16 bits; rows [0, ctx_len[b]) hold the
             context.  They are only read: the rows this call appends at positions
             ctx_len[b] + j are returned in k_new / v_new.
    u_draft  [B, k] uniforms for stochastic drafting (ignored when greedy).
    seqs     optional subset of sequence indices to evaluate (all by default).
    forced_tok  [n, k] optional (teacher forcing): depth j+1 takes
             forced_tok[i, j] as its input token instead of this chain's own
             choice at depth j; the hidden state stays this chain's own, and
             draft_tok still records this chain's own choices.
    Returns a dict with draft_tok [n,k], draft_logits [n,k,V] (float32 values),
    hidden [n,k,d] (x2 of every depth), k_new / v_new [n,k,Hkv,Dh] (bf16 values)
    and attn_in [n,k,d] (each depth's attention input, the vector the K/V
    projections multiply).
    """
    return mtp_draft_modules([(W, k_cache, v_cache)], dims, h, last_tok, ctx_len, k, T, mode,
                             u_draft, seqs, vocab_map, forced_tok)


def module_of_depth(j, n_modules):
    """The module depth j runs when a chain has n_modules distinct modules: its
    own while there are enough (DeepSeek-V3's one module per future token,
    "Optimize vLLM speculative decoding with FastMTP heads", sections "What is
    multi-token prediction?" and "Why fine-tune a single MTP head"), else the
    last one again (one module reused at every depth when n_modules = 1)."""
    return min(j, n_modules - 1)


def mtp_draft_modules(modules, dims, h, last_tok, ctx_len, k, T, mode, u_draft=None, seqs=None,
                      vocab_map=None, forced_tok=None):
    """The chain over distinct modules.

    modules  list of (W, k_cache, v_cache): each module's weights and its own
             K/V cache (each module has its own attention).  Depth j runs module
             m = module_of_depth(j, len(modules)); it attends over module m's
             context rows [0, ctx_len[b]) plus the rows this call appended to
             that cache, its own last, so its row lands at position ctx_len[b] +
             (number of earlier depths that ran module m).
    Other arguments and the returned dict as ``mtp_draft``; the dict also holds
    module [k] (the module of each depth) and row [n, k] (the cache position of
    each depth's K/V row in its module's cache).

    vocab_map  [N] (optional): a reduced draft vocabulary ("Optimize vLLM
    speculative decoding with FastMTP heads", sections "How FastMTP-style
    fine-tuning works in Speculators" and "What's next?", name FR-Spec-style
    reduction; the rule is this build's reading).  The weights then carry
    "head" [N, d], the rows vocab_map of E; the draft distribution is the
    softmax over those N logits, the draft token vocab_map of the choice among
    them, and draft_logits hold the N logits at their ids and -inf elsewhere
    (q = 0 outside the reduced vocabulary).
    """
    seqs = list(range(np.asarray(last_tok).shape[0])) if seqs is None else list(seqs)
    n = len(seqs)
    x = as_f64(np.asarray(h)[seqs])
    tok = np.asarray(last_tok)[seqs].astype(np.int64)
    keys, values = [], []
    for (_, kc, vc) in modules:
        keys.append([as_f64(np.asarray(kc)[b, :, :int(ctx_len[b]), :]) for b in seqs])
        values.append([as_f64(np.asarray(vc)[b, :, :int(ctx_len[b]), :]) for b in seqs])

    out = {
        "draft_tok": np.zeros((n, k), dtype=np.int64),
        "draft_logits": np.zeros((n, k, dims.V), dtype=np.float64),
        "hidden": np.zeros((n, k, dims.d), dtype=np.float64),
        "k_new": np.zeros((n, k, dims.Hkv, dims.Dh), dtype=np.float64),
        "v_new": np.zeros((n, k, dims.Hkv, dims.Dh), dtype=np.float64),
        "module": np.zeros(k, dtype=np.int64),
        "row": np.zeros((n, k), dtype=np.int64),
        "attn_in": np.zeros((n, k, dims.d), dtype=np.float64),
    }
    for j in range(k):
        m = module_of_depth(j, len(modules))
        W = modules[m][0]
        for i in range(n):
            out["row"][i, j] = keys[m][i].shape[1]
        tr = {}
        x, logits, k_new, v_new = draft_depth(W, dims, x, tok, keys[m], values[m], trace=tr)
        out["attn_in"][:, j] = tr["attn_in"]
        logits = round_f32(logits)
        for i, b in enumerate(seqs):
            u = None if mode == GREEDY else float(u_draft[b][j])
            choice = select_token(logits[i], mode, T, u)
            out["draft_tok"][i, j] = choice if vocab_map is None else int(vocab_map[choice])
            keys[m][i] = np.concatenate([keys[m][i], k_new[i][:, None, :]], axis=1)
            values[m][i] = np.concatenate([values[m][i], v_new[i][:, None, :]], axis=1)
        if vocab_map is None:
            out["draft_logits"][:, j] = logits
        else:
            out["draft_logits"][:, j] = -np.inf
            out["draft_logits"][:, j][:, np.asarray(vocab_map)] = logits
        out["hidden"][:, j] = x
        out["k_new"][:, j] = k_new
        out["v_new"][:, j] = v_new
        out["module"][j] = m
        tok = out["draft_tok"][:, j].copy() if forced_tok is None else np.asarray(forced_tok)[:, j].astype(np.int64)
    return out
