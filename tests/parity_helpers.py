"""Comparison helpers for GPU-vs-oracle parity.

Tolerances (stated once here, used by every GPU test):

* greedy tokens, accepted lengths and padded outputs: bit-exact;
* stochastic accept / reject decisions: identical except where the oracle's
  margin |u * q(d) - p(d)| < 1e-6; resampled / bonus tokens: identical except
  where u * S lies within 1e-6 * S of a CDF boundary.  Such cases are counted
  and reported, never silently passed;
* draft logits: relative L2 <= 1e-2 against the float32-master oracle (the
  stated bar) and <= 1e-3 against the oracle on the same bf16 weights;
* draft tokens: greedy identical except where the oracle's top-2 gap is below
  1e-2; stochastic identical except where the CDF margin is below
  2 * max|logit error| / T + 1e-6 (the largest shift the measured logit error
  can cause); the chain is not compared past an excused divergence;
* appended K/V rows (bf16): within one bf16 unit in the last place.
"""

import numpy as np

from oracle.sampling import softmax_T
from oracle.verify import residual

ACCEPT_BAND = 1e-6
SAMPLE_BAND = 1e-6


def stochastic_path_margins(target, draft, d, ua, uf, T):
    """Margins of every decision the oracle takes for one sequence.

    Returns (min accept margin along the path, relative CDF margin of the final
    draw)."""
    k = len(d)
    acc_margin = np.inf
    w = None
    for j in range(k):
        p = softmax_T(target[j], T)
        q = softmax_T(draft[j], T)
        x = ua[j] * q[d[j]]
        acc_margin = min(acc_margin, abs(x - p[d[j]]))
        if not x < p[d[j]]:
            R = residual(p, q)
            w = R if np.any(R > 0) else p
            break
    if w is None:
        w = softmax_T(target[k], T)
    return acc_margin, cdf_margin(w, uf)


def cdf_margin(w, u):
    """Distance of u*S to the nearest CDF boundary, relative to S."""
    C = np.cumsum(np.asarray(w, np.float64))
    S = C[-1]
    x = u * S
    i = int(np.searchsorted(C, x, side="right"))
    lo = C[i - 1] if i > 0 else 0.0
    hi = C[i] if i < len(C) else S
    return min(x - lo, hi - x) / S


def compare_verify(gpu, ora, mode, target=None, draft=None, d=None, ua=None, uf=None, T=1.0):
    """Compare (out_tok, accept_len, num_accepted) element by element.

    Returns the number of excused near-boundary sequences; raises on any other
    difference."""
    g_out, g_len, g_acc = gpu
    o_out, o_len, o_acc = ora
    bad = np.nonzero((g_out != o_out).any(axis=1) | (g_len != o_len) | (g_acc != o_acc))[0]
    if mode == 0:
        assert bad.size == 0, "greedy mismatch at sequences %s" % bad[:10]
        return 0
    excused = 0
    for b in bad:
        am, sm = stochastic_path_margins(target[b], draft[b], d[b], ua[b], float(uf[b]), T)
        assert am < ACCEPT_BAND or sm < SAMPLE_BAND, (
            "sequence %d differs: gpu %s/%d oracle %s/%d (margins %.3g, %.3g)"
            % (b, g_out[b], g_len[b], o_out[b], o_len[b], am, sm))
        excused += 1
    return excused


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def top2_gap(z):
    z = np.sort(np.asarray(z, np.float64))
    return float(z[-1] - z[-2]) if z.size > 1 else np.inf


def bf16_ulp_ok(gpu_vals, ora_vals):
    """Every value within one bf16 ulp (relative spacing 2^-7 of the larger
    magnitude), or, for a value near zero, within 2^-12 of the row's largest
    magnitude: the values are float32 dot products (absolute error about
    2^-24 of the sum of the terms' magnitudes) rounded to bf16, so an entry
    that cancels to near zero can land past its own ulp.  Prints the worst
    entry when the check fails."""
    g = np.asarray(gpu_vals, np.float64)
    o = np.asarray(ora_vals, np.float64)
    scale = float(np.max(np.abs(o))) if o.size else 0.0
    tol = np.maximum(np.abs(g), np.abs(o)) * 2.0 ** -7 + 2.0 ** -12 * scale + 1e-30
    bad = np.abs(g - o) > tol
    if np.any(bad):
        i = np.unravel_index(int(np.argmax(np.abs(g - o) - tol)), g.shape)
        print("bf16 check: gpu %r oracle %r tol %.3g row max %.3g" % (g[i], o[i], tol[i], scale))
    return not bool(np.any(bad))


def accept_threshold_bisection(decide, B, iters=34):
    """The u at which each sequence's accept decision at position 0 flips.

    decide(u) takes float32 uniforms [B] and returns which sequences accepted
    their first draft.  The decision is u * q(d) < p(d), so acceptance is
    monotone in u and the flip lies at p(d) / q(d).  Returns (lo, hi): every
    sequence accepted at lo and rejected at hi."""
    lo = np.zeros(B, np.float32)
    hi = np.ones(B, np.float32)
    for _ in range(iters):
        mid = ((lo.astype(np.float64) + hi) / 2).astype(np.float32)
        a = np.asarray(decide(mid), bool)
        lo = np.where(a, mid, lo)
        hi = np.where(a, hi, mid)
    return lo, hi


def constant_draft_ratio_case(B, V, T, seed):
    """Target rows, a constant draft row (q = 1/V at every id) and, per
    sequence, a draft token d whose V * p(d) is spread over (1e-3, 0.95):
    the flip of u * q(d) < p(d) is then V * p(d)."""
    rng = np.random.default_rng(seed)
    t = (rng.standard_normal((B, 2, V)) * 3.0).astype(np.float32)
    draft = np.zeros((B, 1, V), np.float32)
    p = np.stack([softmax_T(t[b, 0], T) for b in range(B)])
    want = np.exp(rng.uniform(np.log(1e-3), np.log(0.95), size=B))
    d = np.array([[int(np.argmin(np.abs(p[b] * V - want[b])))] for b in range(B)], np.int32)
    ratio = p[np.arange(B), d[:, 0]] * V
    return t, draft, d, ratio
