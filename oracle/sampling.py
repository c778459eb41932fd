"""Temperature softmax, argmax and inverse-CDF sampling over the full vocabulary.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Both the drafter and the verifier work on the whole shared vocabulary: the draft
head is the verifier's own LM head, with no vocabulary reduction ("Optimize vLLM
speculative decoding with FastMTP heads", section "Key features", full-vocabulary
draft head).  Random draws are driven by caller-supplied uniforms u in [0, 1), so
every result is a deterministic function of its inputs.
"""

import numpy as np


def softmax_T(z, T):
    """p_i = exp((z_i - max z) / T) / sum_j exp((z_j - max z) / T), in float64.

    Parity: pinned against ``scipy.special.softmax`` and sum-to-one in the tests.
    """
    z = np.asarray(z, dtype=np.float64)
    w = np.exp((z - np.max(z)) / T)
    return w / np.sum(w)


def argmax_lowest(z):
    """Index of the largest entry; on ties the lowest index wins.

    ``np.argmax`` returns the first occurrence of the maximum, which is exactly
    the lowest-index tie rule.  Parity: pinned by explicit tie cases.
    """
    return int(np.argmax(np.asarray(z, dtype=np.float64)))


def inverse_cdf(w, u):
    """Sample index for non-negative weights w (not necessarily normalised).

    With prefix sums C_i = w_0 + ... + w_i taken in index order and S = C_{V-1},
    return the smallest i with C_i > u * S.  If rounding leaves no such i (u
    just below 1), return the last index with w_i > 0.  This is the plainest
    reading of "draw from the distribution with a uniform": selecting i has
    probability exactly w_i / S over u ~ U[0, 1).

    Parity: pinned in the tests by exact integration over a dyadic grid of u
    (the selection probabilities must equal w_i / S exactly).
    """
    w = np.asarray(w, dtype=np.float64)
    C = np.cumsum(w)
    S = C[-1]
    hit = np.nonzero(C > u * S)[0]
    if hit.size:
        return int(hit[0])
    pos = np.nonzero(w > 0)[0]
    return int(pos[-1])
