"""Acceptance metrics computed on the host from the verifier's outputs.

Names and definitions follow the monitoring section of "Faster Rollouts with MTP
Speculative Decoding" (section "Monitoring acceptance"):

* draft_acceptance_rate          accepted drafts / drafted tokens;
* draft_mean_acceptance_length   tokens emitted per target pass, in [1, k+1];
* draft_acceptance_rate_pos_j    fraction of steps whose j-th draft was accepted
                                 (j = 1..k; a draft counts only if all earlier
                                 drafts of that step were accepted too);
* draft_num_draft_tokens, draft_num_accepted_tokens   raw counts.

With these definitions mean length = 1 + sum_j pos_j, the identity the page's
own figures satisfy (section "Results": 1 + 0.886 + 0.770 + 0.663 = 3.32).
"""

import numpy as np


def acceptance_metrics(accept_len, k):
    """accept_len: emitted tokens per sequence-step (each in [1, k+1])."""
    L = np.asarray(accept_len, dtype=np.int64).reshape(-1)
    if L.size == 0:
        raise ValueError("no verification results")
    if L.min() < 1 or L.max() > k + 1:
        raise ValueError("accept_len outside [1, k+1]")
    a = L - 1
    n = L.size
    out = {
        "draft_num_draft_tokens": int(n * k),
        "draft_num_accepted_tokens": int(a.sum()),
        "draft_acceptance_rate": float(a.sum()) / float(n * k),
        "draft_mean_acceptance_length": float(L.mean()),
    }
    for j in range(1, k + 1):
        out["draft_acceptance_rate_pos_%d" % j] = float((a >= j).sum()) / float(n)
    return out


def mean_length_from_positions(pos):
    """Mean emitted length implied by per-depth acceptance fractions: 1 + sum pos_j."""
    return 1.0 + float(np.sum(pos))
