"""GPU parity of spec_step (draft chain + verification in one call).

The GPU drafts with its own kernels and verifies its own drafts.  The draft is
compared with the oracle chain teacher-forced with the GPU's drafts (oracle
depth j+1 takes the GPU's draft j and keeps its own hidden state); the outputs
with the oracle's verification of the GPU's own drafts and draft logits,
identical except where a decision lies within 1e-6 of its boundary.  Target logits are built from the ORACLE's draft logits
plus seeded noise (position j gets std sigma0 * 1.5^j; the bonus row reuses the
last draft row), so drafts are accepted often enough to exercise every branch.
Sequences not sampled for comparison get noise-only targets.
"""

import numpy as np
import pytest
import torch

from mtp_speculative_decoding_draft_gb300 import workloads as W
from mtp_speculative_decoding_draft_gb300.model import DraftModule, to_device
from oracle.block import Dims, mtp_draft as oracle_draft
from oracle.verify import spec_verify as oracle_verify
from parity_helpers import ACCEPT_BAND, SAMPLE_BAND, cdf_margin, rel_l2, stochastic_path_margins, top2_gap

pytestmark = pytest.mark.gpu

GREEDY, STOCH = 0, 1


def _dims(w):
    return Dims(w.B, w.d, w.Hq, w.Hkv, w.Dh, w.F, w.V, w.Lmax, w.eps)


def run_step_parity(w, mode, T, seqs, sigma0=None, uncorrelated=False):
    wts = W.make_weights(w)
    ctx = W.make_context(w)
    u = W.make_uniforms(w)
    k, B, V = w.k, w.B, w.V
    ora_d = oracle_draft(wts, _dims(w), ctx["h"], ctx["last_tok"], ctx["k_cache"], ctx["v_cache"],
                         ctx["ctx_len"], k, T, mode, u["u_draft"], seqs)
    if uncorrelated:
        target = W.target_logits(w)
    else:
        wn = W.Workload(w.name, B=B, k=k + 1, V=V, seed=w.seed,
                        draft_noise_std0=sigma0 if sigma0 is not None else w.draft_noise_std0,
                        noise_growth=w.noise_growth if w.noise_growth != 1.0 else 1.5)
        target = W.draft_noise(wn, k + 1)
        for i, b in enumerate(seqs):
            for j in range(k + 1):
                target[b, j] += ora_d["draft_logits"][i, min(j, k - 1)].astype(np.float32)
    m = DraftModule(w, wts)
    m.set_context(ctx)
    m.step(T, mode, to_device(target), to_device(u["u_draft"]) if mode == STOCH else None,
           to_device(u["u_accept"]) if mode == STOCH else None,
           to_device(u["u_final"]) if mode == STOCH else None, logits=True)
    torch.cuda.synchronize()
    assert m.status() == 0
    g_tok = m.draft_tok.view(B, k).cpu().numpy()
    g_log = m.draft_logits.view(B, k, V).cpu().numpy()
    g_out = m.out_tok.view(B, k + 1).cpu().numpy()
    g_len = m.accept_len.cpu().numpy()
    g_acc = m.num_accepted.cpu().numpy()
    assert np.all((g_len >= 1) & (g_len <= k + 1)) and np.all(g_acc == g_len - 1)
    # the draft, against the oracle chain teacher-forced with the GPU's drafts
    # (forcing a chain with its own drafts reproduces it, so the free chain
    # serves when nothing diverged)
    ora = ora_d
    if not np.array_equal(g_tok[seqs], ora_d["draft_tok"]):
        ora = oracle_draft(wts, _dims(w), ctx["h"], ctx["last_tok"], ctx["k_cache"], ctx["v_cache"],
                           ctx["ctx_len"], k, T, mode, u["u_draft"], seqs, forced_tok=g_tok[seqs])
    excused = 0
    for i, b in enumerate(seqs):
        for j in range(k):
            ol = ora["draft_logits"][i, j]
            assert rel_l2(g_log[b, j], ol) <= 1e-3, "seq %d depth %d" % (b, j)
            if g_tok[b, j] != ora["draft_tok"][i, j]:
                if mode == GREEDY:
                    assert top2_gap(ol) < 1e-2, "seq %d depth %d" % (b, j)
                else:
                    err = float(np.max(np.abs(g_log[b, j] - ol)))
                    margin = cdf_margin(np.exp((ol - ol.max()) / T), float(u["u_draft"][b, j]))
                    assert margin < 2 * err / T + 1e-6, "seq %d depth %d" % (b, j)
                excused += 1
    # verification, on the GPU's own drafts and draft logits
    gl = g_log[seqs].astype(np.float64)
    o_out, o_len, o_acc = oracle_verify(target[seqs], gl, g_tok[seqs], mode, T, u["u_accept"][seqs],
                                        u["u_final"][seqs])
    for i, b in enumerate(seqs):
        if np.array_equal(g_out[b], o_out[i]) and g_len[b] == o_len[i]:
            continue
        assert mode == STOCH, "greedy outputs differ for sequence %d" % b
        am, sm = stochastic_path_margins(target[b], gl[i], g_tok[b], u["u_accept"][b], float(u["u_final"][b]), T)
        assert am < ACCEPT_BAND or sm < SAMPLE_BAND, "sequence %d: outputs differ (margins %.3g %.3g)" % (b, am, sm)
        excused += 1
    return g_len, excused


@pytest.mark.parametrize("mode", [GREEDY, STOCH])
def test_tiny_step(mode):
    L, exc = run_step_parity(W.TINY, mode, 1.0, seqs=[0], sigma0=0.3)
    L2, _ = run_step_parity(W.TINY, mode, 1.0, seqs=[0], uncorrelated=True)


def test_single_greedy_full_size_step():
    L, exc = run_step_parity(W.SINGLE_GREEDY, GREEDY, 1.0, seqs=[0], sigma0=0.01)
    print("full-size greedy correlated: accept_len", L, "excused", exc)


def test_batched_stochastic_full_size_sampled():
    w = W.BATCHED_STOCHASTIC
    L, exc = run_step_parity(w, STOCH, w.T, seqs=[0, 37, 63])
    print("batched stochastic: mean accept_len %.3f excused %d" % (L.mean(), exc))


def test_deep_chain_full_size_sampled():
    w = W.DEEP_CHAIN
    L, exc = run_step_parity(w, STOCH, w.T, seqs=[5])
    print("deep chain: mean accept_len %.3f excused %d" % (L.mean(), exc))
