"""GPU parity of spec_step (draft chain + verification in one call).

The GPU drafts with its own kernels and verifies its own drafts.  The draft is
compared with the oracle chain teacher-forced with the GPU's drafts (oracle
depth j+1 takes the GPU's draft j and keeps its own hidden state); the outputs
with the oracle's verification of the GPU's own drafts and draft logits,
identical except where a decision lies within 1e-6 of its boundary.  Target
logits are built from the ORACLE's draft logits plus seeded noise (position j
gets std sigma0 * 1.5^j; the bonus row reuses the last draft row), so drafts
are accepted often enough to exercise every branch.  Every sequence of the
batch is compared, at the full batched (64) and deep-chain (32) sizes too.
"""

import numpy as np
import pytest
import torch

from mtp_speculative_decoding_draft_gb300 import workloads as W
from mtp_speculative_decoding_draft_gb300.model import DraftModule, to_device
from oracle.block import Dims, mtp_draft as oracle_draft
from oracle.numerics import bf16_bits_to_f64
from oracle.verify import spec_verify as oracle_verify
from parity_helpers import (bf16_ulp_ok, check_excused, excuse_draft_token, excuse_verify, kv_sum_abs, rel_l2,
                            stochastic_path_margins)

pytestmark = pytest.mark.gpu

GREEDY, STOCH = 0, 1


def _dims(w):
    return Dims(w.B, w.d, w.Hq, w.Hkv, w.Dh, w.F, w.V, w.Lmax, w.eps)


def run_step_parity(w, mode, T, seqs=None, sigma0=None, uncorrelated=False):
    """One spec_step call; every sequence in seqs (all by default) is compared:
    draft logits and tokens at every depth, the K/V rows each depth appended
    (and every other cache row untouched), and the verification outputs."""
    wts = W.make_weights(w)
    ctx = W.make_context(w)
    u = W.make_uniforms(w)
    k, B, V = w.k, w.B, w.V
    seqs = list(range(B)) if seqs is None else list(seqs)
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
    m.check_canaries()
    g_tok = m.draft_tok.view(B, k).cpu().numpy()
    g_log = m.draft_logits.view(B, k, V).cpu().numpy()
    g_out = m.out_tok.view(B, k + 1).cpu().numpy()
    g_len = m.accept_len.cpu().numpy()
    g_acc = m.num_accepted.cpu().numpy()
    g_kc = m.k_cache.view(torch.int16).cpu().numpy().view(np.uint16)
    g_vc = m.v_cache.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.all((g_len >= 1) & (g_len <= k + 1)) and np.all(g_acc == g_len - 1)
    # the draft, against the oracle chain teacher-forced with the GPU's drafts
    # (forcing a chain with its own drafts reproduces it, so the free chain
    # serves when nothing diverged)
    ora = ora_d
    if not np.array_equal(g_tok[seqs], ora_d["draft_tok"]):
        ora = oracle_draft(wts, _dims(w), ctx["h"], ctx["last_tok"], ctx["k_cache"], ctx["v_cache"],
                           ctx["ctx_len"], k, T, mode, u["u_draft"], seqs, forced_tok=g_tok[seqs])
    mags = [kv_sum_abs(wts, ora["attn_in"][:, j]) for j in range(k)]
    excused = 0
    for i, b in enumerate(seqs):
        L = int(ctx["ctx_len"][b])
        for j in range(k):
            ol = ora["draft_logits"][i, j]
            assert rel_l2(g_log[b, j], ol) <= 1e-3, "seq %d depth %d" % (b, j)
            assert bf16_ulp_ok(bf16_bits_to_f64(g_kc[b, :, L + j, :]), ora["k_new"][i, j], mags[j][0][i]), \
                "seq %d depth %d: K row" % (b, j)
            assert bf16_ulp_ok(bf16_bits_to_f64(g_vc[b, :, L + j, :]), ora["v_new"][i, j], mags[j][1][i]), \
                "seq %d depth %d: V row" % (b, j)
            if g_tok[b, j] != ora["draft_tok"][i, j]:
                excused += excuse_draft_token(mode, b, j, g_log[b, j], ol, u["u_draft"][b, j], T)
        # every cache row outside the appended window is untouched
        keep = np.ones(g_kc.shape[2], bool)
        keep[L:L + k] = False
        assert np.array_equal(g_kc[b][:, keep], ctx["k_cache"][b][:, keep]), "seq %d: K cache" % b
        assert np.array_equal(g_vc[b][:, keep], ctx["v_cache"][b][:, keep]), "seq %d: V cache" % b
    check_excused(excused, len(seqs) * k, "draft tokens", "draft_sample" if mode == STOCH else "default")
    # verification, on the GPU's own drafts and draft logits
    gl = g_log[seqs].astype(np.float64)
    o_out, o_len, o_acc = oracle_verify(target[seqs], gl, g_tok[seqs], mode, T, u["u_accept"][seqs],
                                        u["u_final"][seqs])
    n_exc = 0
    for i, b in enumerate(seqs):
        if np.array_equal(g_out[b], o_out[i]) and g_len[b] == o_len[i]:
            continue
        assert mode == STOCH, "greedy outputs differ for sequence %d" % b
        am, sm = stochastic_path_margins(target[b], gl[i], g_tok[b], u["u_accept"][b], float(u["u_final"][b]), T)
        n_exc += excuse_verify(b, am, sm)
    check_excused(n_exc, len(seqs), "verify outputs")
    return g_len, excused + n_exc


@pytest.mark.parametrize("mode", [GREEDY, STOCH])
def test_tiny_step(mode):
    L, exc = run_step_parity(W.TINY, mode, 1.0, seqs=[0], sigma0=0.3)
    L2, _ = run_step_parity(W.TINY, mode, 1.0, seqs=[0], uncorrelated=True)


def test_single_greedy_full_size_step():
    L, exc = run_step_parity(W.SINGLE_GREEDY, GREEDY, 1.0, seqs=[0], sigma0=0.01)
    print("full-size greedy correlated: accept_len", L, "excused", exc)


def test_batched_stochastic_full_size():
    w = W.BATCHED_STOCHASTIC
    L, exc = run_step_parity(w, STOCH, w.T)
    print("batched stochastic: mean accept_len %.3f excused %d" % (L.mean(), exc))


def test_deep_chain_full_size():
    w = W.DEEP_CHAIN
    L, exc = run_step_parity(w, STOCH, w.T)
    print("deep chain: mean accept_len %.3f excused %d" % (L.mean(), exc))
