"""GPU parity of mtp_draft (the chained MTP module) against the oracle."""

import numpy as np
import pytest
import torch

from mtp_speculative_decoding_draft_gb300 import workloads as W
from mtp_speculative_decoding_draft_gb300.model import DraftModule, to_device
from oracle.block import Dims, mtp_draft as oracle_draft
from oracle.numerics import bf16_bits_to_f64
from parity_helpers import bf16_ulp_ok, check_excused, excuse_draft_token, kv_sum_abs, rel_l2

pytestmark = pytest.mark.gpu

GREEDY, STOCH = 0, 1

# A mid-size block: several GEMV tiles per matrix, a ragged vocabulary, Dh = 64,
# context lengths from 1 (only the appended rows are seen) to 200.
MID = W.Workload("mid_b3_d256_v5003", B=3, k=4, V=5003, d=256, Hq=4, Hkv=2, Dh=64, F=768,
                 ctx=(1, 200), T=0.8, seed=2001)
# GQA group of 5 query heads per kv head (as in the deep-chain workload), Dh = 128.
GQA5 = W.Workload("gqa5_b2_d640_v3001", B=2, k=2, V=3001, d=640, Hq=10, Hkv=2, Dh=128, F=1280,
                  ctx=(60, 300), T=1.0, seed=2002)


def _dims(w, k):
    return Dims(w.B, w.d, w.Hq, w.Hkv, w.Dh, w.F, w.V, w.ctx_max + k, w.eps)


def run_draft_parity(w, mode, T, ctx_fix=None, master=False, seqs=None):
    if master:
        wts, full = W.make_weights(w, master=True)
    else:
        wts = W.make_weights(w)
    ctx = W.make_context(w)
    if ctx_fix is not None:
        ctx["ctx_len"][:len(ctx_fix)] = ctx_fix
    u = W.make_uniforms(w)
    m = DraftModule(w, wts)
    m.set_context(ctx)
    m.draft(T, mode, to_device(u["u_draft"]) if mode == STOCH else None, logits=True)
    torch.cuda.synchronize()
    assert m.status() == 0
    m.check_canaries()
    B, k, V = w.B, w.k, w.V
    g_tok = m.draft_tok.view(B, k).cpu().numpy()
    g_log = m.draft_logits.view(B, k, V).cpu().numpy()
    g_kc = m.k_cache.view(torch.int16).cpu().numpy().view(np.uint16)
    g_vc = m.v_cache.view(torch.int16).cpu().numpy().view(np.uint16)
    seqs = list(range(B)) if seqs is None else list(seqs)
    # teacher-forced: oracle depth j+1 takes the GPU's draft j, so every depth
    # is compared even past an excused divergence of the tokens
    ora = oracle_draft(wts, _dims(w, k), ctx["h"], ctx["last_tok"], ctx["k_cache"], ctx["v_cache"],
                       ctx["ctx_len"], k, T, mode, u["u_draft"], seqs, forced_tok=g_tok[seqs])
    report = {"excused": 0, "rel_l2": []}
    # sum_i |w_i n_i| of every appended K/V entry, per depth
    mags = [kv_sum_abs(wts, ora["attn_in"][:, j]) for j in range(k)]
    for i, b in enumerate(seqs):
        L = int(ctx["ctx_len"][b])
        for j in range(k):
            ol = ora["draft_logits"][i, j]
            e = rel_l2(g_log[b, j], ol)
            report["rel_l2"].append(e)
            assert e <= 1e-3, "seq %d depth %d: logits rel L2 %.3g" % (b, j, e)
            # the rows this depth appended to the caches
            assert bf16_ulp_ok(bf16_bits_to_f64(g_kc[b, :, L + j, :]), ora["k_new"][i, j], mags[j][0][i]), \
                "seq %d depth %d: K row" % (b, j)
            assert bf16_ulp_ok(bf16_bits_to_f64(g_vc[b, :, L + j, :]), ora["v_new"][i, j], mags[j][1][i]), \
                "seq %d depth %d: V row" % (b, j)
            if g_tok[b, j] != ora["draft_tok"][i, j]:
                report["excused"] += excuse_draft_token(mode, b, j, g_log[b, j], ol, u["u_draft"][b, j], T)
        # rows outside the appended window are untouched
        mask = np.ones(g_kc.shape[2], bool)
        mask[L:L + k] = False
        assert np.array_equal(g_kc[b][:, mask], ctx["k_cache"][b][:, mask])
        assert np.array_equal(g_vc[b][:, mask], ctx["v_cache"][b][:, mask])
    check_excused(report["excused"], len(seqs) * k, "draft tokens", "draft_sample" if mode == STOCH else "default")
    if master:
        om = oracle_draft(full, _dims(w, k), ctx["h"], ctx["last_tok"], ctx["k_cache"], ctx["v_cache"],
                          ctx["ctx_len"], 1, T, mode, u["u_draft"], seqs)
        for i, b in enumerate(seqs):
            e = rel_l2(g_log[b, 0], om["draft_logits"][i, 0])
            assert e <= 1e-2, "seq %d: logits vs fp32-master oracle rel L2 %.3g" % (b, e)
    return report


@pytest.mark.parametrize("mode", [GREEDY, STOCH])
def test_tiny(mode):
    r = run_draft_parity(W.TINY, mode, 1.0, master=True)
    print("tiny mode=%d max rel L2 %.3g excused %d" % (mode, max(r["rel_l2"]), r["excused"]))


@pytest.mark.parametrize("mode", [GREEDY, STOCH])
def test_mid_ragged(mode):
    r = run_draft_parity(MID, mode, MID.T, ctx_fix=[1, 64, 200])
    print("mid mode=%d max rel L2 %.3g excused %d" % (mode, max(r["rel_l2"]), r["excused"]))


@pytest.mark.parametrize("mode", [GREEDY, STOCH])
def test_gqa_group_of_five(mode):
    run_draft_parity(GQA5, mode, GQA5.T)


@pytest.mark.parametrize("T", [0.05, 20.0])
def test_stochastic_temperature_extremes(T):
    """The draft sampler at a near one-hot and a near-uniform temperature."""
    r = run_draft_parity(MID, STOCH, T, ctx_fix=[1, 64, 200])
    print("mid T=%g max rel L2 %.3g excused %d" % (T, max(r["rel_l2"]), r["excused"]))


def test_single_greedy_full_size():
    r = run_draft_parity(W.SINGLE_GREEDY, GREEDY, 1.0)
    print("full-size greedy: rel L2 per depth", ["%.2e" % e for e in r["rel_l2"]])


def test_repeat_calls_are_bitwise_identical():
    w = MID
    wts = W.make_weights(w)
    ctx = W.make_context(w)
    u = to_device(W.make_uniforms(w)["u_draft"])
    m = DraftModule(w, wts)
    outs = []
    for _ in range(3):
        m.set_context(ctx)
        m.draft(w.T, STOCH, u, logits=True)
        torch.cuda.synchronize()
        outs.append((m.draft_tok.cpu().numpy().copy(), m.draft_logits.cpu().numpy().copy()))
    for t, l in outs[1:]:
        assert np.array_equal(t, outs[0][0]) and np.array_equal(l.view(np.uint32), outs[0][1].view(np.uint32))


def test_bad_context_length_sets_status():
    from mtp_speculative_decoding_draft_gb300 import binding as bd
    w = W.TINY
    m = DraftModule(w, W.make_weights(w))
    ctx = W.make_context(w)
    ctx["ctx_len"][0] = w.Lmax      # no room for the k appended rows
    m.set_context(ctx)
    m.draft(1.0, GREEDY)
    torch.cuda.synchronize()
    assert m.status() & bd.STATUS_BAD_CTX


def test_invalid_draft_arguments():
    from mtp_speculative_decoding_draft_gb300 import binding as bd
    w = W.TINY
    m = DraftModule(w, W.make_weights(w))
    m.set_context(W.make_context(w))
    with pytest.raises(bd.MtpError):
        m.draft(0.0, STOCH, to_device(W.make_uniforms(w)["u_draft"]))     # T = 0
    d = bd.make_dims(w.B, 60, w.Hq, w.Hkv, w.Dh, w.F, w.V, w.Lmax)        # d not a multiple of 8
    assert bd.workspace_size(d, 3) == 0
    small = bd.alloc_workspace(256)
    with pytest.raises(bd.MtpError):
        bd.mtp_draft(m.dims, m.wptr, m.h, m.last_tok, m.k_cache, m.v_cache, m.ctx_len, 3, 1.0, GREEDY,
                     None, m.draft_tok, None, small)
