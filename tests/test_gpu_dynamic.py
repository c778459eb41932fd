"""GPU parity of the dynamic draft length (mtp_draft_dynamic, spec_verify_dynamic,
spec_step_dynamic) against the oracle: the drafts each sequence keeps, the
drafts and logits up to its stopping depth, the verification over its kept
drafts, and the early return of a chain whose every sequence has stopped."""

import numpy as np
import pytest
import torch

from mtp_speculative_decoding_draft_gb300 import binding as bd
from mtp_speculative_decoding_draft_gb300 import workloads as W
from mtp_speculative_decoding_draft_gb300.model import DraftModule, to_device
from oracle.block import Dims, draft_confidence, dynamic_depths, mtp_draft as oracle_draft
from oracle.verify import spec_verify as oracle_verify
from parity_helpers import check_excused, excuse_draft_token, excuse_verify, rel_l2, stochastic_path_margins

pytestmark = pytest.mark.gpu

GREEDY, STOCH = 0, 1

DYN = W.Workload("dyn_b3_d256_v5003", B=3, k=4, V=5003, d=256, Hq=4, Hkv=2, Dh=64, F=768,
                 ctx=(1, 200), T=0.8, seed=2201)
DYN_TC = W.Workload("dyn_tc_b20_d256_v5003", B=20, k=3, V=5003, d=256, Hq=4, Hkv=2, Dh=64, F=768,
                    ctx=(1, 200), T=0.8, seed=2202)
ONE = W.Workload("dyn_b1_d256_v5003", B=1, k=3, V=5003, d=256, Hq=4, Hkv=2, Dh=64, F=768,
                 ctx=50, T=1.0, seed=2203)


def _dims(w):
    return Dims(w.B, w.d, w.Hq, w.Hkv, w.Dh, w.F, w.V, w.Lmax, w.eps)


def _threshold(conf):
    """A stop_p between the chains' confidences, far (relatively) from each."""
    c = np.sort(conf.ravel())
    gaps = [(c[i + 1] / c[i], i) for i in range(len(c) - 1)]
    r, i = max(gaps)
    assert r > 1.001
    return float(np.sqrt(c[i] * c[i + 1]))


def _oracle_chain(w, mode, seqs):
    wts = W.make_weights(w)
    ctx = W.make_context(w)
    u = W.make_uniforms(w)
    ora = oracle_draft(wts, _dims(w), ctx["h"], ctx["last_tok"], ctx["k_cache"], ctx["v_cache"],
                       ctx["ctx_len"], w.k, w.T, mode, u["u_draft"], seqs)
    conf = np.array([[draft_confidence(ora["draft_logits"][i, j], mode, w.T) for j in range(w.k)]
                     for i in range(len(seqs))])
    return wts, ctx, u, ora, conf


def _check_kept(w, mode, wts, ctx, u, stop_p, g_keff, g_log, g_tok, seqs):
    """k_eff equal to the oracle's; logits and tokens equal up to the stop.

    The oracle chain is teacher-forced with the GPU's drafts (its depth j+1
    takes the GPU's draft j), so a token divergence excused by its margin does
    not end the comparison.  k_eff may differ only where a confidence the
    oracle computes on that chain lies within 1e-3 (relative) of stop_p."""
    forced = np.clip(g_tok[seqs], 0, w.V - 1)   # depths past a stop may be unwritten
    ora = oracle_draft(wts, _dims(w), ctx["h"], ctx["last_tok"], ctx["k_cache"], ctx["v_cache"],
                       ctx["ctx_len"], w.k, w.T, mode, u["u_draft"], seqs, forced_tok=forced)
    o_keff = dynamic_depths(ora["draft_logits"], mode, w.T, stop_p)
    excused, n_tok = 0, 0
    for i, b in enumerate(seqs):
        upto = min(int(o_keff[i]), w.k - 1)
        for j in range(upto + 1):
            ol = ora["draft_logits"][i, j]
            assert rel_l2(g_log[b, j], ol) <= 1e-3, "seq %d depth %d" % (b, j)
            n_tok += j < upto
            if j < upto and g_tok[b, j] != ora["draft_tok"][i, j]:
                excused += excuse_draft_token(mode, b, j, g_log[b, j], ol, u["u_draft"][b, j], w.T)
        if g_keff[b] != o_keff[i]:
            conf = [draft_confidence(ora["draft_logits"][i, j], mode, w.T) for j in range(upto + 1)]
            near = min(abs(c / stop_p - 1.0) for c in conf)
            assert near < 1e-3, "seq %d: k_eff %d, oracle %d" % (b, g_keff[b], o_keff[i])
    check_excused(excused, max(n_tok, 1), "draft tokens", "draft_sample" if mode == STOCH else "default")
    return o_keff


@pytest.mark.parametrize("mode", [GREEDY, STOCH])
@pytest.mark.parametrize("w", [DYN, DYN_TC], ids=["gemv", "tensor_core"])
def test_draft_dynamic(w, mode):
    seqs = list(range(w.B)) if w.B <= 4 else [0, 5, 11, 19]
    wts, ctx, u, ora, conf = _oracle_chain(w, mode, seqs)
    stop_p = _threshold(conf)
    m = DraftModule(w, wts)
    m.set_context(ctx)
    k_eff = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    bd.mtp_draft_dynamic(m.dims, m.wptr, m.h, m.last_tok, m.k_cache, m.v_cache, m.ctx_len, w.k, w.T, mode,
                         stop_p, to_device(u["u_draft"]) if mode == STOCH else None, m.draft_tok, m.draft_logits,
                         k_eff, m.ws)
    torch.cuda.synchronize()
    assert m.status() == 0
    g_keff = k_eff.cpu().numpy()
    assert np.all((g_keff >= 0) & (g_keff <= w.k))
    o_keff = _check_kept(w, mode, wts, ctx, u, stop_p, g_keff, m.draft_logits.view(w.B, w.k, w.V).cpu().numpy(),
                         m.draft_tok.view(w.B, w.k).cpu().numpy(), seqs)
    print("k_eff", list(o_keff), "stop_p %.4g" % stop_p)
    # a threshold of zero never stops, one above 1 stops at once
    for sp, expect in ((0.0, w.k), (1.5, 0)):
        m.set_context(ctx)
        bd.mtp_draft_dynamic(m.dims, m.wptr, m.h, m.last_tok, m.k_cache, m.v_cache, m.ctx_len, w.k, w.T, mode,
                             sp, to_device(u["u_draft"]) if mode == STOCH else None, m.draft_tok, m.draft_logits,
                             k_eff, m.ws)
        torch.cuda.synchronize()
        assert np.all(k_eff.cpu().numpy() == expect)


def test_stopped_chain_skips_the_later_depths():
    """B = 1, stop at depth 0: the later depths' kernels return early, so their
    logits, drafts and K/V rows are never written."""
    w = ONE
    wts = W.make_weights(w)
    ctx = W.make_context(w)
    m = DraftModule(w, wts)
    m.set_context(ctx)
    k_eff = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.draft_logits.fill_(float("nan"))
    m.draft_tok.fill_(-5)
    bd.mtp_draft_dynamic(m.dims, m.wptr, m.h, m.last_tok, m.k_cache, m.v_cache, m.ctx_len, w.k, 1.0, GREEDY,
                         1.5, None, m.draft_tok, m.draft_logits, k_eff, m.ws)
    torch.cuda.synchronize()
    assert m.status() == 0 and int(k_eff.item()) == 0
    lg = m.draft_logits.view(w.k, w.V).cpu().numpy()
    assert np.all(np.isfinite(lg[0])) and np.all(np.isnan(lg[1:]))
    assert list(m.draft_tok.cpu().numpy()[1:]) == [-5] * (w.k - 1)
    kc = m.k_cache.view(torch.int16).cpu().numpy().view(np.uint16)
    L = int(ctx["ctx_len"][0])
    assert not np.array_equal(kc[0, :, L], ctx["k_cache"][0, :, L])          # depth 0 appended its row
    assert np.array_equal(kc[0, :, L + 1:], ctx["k_cache"][0, :, L + 1:])    # nothing after it
    # the same call without a stop runs every depth
    m.set_context(ctx)
    bd.mtp_draft_dynamic(m.dims, m.wptr, m.h, m.last_tok, m.k_cache, m.v_cache, m.ctx_len, w.k, 1.0, GREEDY,
                         0.0, None, m.draft_tok, m.draft_logits, k_eff, m.ws)
    torch.cuda.synchronize()
    assert int(k_eff.item()) == w.k and np.all(np.isfinite(m.draft_logits.cpu().numpy()))


@pytest.mark.parametrize("mode", [GREEDY, STOCH])
def test_verify_dynamic(mode):
    w = W.Workload("dynv_b9_v5003", B=9, k=4, V=5003, T=0.9, mode=mode, target_std=2.0,
                   draft_noise_std0=0.6, seed=2204)
    inp = W.verify_inputs(w)
    t, dl = inp["target_logits"], inp["draft_logits"]
    rng = np.random.default_rng(5)
    d = np.array([[int(np.argmax(t[b, j])) if rng.random() < 0.7 else int(rng.integers(w.V))
                   for j in range(w.k)] for b in range(w.B)], dtype=np.int32)
    ke = np.array([0, 1, 2, 3, 4, 2, 0, 4, 1], dtype=np.int32)
    ver = bd.alloc_workspace(bd.verify_workspace_size(w.B, w.k, w.V))
    out = torch.zeros(w.B * (w.k + 1), dtype=torch.int32, device="cuda")
    alen = torch.zeros(w.B, dtype=torch.int32, device="cuda")
    nacc = torch.zeros(w.B, dtype=torch.int32, device="cuda")
    for _ in range(2):   # twice: the call leaves its state zero for the next
        bd.spec_verify_dynamic(w.B, w.k, w.V, w.T, mode, to_device(t), to_device(dl), to_device(d), to_device(ke),
                               to_device(inp["u_accept"]) if mode == STOCH else None,
                               to_device(inp["u_final"]) if mode == STOCH else None, out, alen, nacc, ver)
        torch.cuda.synchronize()
        assert bd.get_status(ver) == 0
        g_out = out.view(w.B, w.k + 1).cpu().numpy()
        g_len = alen.cpu().numpy()
        o_out, o_len, o_acc = oracle_verify(t, dl, d, mode, w.T, inp["u_accept"], inp["u_final"], k_eff=ke)
        assert np.all(g_len <= ke + 1) and np.array_equal(nacc.cpu().numpy(), g_len - 1)
        n_exc = 0
        for b in range(w.B):
            if np.array_equal(g_out[b], o_out[b]) and g_len[b] == o_len[b]:
                continue
            assert mode == STOCH, "greedy sequence %d differs" % b
            kb = int(ke[b])
            am, sm = stochastic_path_margins(t[b, :kb + 1], dl[b, :kb], d[b, :kb], inp["u_accept"][b, :kb],
                                             float(inp["u_final"][b]), w.T)
            n_exc += excuse_verify(b, am, sm)
        check_excused(n_exc, w.B, "verify outputs")


@pytest.mark.parametrize("mode", [GREEDY, STOCH])
def test_step_dynamic(mode):
    """Draft with a stop, then verify over the kept drafts, in one call: the
    outputs equal the oracle's verification of the GPU's own drafts and k_eff."""
    w = DYN
    seqs = list(range(w.B))
    wts, ctx, u, ora, conf = _oracle_chain(w, mode, seqs)
    stop_p = _threshold(conf)
    wn = W.Workload(w.name, B=w.B, k=w.k + 1, V=w.V, seed=w.seed, draft_noise_std0=0.4, noise_growth=1.5)
    target = W.draft_noise(wn, w.k + 1)
    for b in seqs:
        for j in range(w.k + 1):
            target[b, j] += ora["draft_logits"][b, min(j, w.k - 1)].astype(np.float32)
    m = DraftModule(w, wts)
    m.set_context(ctx)
    k_eff = torch.zeros(w.B, dtype=torch.int32, device="cuda")
    st = mode == STOCH
    bd.spec_step_dynamic(m.dims, m.wptr, m.h, m.last_tok, m.k_cache, m.v_cache, m.ctx_len, w.k, w.T, mode, stop_p,
                         to_device(u["u_draft"]) if st else None, to_device(target),
                         to_device(u["u_accept"]) if st else None, to_device(u["u_final"]) if st else None,
                         m.draft_tok, m.draft_logits, k_eff, m.out_tok, m.accept_len, m.num_accepted, m.ws)
    torch.cuda.synchronize()
    assert m.status() == 0
    g_keff = k_eff.cpu().numpy()
    g_tok = m.draft_tok.view(w.B, w.k).cpu().numpy()
    g_log = m.draft_logits.view(w.B, w.k, w.V).cpu().numpy()
    _check_kept(w, mode, wts, ctx, u, stop_p, g_keff, g_log, g_tok, seqs)
    g_out = m.out_tok.view(w.B, w.k + 1).cpu().numpy()
    g_len = m.accept_len.cpu().numpy()
    assert np.all((g_len >= 1) & (g_len <= g_keff + 1))
    o_out, o_len, _ = oracle_verify(target, g_log.astype(np.float64), g_tok, mode, w.T, u["u_accept"], u["u_final"],
                                    k_eff=g_keff)
    n_exc = 0
    for b in seqs:
        if np.array_equal(g_out[b], o_out[b]) and g_len[b] == o_len[b]:
            continue
        assert mode == STOCH, "greedy sequence %d differs" % b
        kb = int(g_keff[b])
        am, sm = stochastic_path_margins(target[b, :kb + 1], g_log[b, :kb].astype(np.float64), g_tok[b, :kb],
                                         u["u_accept"][b, :kb], float(u["u_final"][b]), w.T)
        n_exc += excuse_verify(b, am, sm)
    check_excused(n_exc, len(seqs), "verify outputs")
