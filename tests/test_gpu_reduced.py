"""GPU parity of the reduced draft vocabulary (mtp_draft_reduced,
spec_step_reduced) against the oracle: the head's logits at their vocabulary
ids and -inf elsewhere, the drafts chosen among the N rows, and the
verification of those drafts over the full vocabulary."""

import numpy as np
import pytest
import torch

from mtp_speculative_decoding_draft_gb300 import binding as bd
from mtp_speculative_decoding_draft_gb300 import workloads as W
from mtp_speculative_decoding_draft_gb300.model import DraftModule, to_device, to_device_bf16
from oracle.block import Dims, mtp_draft as oracle_draft
from oracle.numerics import bf16_bits_to_f64
from oracle.verify import spec_verify as oracle_verify
from parity_helpers import (bf16_ulp_ok, check_excused, excuse_draft_token, excuse_verify, kv_sum_abs, rel_l2,
                            stochastic_path_margins)

pytestmark = pytest.mark.gpu

GREEDY, STOCH = 0, 1

RED = W.Workload("red_b3_d256_v5003", B=3, k=3, V=5003, d=256, Hq=4, Hkv=2, Dh=64, F=768,
                 ctx=(1, 200), T=0.8, seed=2301)
RED_TC = W.Workload("red_tc_b20_d256_v5003", B=20, k=3, V=5003, d=256, Hq=4, Hkv=2, Dh=64, F=768,
                    ctx=(1, 200), T=0.8, seed=2302)


def _dims(w):
    return Dims(w.B, w.d, w.Hq, w.Hkv, w.Dh, w.F, w.V, w.Lmax, w.eps)


def _setup(w, n):
    wts = W.make_weights(w)
    ctx = W.make_context(w)
    u = W.make_uniforms(w)
    vmap, head = W.make_draft_vocab(w, n)
    m = DraftModule(w, wts)
    m.set_context(ctx)
    return wts, ctx, u, vmap, head, m


@pytest.mark.parametrize("mode", [GREEDY, STOCH])
@pytest.mark.parametrize("w", [RED, RED_TC], ids=["gemv", "tensor_core"])
def test_draft_reduced(w, mode):
    n = 1500
    wts, ctx, u, vmap, head, m = _setup(w, n)
    m.draft_logits.fill_(0.0)
    bd.mtp_draft_reduced(m.dims, m.wptr, to_device_bf16(head), to_device(vmap), m.h, m.last_tok, m.k_cache,
                         m.v_cache, m.ctx_len, w.k, w.T, mode, to_device(u["u_draft"]) if mode == STOCH else None,
                         m.draft_tok, m.draft_logits, m.ws)
    torch.cuda.synchronize()
    assert m.status() == 0
    B, k, V = w.B, w.k, w.V
    seqs = list(range(B)) if B <= 4 else [0, 9, 19]
    g_log = m.draft_logits.view(B, k, V).cpu().numpy()
    g_tok = m.draft_tok.view(B, k).cpu().numpy()
    # teacher-forced: oracle depth j+1 takes the GPU's draft j
    ora = oracle_draft(dict(wts, head=head), _dims(w), ctx["h"], ctx["last_tok"], ctx["k_cache"], ctx["v_cache"],
                       ctx["ctx_len"], k, w.T, mode, u["u_draft"], seqs, vocab_map=vmap, forced_tok=g_tok[seqs])
    g_kc = m.k_cache.view(torch.int16).cpu().numpy().view(np.uint16)
    outside = np.ones(V, bool)
    outside[vmap] = False
    ids = set(vmap.tolist())
    mags = [kv_sum_abs(wts, ora["attn_in"][:, j]) for j in range(k)]
    excused = 0
    for i, b in enumerate(seqs):
        L = int(ctx["ctx_len"][b])
        for j in range(k):
            assert np.all(g_log[b, j][outside] == -np.inf), "seq %d depth %d: ids outside the head" % (b, j)
            ol = ora["draft_logits"][i, j][vmap]
            assert rel_l2(g_log[b, j][vmap], ol) <= 1e-3, "seq %d depth %d" % (b, j)
            assert int(g_tok[b, j]) in ids
            assert bf16_ulp_ok(bf16_bits_to_f64(g_kc[b, :, L + j, :]), ora["k_new"][i, j], mags[j][0][i]), (b, j)
            if g_tok[b, j] != ora["draft_tok"][i, j]:
                excused += excuse_draft_token(mode, b, j, g_log[b, j][vmap], ol, u["u_draft"][b, j], w.T)
    check_excused(excused, len(seqs) * k, "draft tokens", "draft_sample" if mode == STOCH else "default")


@pytest.mark.parametrize("w", [RED, RED_TC], ids=["gemv", "tensor_core"])
def test_full_map_reproduces_mtp_draft(w):
    """N = V with the identity map computes exactly what mtp_draft computes."""
    wts, ctx, u, _, _, m = _setup(w, 128)
    ud = to_device(u["u_draft"])
    m.draft(w.T, STOCH, ud, logits=True)
    torch.cuda.synchronize()
    ref_tok, ref_log = m.draft_tok.cpu().numpy().copy(), m.draft_logits.cpu().numpy().copy()
    m.set_context(ctx)
    bd.mtp_draft_reduced(m.dims, m.wptr, m.weights["E"], to_device(np.arange(w.V, dtype=np.int32)), m.h,
                         m.last_tok, m.k_cache, m.v_cache, m.ctx_len, w.k, w.T, STOCH, ud, m.draft_tok,
                         m.draft_logits, m.ws)
    torch.cuda.synchronize()
    assert np.array_equal(m.draft_tok.cpu().numpy(), ref_tok)
    assert np.array_equal(m.draft_logits.cpu().numpy().view(np.uint32), ref_log.view(np.uint32))


@pytest.mark.parametrize("mode", [GREEDY, STOCH])
def test_step_reduced(mode):
    """Draft over the reduced head, then verify over the full vocabulary: the
    outputs equal the oracle's verification of the GPU's own drafts."""
    w = RED
    n = 1200
    wts, ctx, u, vmap, head, m = _setup(w, n)
    rng = np.random.default_rng(7)
    # targets near the full-vocabulary logits (drafts accepted often; ids outside the head carry mass too)
    ora = oracle_draft(dict(wts, head=head), _dims(w), ctx["h"], ctx["last_tok"], ctx["k_cache"], ctx["v_cache"],
                       ctx["ctx_len"], w.k, w.T, mode, u["u_draft"], vocab_map=vmap)
    target = (rng.standard_normal((w.B, w.k + 1, w.V)) * 0.5).astype(np.float32)
    for j in range(w.k + 1):
        row = ora["draft_logits"][:, min(j, w.k - 1)]
        target[:, j] += np.where(np.isfinite(row), row, np.median(row[np.isfinite(row)])).astype(np.float32)
    st = mode == STOCH
    bd.spec_step_reduced(m.dims, m.wptr, to_device_bf16(head), to_device(vmap), m.h, m.last_tok, m.k_cache,
                         m.v_cache, m.ctx_len, w.k, w.T, mode, to_device(u["u_draft"]) if st else None,
                         to_device(target), to_device(u["u_accept"]) if st else None,
                         to_device(u["u_final"]) if st else None, m.draft_tok, m.draft_logits, m.out_tok,
                         m.accept_len, m.num_accepted, m.ws)
    torch.cuda.synchronize()
    assert m.status() == 0
    B, k, V = w.B, w.k, w.V
    g_tok = m.draft_tok.view(B, k).cpu().numpy()
    g_log = m.draft_logits.view(B, k, V).cpu().numpy().astype(np.float64)
    g_out = m.out_tok.view(B, k + 1).cpu().numpy()
    g_len = m.accept_len.cpu().numpy()
    o_out, o_len, _ = oracle_verify(target, g_log, g_tok, mode, w.T, u["u_accept"], u["u_final"])
    n_exc = 0
    for b in range(B):
        if np.array_equal(g_out[b], o_out[b]) and g_len[b] == o_len[b]:
            continue
        assert mode == STOCH, "greedy sequence %d differs" % b
        am, sm = stochastic_path_margins(target[b], g_log[b], g_tok[b], u["u_accept"][b], float(u["u_final"][b]),
                                         w.T)
        n_exc += excuse_verify(b, am, sm)
    check_excused(n_exc, B, "verify outputs")


def test_bad_map_ids_flag_the_status():
    """An id outside [0, V) in the map is reported, never written."""
    w = RED
    wts, ctx, u, vmap, head, m = _setup(w, 300)
    bad = vmap.copy()
    bad[7] = w.V + 5
    bad[8] = -3
    m.draft_logits.fill_(0.0)
    bd.mtp_draft_reduced(m.dims, m.wptr, to_device_bf16(head), to_device(bad), m.h, m.last_tok, m.k_cache,
                         m.v_cache, m.ctx_len, w.k, w.T, STOCH, to_device(u["u_draft"]), m.draft_tok,
                         m.draft_logits, m.ws)
    torch.cuda.synchronize()
    assert m.status() & bd.STATUS_BAD_TOKEN
    lg = m.draft_logits.view(w.B, w.k, w.V).cpu().numpy()
    good = np.delete(bad, [7, 8])
    outside = np.ones(w.V, bool)
    outside[good] = False
    assert np.all(lg[:, :, outside] == -np.inf)   # nothing landed outside the valid ids


def test_reduced_arguments_rejected_on_the_host():
    w = RED
    wts, ctx, u, vmap, head, m = _setup(w, 300)
    small_map, small_head = vmap[:100], head[:100]          # fewer than 128 rows
    with pytest.raises(bd.MtpError):
        bd.mtp_draft_reduced(m.dims, m.wptr, to_device_bf16(small_head), to_device(small_map), m.h, m.last_tok,
                             m.k_cache, m.v_cache, m.ctx_len, w.k, w.T, GREEDY, None, m.draft_tok, None, m.ws)
