"""GPU parity of the chain over distinct modules (mtp_draft_modules and
spec_step_modules) against the oracle: module m's weights and K/V cache at the
depths that run it, its cache rows at ctx_len + (earlier depths on the same
module), every other cache row untouched."""

import numpy as np
import pytest
import torch

from mtp_speculative_decoding_draft_gb300 import binding as bd
from mtp_speculative_decoding_draft_gb300 import workloads as W
from mtp_speculative_decoding_draft_gb300.model import Guarded, to_device, to_device_bf16
from oracle.block import Dims, mtp_draft_modules as oracle_draft_modules
from oracle.numerics import bf16_bits_to_f64
from oracle.verify import spec_verify as oracle_verify
from parity_helpers import (bf16_ulp_ok, check_excused, excuse_draft_token, excuse_verify, kv_sum_abs, rel_l2,
                            stochastic_path_margins)

pytestmark = pytest.mark.gpu

GREEDY, STOCH = 0, 1

# GEMV path (a batch of three), ragged vocabulary, contexts from 1 to 200.
MODS = W.Workload("mods_b3_d256_v5003", B=3, k=3, V=5003, d=256, Hq=4, Hkv=2, Dh=64, F=768,
                  ctx=(1, 200), T=0.8, seed=2101)
# Tensor-core path (a batch of 20).
MODS_TC = W.Workload("mods_tc_b20_d256_v5003", B=20, k=3, V=5003, d=256, Hq=4, Hkv=2, Dh=64, F=768,
                     ctx=(1, 200), T=0.8, seed=2102)


def _dims(w):
    return Dims(w.B, w.d, w.Hq, w.Hkv, w.Dh, w.F, w.V, w.Lmax, w.eps)


class Modules:
    """n_modules modules' weights and caches on the device, plus the numpy copies."""

    def __init__(self, w, n_modules, ctx_fix=None):
        self.w = w
        self.ctx = W.make_context(w)
        if ctx_fix is not None:
            self.ctx["ctx_len"][:len(ctx_fix)] = ctx_fix
        self.host = []
        self.dev = []
        for m in range(n_modules):
            wts = W.make_module_weights(w, m)
            kc, vc = W.make_module_cache(w, m)
            self.host.append((wts, kc, vc))
            self.dev.append(({n: to_device_bf16(wts[n]) for n in bd.WEIGHT_FIELDS}, to_device_bf16(kc),
                             to_device_bf16(vc)))
        self.arr = bd.make_modules(self.dev)
        self.dims = bd.make_dims(w.B, w.d, w.Hq, w.Hkv, w.Dh, w.F, w.V, w.Lmax, w.eps)
        self.guard = Guarded()
        self.ws = self.guard.alloc("workspace", bd.workspace_size(self.dims, w.k), torch.uint8)
        self.h = to_device_bf16(self.ctx["h"])
        self.last_tok = to_device(self.ctx["last_tok"].astype(np.int32))
        self.ctx_len = to_device(self.ctx["ctx_len"].astype(np.int32))
        B, k, V = w.B, w.k, w.V
        self.draft_tok = self.guard.alloc("draft_tok", B * k, torch.int32)
        self.draft_logits = self.guard.alloc("draft_logits", B * k * V, torch.float32)

    def caches(self):
        return [(kc.view(torch.int16).cpu().numpy().view(np.uint16), vc.view(torch.int16).cpu().numpy().view(np.uint16))
                for (_, kc, vc) in self.dev]


def gpu_tokens(M):
    return M.draft_tok.view(M.w.B, M.w.k).cpu().numpy()


def check_draft(M, ora, mode, T, u, seqs):
    """ora: the oracle chain teacher-forced with the GPU's drafts (its depth
    j+1 takes the GPU's draft j), so every depth is compared."""
    w = M.w
    B, k, V = w.B, w.k, w.V
    torch.cuda.synchronize()
    M.guard.check()
    g_tok = M.draft_tok.view(B, k).cpu().numpy()
    g_log = M.draft_logits.view(B, k, V).cpu().numpy()
    caches = M.caches()
    n_mod = len(M.host)
    written = [np.zeros((B, w.Lmax), bool) for _ in range(n_mod)]
    excused = 0
    # sum_i |w_i n_i| of every appended K/V entry, per depth (that depth's module)
    mags = [kv_sum_abs(M.host[int(ora["module"][j])][0], ora["attn_in"][:, j]) for j in range(k)]
    for i, b in enumerate(seqs):
        for j in range(k):
            m = int(ora["module"][j])
            row = int(ora["row"][i, j])
            written[m][b, row] = True
            ol = ora["draft_logits"][i, j]
            assert rel_l2(g_log[b, j], ol) <= 1e-3, "seq %d depth %d" % (b, j)
            gk, gv = caches[m]
            assert bf16_ulp_ok(bf16_bits_to_f64(gk[b, :, row, :]), ora["k_new"][i, j], mags[j][0][i]), (b, j)
            assert bf16_ulp_ok(bf16_bits_to_f64(gv[b, :, row, :]), ora["v_new"][i, j], mags[j][1][i]), (b, j)
            if g_tok[b, j] != ora["draft_tok"][i, j]:
                excused += excuse_draft_token(mode, b, j, g_log[b, j], ol, u[b, j], T)
    # every row no depth wrote is untouched, in every module's cache
    for m in range(n_mod):
        gk, gv = caches[m]
        _, kc, vc = M.host[m]
        for b in seqs:
            keep = ~written[m][b]
            assert np.array_equal(gk[b][:, keep], kc[b][:, keep]), "module %d seq %d" % (m, b)
            assert np.array_equal(gv[b][:, keep], vc[b][:, keep]), "module %d seq %d" % (m, b)
    check_excused(excused, len(seqs) * k, "draft tokens", "draft_sample" if mode == STOCH else "default")
    return excused


@pytest.mark.parametrize("n_modules", [3, 2])
@pytest.mark.parametrize("mode", [GREEDY, STOCH])
def test_modules_gemv_path(n_modules, mode):
    w = MODS
    M = Modules(w, n_modules, ctx_fix=[1, 77, 200])
    u = W.make_uniforms(w)["u_draft"]
    bd.mtp_draft_modules(M.dims, M.arr, M.h, M.last_tok, M.ctx_len, w.k, w.T, mode,
                         to_device(u) if mode == STOCH else None, M.draft_tok, M.draft_logits, M.ws)
    torch.cuda.synchronize()
    assert bd.get_status(M.ws) == 0
    seqs = list(range(w.B))
    ora = oracle_draft_modules(M.host, _dims(w), M.ctx["h"], M.ctx["last_tok"], M.ctx["ctx_len"], w.k, w.T,
                               mode, u, seqs, forced_tok=gpu_tokens(M)[seqs])
    check_draft(M, ora, mode, w.T, u, seqs)


@pytest.mark.parametrize("mode", [GREEDY, STOCH])
def test_modules_tensor_core_path(mode):
    w = MODS_TC
    M = Modules(w, 3)
    u = W.make_uniforms(w)["u_draft"]
    bd.mtp_draft_modules(M.dims, M.arr, M.h, M.last_tok, M.ctx_len, w.k, w.T, mode,
                         to_device(u) if mode == STOCH else None, M.draft_tok, M.draft_logits, M.ws)
    torch.cuda.synchronize()
    assert bd.get_status(M.ws) == 0
    seqs = [0, 7, 19]
    ora = oracle_draft_modules(M.host, _dims(w), M.ctx["h"], M.ctx["last_tok"], M.ctx["ctx_len"], w.k, w.T,
                               mode, u, seqs, forced_tok=gpu_tokens(M)[seqs])
    check_draft(M, ora, mode, w.T, u, seqs)


def test_spec_step_modules_stochastic():
    """The draft over three modules, then verification of the GPU's own drafts:
    the outputs equal the oracle's verification of the same drafts and logits."""
    w = MODS
    M = Modules(w, 3)
    uu = W.make_uniforms(w)
    B, k, V = w.B, w.k, w.V
    seqs = list(range(B))
    ora = oracle_draft_modules(M.host, _dims(w), M.ctx["h"], M.ctx["last_tok"], M.ctx["ctx_len"], k, w.T,
                               STOCH, uu["u_draft"], seqs)
    wn = W.Workload(w.name, B=B, k=k + 1, V=V, seed=w.seed, draft_noise_std0=0.5, noise_growth=1.5)
    target = W.draft_noise(wn, k + 1)
    for b in seqs:
        for j in range(k + 1):
            target[b, j] += ora["draft_logits"][b, min(j, k - 1)].astype(np.float32)
    out_tok = M.guard.alloc("out_tok", B * (k + 1), torch.int32)
    alen = M.guard.alloc("accept_len", B, torch.int32)
    nacc = M.guard.alloc("num_accepted", B, torch.int32)
    bd.spec_step_modules(M.dims, M.arr, M.h, M.last_tok, M.ctx_len, k, w.T, STOCH, to_device(uu["u_draft"]),
                         to_device(target), to_device(uu["u_accept"]), to_device(uu["u_final"]), M.draft_tok,
                         M.draft_logits, out_tok, alen, nacc, M.ws)
    torch.cuda.synchronize()
    assert bd.get_status(M.ws) == 0
    ora_tf = oracle_draft_modules(M.host, _dims(w), M.ctx["h"], M.ctx["last_tok"], M.ctx["ctx_len"], k, w.T,
                                  STOCH, uu["u_draft"], seqs, forced_tok=gpu_tokens(M)[seqs])
    check_draft(M, ora_tf, STOCH, w.T, uu["u_draft"], seqs)
    g_tok = M.draft_tok.view(B, k).cpu().numpy()
    g_log = M.draft_logits.view(B, k, V).cpu().numpy()
    g_out = out_tok.view(B, k + 1).cpu().numpy()
    g_len = alen.cpu().numpy()
    assert np.all((g_len >= 1) & (g_len <= k + 1)) and np.array_equal(nacc.cpu().numpy(), g_len - 1)
    # verification of the GPU's own drafts, re-done by the oracle
    o_out, o_len, _ = oracle_verify(target, g_log.astype(np.float64), g_tok, STOCH, w.T, uu["u_accept"],
                                    uu["u_final"])
    n_exc = 0
    for b in seqs:
        if np.array_equal(g_out[b], o_out[b]) and g_len[b] == o_len[b]:
            continue
        am, sm = stochastic_path_margins(target[b], g_log[b].astype(np.float64), g_tok[b], uu["u_accept"][b],
                                         float(uu["u_final"][b]), w.T)
        n_exc += excuse_verify(b, am, sm)
    check_excused(n_exc, len(seqs), "verify outputs")
