"""Pins of the oracle's chain over distinct modules (one module per depth, as
DeepSeek-V3 trains them: "Optimize vLLM speculative decoding with FastMTP
heads", sections "What is multi-token prediction?" and "Why fine-tune a single
MTP head").

Each depth is rebuilt here from the one-application function ``draft_depth``
(pinned on its own in test_oracle_block.py), with the module, the cache and the
cache rows each depth must see written out by hand.
"""

import numpy as np

from oracle.block import (GREEDY, STOCHASTIC, Dims, draft_depth, module_of_depth, mtp_draft,
                          mtp_draft_modules, select_token)
from oracle.numerics import as_f64, round_f32
from mtp_speculative_decoding_draft_gb300 import workloads as W


def _setup(n_modules):
    w = W.TINY
    dims = Dims(w.B, w.d, w.Hq, w.Hkv, w.Dh, w.F, w.V, w.Lmax, w.eps)
    ctx = W.make_context(w)
    mods = []
    for m in range(n_modules):
        kc, vc = W.make_module_cache(w, m)
        mods.append((W.make_module_weights(w, m), kc, vc))
    return w, dims, ctx, mods


def test_module_of_depth():
    assert [module_of_depth(j, 1) for j in range(4)] == [0, 0, 0, 0]
    assert [module_of_depth(j, 4) for j in range(4)] == [0, 1, 2, 3]
    assert [module_of_depth(j, 2) for j in range(4)] == [0, 1, 1, 1]


def test_module_zero_is_the_single_module():
    w, dims, ctx, mods = _setup(2)
    assert all(np.array_equal(mods[0][0][n], W.make_weights(w)[n]) for n in mods[0][0])
    assert np.array_equal(mods[0][1], ctx["k_cache"]) and np.array_equal(mods[0][2], ctx["v_cache"])
    # the shared embedding / head, distinct everything else
    assert np.array_equal(mods[1][0]["E"], mods[0][0]["E"])
    assert not np.array_equal(mods[1][0]["fc"], mods[0][0]["fc"])
    assert not np.array_equal(mods[1][1], mods[0][1])


def _by_hand(dims, ctx, mods, k, T, mode, u):
    """The chain written out: depth j runs module min(j, n-1) over that module's
    context rows plus the rows earlier depths appended to the same cache."""
    L = int(ctx["ctx_len"][0])
    keys = [as_f64(kc[0, :, :L, :]) for (_, kc, _) in mods]
    values = [as_f64(vc[0, :, :L, :]) for (_, _, vc) in mods]
    x = as_f64(ctx["h"])
    tok = ctx["last_tok"].astype(np.int64)
    logits_all, toks, rows = [], [], []
    for j in range(k):
        m = min(j, len(mods) - 1)
        rows.append(keys[m].shape[1])
        x, logits, kn, vn = draft_depth(mods[m][0], dims, x, tok, [keys[m]], [values[m]])
        logits = round_f32(logits)
        t = select_token(logits[0], mode, T, None if mode == GREEDY else float(u[0, j]))
        keys[m] = np.concatenate([keys[m], kn[0][:, None]], axis=1)
        values[m] = np.concatenate([values[m], vn[0][:, None]], axis=1)
        logits_all.append(logits[0])
        toks.append(t)
        tok = np.array([t])
    return np.array(logits_all), np.array(toks), np.array(rows)


def test_chain_of_distinct_modules_by_hand():
    for n_modules, k in ((3, 3), (2, 3), (1, 3)):
        w, dims, ctx, mods = _setup(n_modules)
        u = W.make_uniforms(w)["u_draft"]
        for mode in (GREEDY, STOCHASTIC):
            res = mtp_draft_modules(mods, dims, ctx["h"], ctx["last_tok"], ctx["ctx_len"], k, 0.8, mode, u)
            lg, tk, rows = _by_hand(dims, ctx, mods, k, 0.8, mode, u)
            np.testing.assert_array_equal(res["draft_logits"][0], lg)
            np.testing.assert_array_equal(res["draft_tok"][0], tk)
            np.testing.assert_array_equal(res["row"][0], rows)
            L = int(ctx["ctx_len"][0])
            expect_rows = [L + j - min(j, n_modules - 1) for j in range(k)]
            assert list(rows) == expect_rows
            assert list(res["module"]) == [min(j, n_modules - 1) for j in range(k)]


def test_one_module_equals_the_reused_module_chain():
    w, dims, ctx, mods = _setup(1)
    u = W.make_uniforms(w)["u_draft"]
    a = mtp_draft(mods[0][0], dims, ctx["h"], ctx["last_tok"], ctx["k_cache"], ctx["v_cache"],
                  ctx["ctx_len"], 3, 1.0, STOCHASTIC, u)
    lg, tk, rows = _by_hand(dims, ctx, mods, 3, 1.0, STOCHASTIC, u)
    np.testing.assert_array_equal(a["draft_logits"][0], lg)
    assert list(rows) == [int(ctx["ctx_len"][0]) + j for j in range(3)]


def test_a_module_affects_only_its_depths_and_later():
    w, dims, ctx, mods = _setup(3)
    base = mtp_draft_modules(mods, dims, ctx["h"], ctx["last_tok"], ctx["ctx_len"], 3, 1.0, GREEDY)
    W2 = dict(mods[2][0])
    W2["wdown"] = W.to_bf16_bits(-as_f64(W2["wdown"]).astype(np.float32))  # flip module 2's MLP output
    mods2 = [mods[0], mods[1], (W2, mods[2][1], mods[2][2])]
    alt = mtp_draft_modules(mods2, dims, ctx["h"], ctx["last_tok"], ctx["ctx_len"], 3, 1.0, GREEDY)
    np.testing.assert_array_equal(base["draft_logits"][:, :2], alt["draft_logits"][:, :2])
    assert not np.array_equal(base["draft_logits"][:, 2], alt["draft_logits"][:, 2])
    # and a module's cache is its own: module 1's context never reaches depth 0
    kc1 = mods[1][1].copy()
    kc1[:] = 0
    mods3 = [mods[0], (mods[1][0], kc1, mods[1][2]), mods[2]]
    alt3 = mtp_draft_modules(mods3, dims, ctx["h"], ctx["last_tok"], ctx["ctx_len"], 3, 1.0, GREEDY)
    np.testing.assert_array_equal(base["draft_logits"][:, 0], alt3["draft_logits"][:, 0])
    assert not np.array_equal(base["draft_logits"][:, 1], alt3["draft_logits"][:, 1])
