"""GPU parity of spec_verify_fused (verification from the target's hidden
states) against the oracle, through the C ABI.

The stochastic call keeps the target's fp32 logits in its workspace (its
residual draw needs them); the test reads them back from there, so that

* the logits are compared with the oracle's float64 head . hidden;
* the stochastic decisions are compared with the oracle's verification of
  those same fp32 logits, identical except within 1e-6 of a boundary;
* the greedy decisions are compared with the oracle's verification of its
  own float64 logits, identical except where the deciding row's top-2 gap is
  below twice that row's measured logit error.
"""

import numpy as np
import pytest
import torch

from mtp_speculative_decoding_draft_gb300 import binding as bd
from mtp_speculative_decoding_draft_gb300 import workloads as W
from mtp_speculative_decoding_draft_gb300.model import FusedVerifier, to_device, to_device_bf16
from oracle.block import linear, select_token
from oracle.numerics import bf16_bits_to_f64
from oracle.verify import spec_verify as oracle_verify, target_logits_from_hidden
from parity_helpers import check_excused, compare_verify, record_excused, rel_l2

pytestmark = pytest.mark.gpu

GREEDY, STOCH = 0, 1
VT = 256  # vocabulary rows per partial in the workspace layout


def _inputs(B, k, V, d, T, seed, noise=0.5, hidden_std=1.0):
    """head ~ N(0, 0.02^2) and hidden ~ N(0, hidden_std^2) as bf16; the oracle's
    float64 target logits; draft = target + N(0, noise^2) (float32); drafts
    drawn from q with the oracle's sampler; uniforms."""
    w = W.Workload("fused_case", B=B, k=k, V=V, d=d, seed=seed)
    head = W.to_bf16_bits(W.normal(seed, "fused.head", (V, d), std=0.02))
    hidden = W.to_bf16_bits(W.normal(seed, "fused.hidden", (B, k + 1, d), std=hidden_std))
    t = target_logits_from_hidden(head, hidden)
    draft = (t[:, :k] + W.normal(seed, "fused.noise", (B, k, V), std=noise)).astype(np.float32)
    u = W.make_uniforms(W.Workload("fused_case", B=B, k=k, V=V, seed=seed))
    dtok = np.array([[select_token(draft[b, j], STOCH, T, float(u["u_draft"][b, j])) for j in range(k)]
                     for b in range(B)], dtype=np.int32)
    return head, hidden, t, draft, dtok, u


def _up256(n):
    return (n + 255) // 256 * 256


def _stored_logits(fv):
    """The stochastic call's fp32 logits [B (k+1), V] from its workspace: after
    the 256-byte status slot, the per-(row, 256-token tile) partials of the
    target rows and those of the draft rows."""
    Na = fv.B * (fv.k + 1)
    n_vt = (fv.V + VT - 1) // VT
    off = 256 + _up256(Na * n_vt * 16) + _up256(fv.B * fv.k * n_vt * 16)
    raw = fv.ws[off:off + Na * fv.V * 4]
    return raw.view(torch.float32).view(Na, fv.V).cpu().numpy()


def run_fused_parity(B, k, V, d, T, seed, noise=0.5):
    head, hidden, t, draft, dtok, u = _inputs(B, k, V, d, T, seed, noise)
    head_d, hid_d = to_device_bf16(head), to_device_bf16(hidden)
    draft_d, dtok_d = to_device(draft), to_device(dtok)
    ua, uf = to_device(u["u_accept"]), to_device(u["u_final"])
    # stochastic: its stored logits first
    fs = FusedVerifier(B, k, V, d, STOCH)
    fs(T, head_d, hid_d, draft_d, dtok_d, ua, uf)
    g_s = fs.results()
    fs.check_canaries()
    assert bd.get_status(fs.ws) == 0
    G = _stored_logits(fs).reshape(B, k + 1, V).astype(np.float64)
    err = np.max(np.abs(G - t), axis=2)                          # per row
    # sum_i |E_vi h_i| per entry (|bf16| by clearing the sign bit; the head is
    # widened in row blocks)
    scale = linear(head & np.uint16(0x7FFF), np.abs(bf16_bits_to_f64(hidden)))
    # float32 accumulation of exact bf16 products: within 64 u sum|E h| per entry
    assert np.all(np.abs(G - t) <= 64 * 2.0 ** -24 * scale + 1e-30), "logits beyond the float32 bound"
    assert rel_l2(G, t) <= 1e-5
    del scale
    # stochastic decisions: the oracle's rule on the GPU's own logits
    o = oracle_verify(G, draft.astype(np.float64), dtok, STOCH, T, u["u_accept"], u["u_final"])
    exc = compare_verify(g_s, o, STOCH, G, draft.astype(np.float64), dtok, u["u_accept"], u["u_final"], T)
    check_excused(exc, B, "fused stochastic outputs")
    g_out, g_len, g_acc = g_s
    assert np.all((g_len >= 1) & (g_len <= k + 1)) and np.all(g_acc == g_len - 1)
    # greedy: against the oracle's float64 logits
    fg = FusedVerifier(B, k, V, d, GREEDY)
    fg(T, head_d, hid_d, None, dtok_d)
    gg = fg.results()
    fg.check_canaries()
    assert bd.get_status(fg.ws) == 0
    og = oracle_verify(t, None, dtok, GREEDY)
    n_exc = 0
    for b in np.nonzero((gg[0] != og[0]).any(axis=1) | (gg[1] != og[1]))[0]:
        # the first row where the two disagree decides; its top-2 gap must be
        # within twice the measured logit error
        j = int(min(gg[1][b], og[1][b])) - 1
        z = np.sort(t[b, j])
        gap = float(z[-1] - z[-2])
        assert gap < 2 * err[b, j], "seq %d: greedy differs, top-2 gap %.3g, logit error %.3g" % (b, gap, err[b, j])
        record_excused("fused_argmax", b, j, gap, 2 * err[b, j])
        n_exc += 1
    check_excused(n_exc, B, "fused greedy outputs")
    # the greedy emitted tokens are the argmax of the GPU's own logits (lowest index on ties)
    for b in range(B):
        L = int(gg[1][b])
        assert gg[0][b][L - 1] == int(np.argmax(G[b, L - 1])), "seq %d: emitted token is not the argmax" % b
    return g_s, gg


@pytest.mark.parametrize("B,k,V,d,T", [(1, 3, 9000, 128, 1.0),       # one sequence: two residual chunks
                                       (3, 3, 5003, 256, 1.0),       # one 128-row tile, ragged vocabulary
                                       (37, 2, 20011, 512, 0.7),     # 111 rows
                                       (50, 3, 4099, 320, 1.3),      # two row tiles, the second partial
                                       (100, 3, 3001, 192, 1.0),     # two row groups: the head streams twice
                                       (6, 3, 9000, 128, 0.05),      # near one-hot rows
                                       (6, 3, 9000, 128, 20.0)])     # near-uniform rows, small residual
def test_fused_ragged_shapes(B, k, V, d, T):
    run_fused_parity(B, k, V, d, T, seed=9000 + B)


def test_fused_batched_shape_full_size():
    """The batched workload's verification: 64 sequences, k = 3 (256 rows), d =
    4096, the full 151936-token head."""
    w = W.BATCHED_STOCHASTIC
    (out, L, _), _ = run_fused_parity(w.B, w.k, w.V, w.d, w.T, seed=9100, noise=0.3)
    print("fused batched shape: mean accepted length %.3f" % L.mean())


def test_fused_everything_accepted_and_bad_tokens():
    B, k, V, d, T = 4, 2, 1031, 128, 1.0
    head, hidden, t, draft, dtok, u = _inputs(B, k, V, d, T, seed=9200)
    head_d, hid_d = to_device_bf16(head), to_device_bf16(hidden)
    # draft = the target's own argmax (greedy all accepted)
    d_arg = np.argmax(t[:, :k], axis=2).astype(np.int32)
    fg = FusedVerifier(B, k, V, d, GREEDY)
    fg(T, head_d, hid_d, None, to_device(d_arg))
    out, L, acc = fg.results()
    og = oracle_verify(t, None, d_arg, GREEDY)
    assert np.array_equal(out, og[0]) and np.array_equal(L, og[1])
    assert np.all(L == k + 1)
    # an out-of-range draft token is never accepted and flags the status
    bad = d_arg.copy()
    bad[1, 0] = V
    bad[2, 1] = -1
    fb = FusedVerifier(B, k, V, d, GREEDY)
    fb(T, head_d, hid_d, None, to_device(bad))
    out, L, _ = fb.results()
    assert L[1] == 1 and L[2] == 2
    assert bd.get_status(fb.ws) & bd.STATUS_BAD_TOKEN


def test_fused_invalid_arguments():
    B, k, V, d = 2, 3, 1000, 64
    fv = FusedVerifier(B, k, V, d, GREEDY)
    h = torch.zeros(V * d, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros(B * (k + 1) * d, dtype=torch.bfloat16, device="cuda")
    dt = torch.zeros(B * k, dtype=torch.int32, device="cuda")
    with pytest.raises(bd.MtpError):      # T = 0 in stochastic mode
        bd.spec_verify_fused(B, k, V, d, 0.0, STOCH, h, x, None, dt, None, None, fv.out_tok, fv.accept_len,
                             fv.num_accepted, fv.ws)
    assert bd.fused_workspace_size(B, 0, V, d, GREEDY) == 0      # k outside 1..8
    assert bd.fused_workspace_size(B, k, V, 60, GREEDY) == 0     # d not a multiple of 8
    small = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(bd.MtpError):      # workspace too small
        bd.spec_verify_fused(B, k, V, d, 1.0, GREEDY, h, x, None, dt, None, None, fv.out_tok, fv.accept_len,
                             fv.num_accepted, small)


def test_fused_stochastic_out_of_range_tokens():
    """Stochastic: a draft token outside [0, V) is never accepted; its position
    is rejected and replaced by that position's residual draw, as after any
    rejection.  The oracle defines no such token, so the expected outputs are
    the oracle's on the call's own stored logits with, at that position, a
    valid token where q(d) >= p(d) and u_accept = 1 (which rejects)."""
    from oracle.sampling import softmax_T
    B, k, V, d, T = 4, 3, 5003, 256, 1.0
    head, hidden, t, draft, dtok, u = _inputs(B, k, V, d, T, seed=9300)
    dtok = dtok.copy()
    bad = {(0, 1): V + 7, (2, 0): -1}
    for (b, j), v in bad.items():
        dtok[b, j] = v
    ua = u["u_accept"].copy()
    ua[0, 0] = 0.0  # sequence 0 accepts position 0 (0 < p(d) / q(d))
    fs = FusedVerifier(B, k, V, d, STOCH)
    fs(T, to_device_bf16(head), to_device_bf16(hidden), to_device(draft), to_device(dtok), to_device(ua),
       to_device(u["u_final"]))
    g = fs.results()
    fs.check_canaries()
    assert bd.get_status(fs.ws) & bd.STATUS_BAD_TOKEN
    G = _stored_logits(fs).reshape(B, k + 1, V).astype(np.float64)
    l64 = draft.astype(np.float64)
    d2, ua2 = dtok.copy(), ua.copy()
    for (b, j) in bad:
        d2[b, j] = int(np.argmax(softmax_T(l64[b, j], T) - softmax_T(G[b, j], T)))
        ua2[b, j] = 1.0
    o = oracle_verify(G, l64, d2, STOCH, T, ua2, u["u_final"])
    exc = compare_verify(g, o, STOCH, G, l64, d2, ua2, u["u_final"], T)
    check_excused(exc, B, "fused stochastic outputs with out-of-range tokens")
    assert g[1][0] == 2 and g[1][2] == 1
