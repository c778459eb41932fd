"""mtp_draft_noalloc (the draft chain on the library's static scratch) against
mtp_draft with a caller workspace: same inputs, bit-identical outputs, on two
calls in a row.  The same kernels run in the same order on both paths, and the
library's results are a deterministic function of the inputs, so nothing may
differ by even one bit.  Collected last so that it also runs after every other
GPU test in one process; it passes on its own in a fresh process too."""

import numpy as np
import pytest
import torch

from mtp_speculative_decoding_draft_gb300 import binding as bd
from mtp_speculative_decoding_draft_gb300 import workloads as W
from mtp_speculative_decoding_draft_gb300.model import DraftModule, to_device

pytestmark = pytest.mark.gpu

GREEDY, STOCH = 0, 1

# several GEMV tiles, a ragged vocabulary and ragged contexts
CASE = W.Workload("noalloc_b3_d256_v5003", B=3, k=3, V=5003, d=256, Hq=4, Hkv=2, Dh=64, F=768,
                  ctx=(1, 200), T=0.8, seed=2101)
# a vocabulary whose stochastic logits (B k V floats, 5.4 MB) would not fit the
# 4 MiB array: mtp_draft_noalloc keeps no logits in its scratch, so it runs
WIDE_V = W.Workload("noalloc_b3_d256_v150001", B=3, k=3, V=150001, d=256, Hq=4, Hkv=2, Dh=64, F=768,
                    ctx=(1, 120), T=1.0, seed=2102)


def _fresh(w, wts, ctx):
    m = DraftModule(w, wts)
    m.set_context(ctx)
    return m


@pytest.mark.parametrize("mode", [GREEDY, STOCH])
@pytest.mark.parametrize("w", [W.TINY, CASE, WIDE_V], ids=lambda w: w.name)
def test_noalloc_matches_workspace_call(w, mode):
    wts = W.make_weights(w)
    ctx = W.make_context(w)
    u = to_device(W.make_uniforms(w)["u_draft"]) if mode == STOCH else None
    T = w.T
    B, k, V = w.B, w.k, w.V

    ref = _fresh(w, wts, ctx)
    ref.draft(T, mode, u, logits=True)
    torch.cuda.synchronize()
    assert ref.status() == 0
    r_tok = ref.draft_tok.cpu().numpy()
    r_log = ref.draft_logits.cpu().numpy()
    r_kc = ref.k_cache.view(torch.int16).cpu().numpy()

    for call in range(2):           # two calls in a row on the same scratch
        m = _fresh(w, wts, ctx)
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        bd.mtp_draft_noalloc(m.dims, m.wptr, m.h, m.last_tok, m.k_cache, m.v_cache, m.ctx_len, k, T,
                             mode, u, m.draft_tok, m.draft_logits, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, "call %d: status %d" % (call, int(status.item()))
        g_tok = m.draft_tok.cpu().numpy()
        g_log = m.draft_logits.cpu().numpy()
        assert np.array_equal(g_tok, r_tok), "call %d: draft tokens differ" % call
        assert np.array_equal(g_log.view(np.uint32), r_log.view(np.uint32)), "call %d: logits differ" % call
        assert np.array_equal(m.k_cache.view(torch.int16).cpu().numpy(), r_kc)
        m.check_canaries()
        assert g_log.reshape(B, k, V).shape == (B, k, V)


def test_noalloc_rejects_oversized_problem():
    """A problem whose scratch exceeds the static array is refused before any launch."""
    w = W.SINGLE_GREEDY
    dims = bd.make_dims(256, w.d, w.Hq, w.Hkv, w.Dh, w.F, w.V, 64, w.eps)
    assert bd.workspace_size(dims, 3) > (4 << 20)
    t = {n: torch.zeros(16, dtype=torch.bfloat16, device="cuda") for n in bd.WEIGHT_FIELDS}
    wptr = bd.make_weights(t)
    i32 = torch.zeros(256 * 4, dtype=torch.int32, device="cuda")
    bf = torch.zeros(256 * w.d, dtype=torch.bfloat16, device="cuda")
    before = bd.launch_count()
    with pytest.raises(bd.MtpError) as ei:
        bd.mtp_draft_noalloc(dims, wptr, bf, i32, bf, bf, i32, 3, 1.0, GREEDY, None, i32, None)
    assert ei.value.code == -5
    assert bd.launch_count() == before
