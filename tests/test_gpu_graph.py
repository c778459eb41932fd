"""spec_step and mtp_draft captured in a CUDA graph and replayed.

The calls make no allocation and no host synchronisation, and every launch
takes its arguments by value, so a captured step can be replayed: each replay
must give exactly what a direct call on the same inputs gives (bit for bit),
and reads the inputs' current contents."""

import numpy as np
import pytest
import torch

from mtp_speculative_decoding_draft_gb300 import workloads as W
from mtp_speculative_decoding_draft_gb300.model import DraftModule, to_device, to_device_bf16

pytestmark = pytest.mark.gpu

GREEDY, STOCH = 0, 1

MID = W.Workload("graph_b3_d256_v5003", B=3, k=3, V=5003, d=256, Hq=4, Hkv=2, Dh=64, F=768,
                 ctx=(1, 200), T=0.8, seed=2501)
TC20 = W.Workload("graph_tc_b20_d256_v5003", B=20, k=3, V=5003, d=256, Hq=4, Hkv=2, Dh=64, F=768,
                  ctx=(1, 300), T=0.9, seed=2502)


def _restore(m, ctx):
    """The step's inputs and caches back to ctx, in place: a captured graph
    keeps the buffers it was captured with."""
    m.h.copy_(to_device_bf16(ctx["h"]))
    m.last_tok.copy_(to_device(ctx["last_tok"].astype(np.int32)))
    m.ctx_len.copy_(to_device(ctx["ctx_len"].astype(np.int32)))
    m.k_cache.copy_(to_device_bf16(ctx["k_cache"]))
    m.v_cache.copy_(to_device_bf16(ctx["v_cache"]))


def _outputs(m):
    return [t.clone() for t in (m.draft_tok, m.draft_logits, m.out_tok, m.accept_len, m.num_accepted,
                                m.k_cache, m.v_cache)]


def _same(a, b):
    return all(torch.equal(x.view(torch.int32) if x.dtype == torch.float32 else x,
                           y.view(torch.int32) if y.dtype == torch.float32 else y) for x, y in zip(a, b))


@pytest.mark.parametrize("w,mode", [(MID, STOCH), (MID, GREEDY), (TC20, STOCH), (TC20, GREEDY)],
                         ids=["gemv-stochastic", "gemv-greedy", "tensor_core-stochastic", "tensor_core-greedy"])
def test_spec_step_graph_replay(w, mode):
    wts = W.make_weights(w)
    ctx = W.make_context(w)
    u = W.make_uniforms(w)
    rng = np.random.default_rng(w.seed)
    targets = [(rng.standard_normal((w.B, w.k + 1, w.V)) * 2.0).astype(np.float32) for _ in range(2)]
    m = DraftModule(w, wts)
    m.set_context(ctx)
    st = mode == STOCH
    ud, ua, uf = ((to_device(u["u_draft"]), to_device(u["u_accept"]), to_device(u["u_final"])) if st
                  else (None, None, None))
    tgt = to_device(targets[0])

    def step():
        m.step(w.T, mode, tgt, ud, ua, uf, logits=True)

    # direct calls on each target
    direct = []
    for t in targets:
        _restore(m, ctx)
        tgt.copy_(to_device(t))
        step()
        torch.cuda.synchronize()
        assert m.status() == 0
        direct.append(_outputs(m))

    # capture (after a warm-up call on a side stream), then replay
    _restore(m, ctx)
    tgt.copy_(to_device(targets[0]))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for rep in range(3):
        i = rep % 2
        _restore(m, ctx)
        tgt.copy_(to_device(targets[i]))
        g.replay()
        torch.cuda.synchronize()
        assert m.status() == 0
        assert _same(_outputs(m), direct[i]), "replay %d differs from the direct call" % rep
