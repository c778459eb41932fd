"""GPU parity of the GEMV path's ops run in cooperative chain launches
(MTP_CHAIN=1: several ops per launch with grid barriers, the draft token
selected inside the barrier after the LM head) against the oracle: the same
checks as the one-launch-per-op path."""

import pytest

from mtp_speculative_decoding_draft_gb300 import workloads as W
from test_gpu_draft import GQA5, MID, GREEDY, STOCH, run_draft_parity

pytestmark = pytest.mark.gpu


@pytest.fixture
def chain(monkeypatch):
    monkeypatch.setenv("MTP_CHAIN", "1")   # the library reads it at every call


@pytest.mark.parametrize("mode", [GREEDY, STOCH])
@pytest.mark.parametrize("w,ctx_fix", [(W.TINY, None), (MID, [1, 64, 200]), (GQA5, None)],
                         ids=["tiny", "mid_b3", "gqa5_b2"])
def test_chain_draft(chain, w, ctx_fix, mode):
    run_draft_parity(w, mode, w.T if w is not W.TINY else 1.0, ctx_fix=ctx_fix)


def test_chain_single_greedy_full_size(chain):
    run_draft_parity(W.SINGLE_GREEDY, GREEDY, 1.0)
