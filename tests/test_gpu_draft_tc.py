"""GPU parity of the tensor-core draft path (batches of five sequences and
more) against the oracle: the tcgen05 GEMMs, the split-K epilogues, the
per-sequence draft-token selection and the K/V append."""

import pytest

from mtp_speculative_decoding_draft_gb300 import workloads as W
from test_gpu_draft import GREEDY, STOCH, run_draft_parity

pytestmark = pytest.mark.gpu

# One batch group of 32 MMA columns (20 used), K-split GEMMs, a vocabulary
# whose last 128-row tile is partial, contexts from 1 to 200.
TC20 = W.Workload("tc_b20_d256_v5003", B=20, k=3, V=5003, d=256, Hq=4, Hkv=2, Dh=64, F=768,
                  ctx=(1, 200), T=0.8, seed=2003)
# Two batch groups of 128 columns, the second partial; GQA group of five.
TC150 = W.Workload("tc_b150_d640_v3001", B=150, k=2, V=3001, d=640, Hq=10, Hkv=2, Dh=128, F=1280,
                   ctx=(60, 300), T=1.0, seed=2004)


@pytest.mark.parametrize("mode", [GREEDY, STOCH])
def test_tc_batch_of_20(mode):
    r = run_draft_parity(TC20, mode, TC20.T)
    print("tc20 mode=%d max rel L2 %.3g excused %d" % (mode, max(r["rel_l2"]), r["excused"]))


@pytest.mark.parametrize("mode", [GREEDY, STOCH])
def test_tc_two_batch_groups(mode):
    r = run_draft_parity(TC150, mode, TC150.T, seqs=[0, 63, 127, 128, 149])
    print("tc150 mode=%d max rel L2 %.3g excused %d" % (mode, max(r["rel_l2"]), r["excused"]))


# Batch of 40: MMA columns padded to 64, the three activation terms side by side
# in one MMA of N = 192.
TC40 = W.Workload("tc_b40_d384_v4099", B=40, k=3, V=4099, d=384, Hq=6, Hkv=2, Dh=64, F=1152,
                  ctx=(1, 150), T=0.9, seed=2005)


@pytest.mark.parametrize("mode", [GREEDY, STOCH])
def test_tc_batch_of_40(mode):
    r = run_draft_parity(TC40, mode, TC40.T, seqs=[0, 17, 31, 32, 39])
    print("tc40 mode=%d max rel L2 %.3g excused %d" % (mode, max(r["rel_l2"]), r["excused"]))


@pytest.mark.parametrize("T", [0.05, 20.0])
def test_tc_stochastic_temperature_extremes(T):
    """The tensor-core path's sampler at a near one-hot and a near-uniform
    temperature."""
    r = run_draft_parity(TC20, STOCH, T)
    print("tc20 T=%g max rel L2 %.3g excused %d" % (T, max(r["rel_l2"]), r["excused"]))
