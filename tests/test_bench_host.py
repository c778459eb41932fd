"""Host-side logic of bench.py: the algorithmic step bytes its roofline fraction
divides by, for the plain chain and the next rows' options, and the traffic
table's source check."""

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from mtp_speculative_decoding_draft_gb300 import workloads as W  # noqa: E402


def test_single_sequence_step_bytes():
    w = W.SINGLE_GREEDY
    ctx = np.array([4096])
    block = (w.d * 2 * w.d + (w.Hq + 2 * w.Hkv) * w.Dh * w.d + w.d * w.Hq * w.Dh + 3 * w.d * w.F + 5 * w.d)
    weights = 3 * (block + w.V * w.d) * 2
    kv = sum(4096 + j + 1 for j in range(3)) * w.Hkv * w.Dh * 2 * 2
    target = 1 * 4 * w.V * 4
    assert bench.step_bytes(w, ctx, False) == weights + kv + target
    assert abs(bench.step_bytes(w, ctx, False) / 1e9 - 5.146) < 1e-3


def test_options_change_the_counted_bytes():
    w = W.SINGLE_GREEDY
    ctx = np.array([4096])
    full = bench.step_bytes(w, ctx, False)
    per_row = w.Hkv * w.Dh * 2 * 2
    # one module per depth: every depth sees its own context plus one row
    assert full - bench.step_bytes(w, ctx, False, n_modules=3) == (1 + 2) * per_row
    # a chain stopped after depth 0 streams one depth of weights and K/V
    one = bench.step_bytes(w, ctx, False, depths=1)
    assert full - one == 2 * (bench.block_elements(w) + w.V * w.d) * 2 + (4098 + 4099) * per_row
    # a reduced head of 32768 rows
    red = bench.step_bytes(w, ctx, False, head_rows=32768)
    assert full - red == 3 * (w.V - 32768) * w.d * 2
    assert bench.lmhead_bytes(w, False, 32768) == 32768 * w.d * 2


def test_stochastic_counts_the_draft_logits():
    w4 = W.replace(W.BATCHED_STOCHASTIC, B=4)
    w = w4
    ctx = np.array([1024, 2000, 5000, 8192])
    assert bench.step_bytes(w4, ctx, True) - bench.step_bytes(w4, ctx, False) == 2 * 4 * w.k * w.V * 4


def test_traffic_is_reported_only_for_unchanged_sources(tmp_path, monkeypatch):
    key = ("lm_head_gemv", "single_greedy_b1_d4096_v151936_ctx4096")
    rec = bench.NCU_TRAFFIC[key]
    # a recorded digest that no longer matches the source: no figure
    monkeypatch.setitem(bench.NCU_TRAFFIC, key, {"bytes": rec["bytes"],
                                                 "sources": {"csrc/draft.cu": "0" * 64}})
    assert bench.ncu_traffic(*key) is None
    assert bench.ncu_traffic("no_such_kernel", "no_such_workload") is None


def test_default_line_traffic_matches_the_committed_sources():
    """The default line's dominant kernel (the LM-head GEMV of the single
    sequence) has a DRAM-traffic capture taken from the sources as committed:
    a change to them that alters the kernel needs a new capture (and its
    digests) before the line can report traffic again."""
    key = ("lm_head_gemv", "single_greedy_b1_d4096_v151936_ctx4096")
    t = bench.ncu_traffic(*key)
    assert t is not None, "sources changed since the LM-head capture: take it again"
    # within a few MB of the algorithmic bytes (the head once, 1.245 GB)
    assert abs(t - 151936 * 4096 * 2) < 8e6


def test_batched_and_deep_chain_step_bytes_match_the_worked_totals():
    """The hot-path scope's worked totals per step: about 9.1 GB for the batch of
    64 (weights 5.09 GB, K/V about 3.62 GB at the mean context of 4608, logits
    0.39 GB) and about 28.2 GB for the deep chain (weights 16.93 GB, K/V 10.74 GB,
    logits 0.52 GB)."""
    b64 = W.BATCHED_STOCHASTIC
    assert abs(bench.step_bytes(b64, np.full(b64.B, 4608), True) / 1e9 - 9.1) < 0.05
    deep = W.WORKLOADS["deep_chain_b32_k5_d5120_v256000_ctx16384"]
    assert abs(bench.step_bytes(deep, np.full(deep.B, 16384), True) / 1e9 - 28.2) < 0.05


def test_oracle_timing_stops_at_its_budget():
    """The reference arm's oracle loop ends after its wall-clock budget, with at
    least one timed sample, however many steps were asked for."""
    import time
    t0 = time.perf_counter()
    out = bench._oracle_samples("tiny_b1_d64_v1000", 1, 10 ** 7, budget_s=0.3)
    assert 1 <= len(out) < 10 ** 7
    assert time.perf_counter() - t0 < 30.0
    assert all(a > 0 and b > 0 for a, b in out)
    one = bench._oracle_samples("tiny_b1_d64_v1000", 1, 10 ** 7, budget_s=0.0)
    assert len(one) == 1


def test_options_parse_and_name_the_workload():
    """Every option is accepted, and each run's config names what it ran."""
    import argparse
    import subprocess
    import sys as _sys
    r = subprocess.run([_sys.executable, os.path.join(ROOT, "bench.py"), "--help"], capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0
    for opt in ("--graph", "--correlated", "--modules", "--stop-p", "--draft-vocab", "--impl", "--greedy"):
        assert opt in r.stdout
    base = dict(gpus=1, modules=1, stop_p=None, draft_vocab=0, correlated=0.0, graph=False, k=0, greedy=False)
    cfg = bench.config_of(W.SINGLE_GREEDY, argparse.Namespace(**dict(base, correlated=0.1, graph=True)))
    assert cfg["workload"] == W.SINGLE_GREEDY.name + "_correlated0.1" and cfg["launch"] == "cuda graph replay"
    cfg = bench.config_of(W.SINGLE_GREEDY, argparse.Namespace(**dict(base, modules=3)))
    assert cfg["workload"].endswith("_modules3") and cfg["launch"] == "direct calls"
    w = bench._verify_workload(argparse.Namespace(workload=W.VERIFY_SWEEP.name, k=5, greedy=True))
    assert w.k == 5 and w.mode == W.GREEDY
    cfg = bench.config_of(w, argparse.Namespace(**base))
    assert "logits read per call" in cfg["l2"]
