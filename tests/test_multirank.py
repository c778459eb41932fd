"""The multi-rank logic of bench.py on CPU: two gloo ranks.

Each rank is an independent replica (the draft chain and its verification
exchange nothing between sequences), so the only cross-rank steps are the
barriers around the timed region and the maximum of the per-rank times.  These
tests run that reduction, and the reference arm under the launcher the bench
is run with, as two processes on 127.0.0.1."""

import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # per-rank step times 1.5 ms and 4.0 ms: the job's time is the slower one
        ms = bench.max_over_ranks([1.5, 4.0][rank], device="cpu")
        dist.barrier()
        with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as f:
            json.dump({"ms": ms, "rate": bench.job_rate(ms, world)}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    for r in range(world):
        got = json.load(open(tmp_path / ("rank%d.json" % r)))
        assert got["ms"] == 4.0
        # two replicas, each 250 steps/s at the slower rank's time
        assert abs(got["rate"] - 500.0) < 1e-9


def test_single_process_reduction_is_the_identity():
    assert bench.max_over_ranks(3.25, device="cpu") == 3.25
    assert bench.job_rate(2.0, 1) == 500.0


def test_reference_arm_under_the_launcher_prints_one_line():
    """The launch the bench is run with at N = 2: rank 0 alone times the
    oracle and prints; rank 1 exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--workload", "tiny_b1_d64_v1000", "--steps", "2",
           "--warmup", "1"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["cpu_baseline"]["host_cores"] >= 1 and line["cpu_baseline"]["cpu"]
