#!/usr/bin/env python3
"""Benchmark of the MTP draft + verify step (spec_step) on GB300.

Default workload: one sequence, greedy, k = 3 drafts, hidden 4096, 32/8 heads of
128, SwiGLU 12288, vocabulary 151936, 4096 context tokens (all synthetic and
seeded; random bf16 weights of that shape).  One "step" is one spec_step call:
k chained draft-module applications followed by verification.

Prints one JSON line (rank 0).  With --impl reference it times the CPU oracle on
the host cores instead.  Under torchrun every rank runs an independent replica
of the workload (the path has no cross-sequence exchange); the reported time is
the maximum over ranks.
"""

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mtp_speculative_decoding_draft_gb300 import workloads as W  # noqa: E402
from mtp_speculative_decoding_draft_gb300.metrics import acceptance_metrics  # noqa: E402

METRIC = "spec-decode steps/s & accepted tok/s (MTP draft+verify); % of HBM roofline"


def block_elements(w):
    return (w.d * 2 * w.d + (w.Hq + 2 * w.Hkv) * w.Dh * w.d + w.d * w.Hq * w.Dh + 3 * w.d * w.F + 5 * w.d)


def step_bytes(w, ctx_len, logits_out, n_modules=1, depths=None, head_rows=None):
    """Algorithmic HBM bytes of one spec_step: weights re-streamed at every
    depth, the visible KV rows read once per depth, target logits read once,
    draft logits written and read once when they are materialised.  With
    distinct modules depth j runs module min(j, n - 1) and sees that module's
    context plus the rows earlier depths appended to the same cache."""
    k = w.k
    kd = k if depths is None else depths  # depths whose weights are streamed (a stopped chain skips the rest)
    weights = kd * (block_elements(w) + (w.V if head_rows is None else head_rows) * w.d) * 2
    kv = sum(int(L) + j - min(j, n_modules - 1) + 1 for L in ctx_len for j in range(kd)) * w.Hkv * w.Dh * 2 * 2
    target = w.B * (k + 1) * w.V * 4
    draft = 2 * w.B * k * w.V * 4 if logits_out else 0
    return weights + kv + target + draft


def lmhead_bytes(w, logits_out, head_rows=None):
    return (w.V if head_rows is None else head_rows) * w.d * 2 + (w.B * w.V * 4 if logits_out else 0)


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of a
# kernel from one ncu capture, with the SHA-256 of the sources the kernel is
# built from at capture time.  A figure is reported only while those sources
# are unchanged; the summaries of the captures are kept under profiles/.
NCU_TRAFFIC = {
    ("lm_head_gemv", "single_greedy_b1_d4096_v151936_ctx4096"): {
        "bytes": 1244775424 + 2836992,
        "sources": {
            "csrc/draft.cu": "676f8d49f732a1dd64718ab494595f3138735d323cd0ad43c44d9c3c89978e7d",
            "csrc/draft_ops.cuh": "ad62698d95aa35a07e07854a0daa62b73bffc314f886982abd3a02a0da033f38",
            "csrc/common.cuh": "ccc7be3ffbab76f32e48e064231311046ac5ebb3caee7e3f3df14b4629b22b95",
            "csrc/internal.h": "2ab350d5622c22f47de0c469aabd5010981632626e75291fc2273994f1968187",
        },
    },
    ("verify_kernel", "verify_sweep_b256_v151936_k3/greedy"): {
        "bytes": 622470656 + 2755328,
        "sources": {
            "csrc/verify.cu": "f5fc0310bc0803d8610b522263a676741829b2d28da6924a064b3d3158681d56",
            "csrc/common.cuh": "ccc7be3ffbab76f32e48e064231311046ac5ebb3caee7e3f3df14b4629b22b95",
            "csrc/internal.h": "2ab350d5622c22f47de0c469aabd5010981632626e75291fc2273994f1968187",
        },
    },
    ("verify_split_kernel", "verify_sweep_b256_v151936_k3/stochastic"): {
        "bytes": 1165680640 + 2998272,
        "sources": {
            "csrc/verify_split.cu": "80abf6cfe5259b2b43e8243c5342d705d37e519c4cb025db89ecaea85f0ffeae",
            "csrc/verify_rule.cuh": "ea886aaf8280a01a05f400afc2d1e3873420801473ab364cfacf465340a0eb5b",
            "csrc/verify.cu": "f5fc0310bc0803d8610b522263a676741829b2d28da6924a064b3d3158681d56",
            "csrc/common.cuh": "ccc7be3ffbab76f32e48e064231311046ac5ebb3caee7e3f3df14b4629b22b95",
            "csrc/internal.h": "2ab350d5622c22f47de0c469aabd5010981632626e75291fc2273994f1968187",
        },
    },
    ("fv_gemm_kernel + fv_finish_kernel", "fused_verify_b64_k3_d4096_v151936/greedy"): {
        "bytes": 1250486528 + 4050432 + 2442240,
        "sources": {
            "csrc/fused.cu": "05994466aa93f37ec2e519d2518c65c2240abdaf995b6fcec71b6339d6629c3a",
            "csrc/verify_rule.cuh": "ea886aaf8280a01a05f400afc2d1e3873420801473ab364cfacf465340a0eb5b",
            "csrc/tcgen05.cuh": "e128ff6d7c8451d618848063024b7cd0a98c722dd1b86ef0d04e6a07a9070ee7",
            "csrc/common.cuh": "ccc7be3ffbab76f32e48e064231311046ac5ebb3caee7e3f3df14b4629b22b95",
            "csrc/internal.h": "2ab350d5622c22f47de0c469aabd5010981632626e75291fc2273994f1968187",
        },
    },
}


def ncu_traffic(kernel, workload):
    import hashlib
    rec = NCU_TRAFFIC.get((kernel, workload))
    if rec is None:
        return None
    pkg = os.path.join(ROOT, "mtp_speculative_decoding_draft_gb300")
    for rel, digest in rec["sources"].items():
        with open(os.path.join(pkg, rel), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != digest:
                return None
    return rec["bytes"]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix="clocks_gpu%d_" % self.index, suffix=".csv")
            self.f = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
            if self.path:
                self.f.close()
                os.remove(self.path)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            lines = fh.readlines()
        os.remove(self.path)
        for line in lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- CPU oracle timing

def _oracle_samples(workload_name, depths, n, budget_s=None):
    """Generate the workload once, then time the oracle up to n times (fewer
    once budget_s seconds have passed since the first, at least once) on `depths`
    draft depths plus the verification of one step; returns a list of
    (seconds for the depths, seconds for the verification)."""
    from oracle.block import Dims, mtp_draft
    from oracle.verify import spec_verify
    w = W.WORKLOADS[workload_name]
    wts = W.make_weights(w)
    ctx = W.make_context(w)
    u = W.make_uniforms(w)
    tl = W.target_logits(w)
    dims = Dims(w.B, w.d, w.Hq, w.Hkv, w.Dh, w.F, w.V, w.Lmax, w.eps)
    out = []
    start = time.perf_counter()
    for _ in range(n):
        t0 = time.perf_counter()
        dr = mtp_draft(wts, dims, ctx["h"], ctx["last_tok"], ctx["k_cache"], ctx["v_cache"], ctx["ctx_len"],
                       depths, w.T, w.mode, u["u_draft"])
        t1 = time.perf_counter()
        dt = np.zeros((w.B, w.k), np.int64)
        dt[:, :depths] = dr["draft_tok"]
        dl = np.zeros((w.B, w.k, w.V))
        dl[:, :depths] = dr["draft_logits"]
        spec_verify(tl, dl, dt, w.mode, w.T, u["u_accept"], u["u_final"])
        t2 = time.perf_counter()
        out.append((t1 - t0, t2 - t1))
        if budget_s is not None and t2 - start > budget_s:
            break
    return out


def _verify_workload(args):
    """The verify sweep's workload with the --k and --greedy options applied."""
    w = W.WORKLOADS[args.workload]
    if args.k:
        w = W.with_k(w, args.k)
    if args.greedy:
        w = W.replace(w, mode=W.GREEDY)
    return w


def _oracle_verify_samples(workload_name, k, greedy, n, n_seq, budget_s=None):
    """Time the oracle's verification of the verify sweep up to n times (fewer
    once budget_s seconds have passed since the first, at least once) on its
    first n_seq sequences; returns seconds per call scaled to all B sequences."""
    from oracle.block import STOCHASTIC, select_token
    from oracle.verify import spec_verify
    import argparse as _ap
    w = _verify_workload(_ap.Namespace(workload=workload_name, k=k, greedy=greedy))
    inp = W.verify_inputs(w)
    s = slice(0, min(n_seq, w.B))
    # drafts drawn from q at u_draft, as the GPU arm draws them
    d = np.zeros((w.B, w.k), np.int32)
    for b in range(s.start, s.stop):
        for j in range(w.k):
            d[b, j] = select_token(inp["draft_logits"][b, j], STOCHASTIC, w.T, float(inp["u_draft"][b, j]))
    out = []
    start = time.perf_counter()
    for _ in range(n):
        t0 = time.perf_counter()
        spec_verify(inp["target_logits"][s], inp["draft_logits"][s], d[s], w.mode, w.T, inp["u_accept"][s],
                    inp["u_final"][s])
        t1 = time.perf_counter()
        out.append((t1 - t0) * w.B / (s.stop - s.start))
        if budget_s is not None and t1 - start > budget_s:
            break
    return out


def _oracle_fused_samples(workload_name, greedy, n, n_seq, budget_s=None):
    """Time the oracle's verification from hidden states on the first n_seq
    sequences of the fused workload, up to n times (fewer once budget_s seconds
    have passed, at least once); seconds per call scaled to all B sequences."""
    from oracle.block import STOCHASTIC, select_token
    from oracle.verify import spec_verify_fused, target_logits_from_hidden
    w = W.WORKLOADS[workload_name]
    if greedy:
        w = W.replace(w, mode=W.GREEDY)
    inp = W.fused_inputs(w)
    s = list(range(min(n_seq, w.B)))
    # the sampled sequences' draft logits and tokens (inputs of the call, prepared untimed)
    draft = np.zeros((w.B, w.k, w.V))
    draft[s] = target_logits_from_hidden(inp["head"], inp["hidden"][s])[:, :w.k] + inp["noise"][s]
    d = np.zeros((w.B, w.k), np.int32)
    for b in s:
        for j in range(w.k):
            d[b, j] = select_token(draft[b, j], STOCHASTIC, w.T, float(inp["u_draft"][b, j]))
    out = []
    start = time.perf_counter()
    for _ in range(n):
        t0 = time.perf_counter()
        spec_verify_fused(inp["head"], inp["hidden"], draft, d, w.mode, w.T, inp["u_accept"], inp["u_final"],
                          seqs=s)
        t1 = time.perf_counter()
        out.append((t1 - t0) * w.B / len(s))
        if budget_s is not None and t1 - start > budget_s:
            break
    return out


def cpu_oracle_fused_times(args, n, n_seq=4, budget_s=None):
    code = ("import json,sys; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench._oracle_fused_samples(%r, %r, %d, %d, %r)))"
            % (ROOT, args.workload, bool(args.greedy), n, n_seq, budget_s))
    return _single_threaded(code)


def _single_threaded(code):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=3600)
    if r.returncode != 0:
        raise RuntimeError("oracle timing failed: " + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_oracle_verify_times(args, n, n_seq=16, budget_s=None):
    """Seconds per verify-sweep call of the oracle, in a fresh single-threaded
    process, on a sample of n_seq sequences scaled to the batch."""
    code = ("import json,sys; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench._oracle_verify_samples(%r, %d, %r, %d, %d, %r)))"
            % (ROOT, args.workload, args.k, bool(args.greedy), n, n_seq, budget_s))
    return _single_threaded(code)


def cpu_oracle_step_times(workload_name, depths, n, budget_s=None):
    """Step times of the oracle, measured in a fresh single-threaded process
    (BLAS pinned to one thread); each sample runs `depths` draft depths and
    the verification, and is scaled to the workload's k depths (a full step
    when depths = k)."""
    code = ("import json,sys; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench._oracle_samples(%r, %d, %d, %r)))" % (ROOT, workload_name, depths, n, budget_s))
    w = W.WORKLOADS[workload_name]
    return [td / depths * w.k + tv for td, tv in _single_threaded(code)]


def host_cpu():
    """The host's CPU as /proc/cpuinfo names it (model name, else the Arm
    implementer and part codes), with its logical core count."""
    import platform
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read().splitlines()
        names = [ln.split(":", 1)[1].strip() for ln in info if ln.lower().startswith("model name")]
        if names:
            model = names[0]
        else:
            impl = [ln.split(":", 1)[1].strip() for ln in info if ln.startswith("CPU implementer")]
            part = [ln.split(":", 1)[1].strip() for ln in info if ln.startswith("CPU part")]
            if impl and part:
                model = "%s implementer %s part %s" % (platform.machine(), impl[0], part[0])
    except OSError:
        pass
    return {"host_cores": os.cpu_count(), "cpu": model or platform.machine()}


def max_over_ranks(x, device="cuda"):
    """The largest x over the ranks of the process group (x itself without one):
    the slowest replica's time is the job's time."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(ms_per_step, world):
    """Whole-job steps per second: each of the world replicas ran its steps
    within ms_per_step (the maximum over ranks)."""
    return 1e3 / ms_per_step * world


# Wall-clock seconds the reference arm's timing loop runs at most, so that its
# run ends within a few minutes whatever --steps asks for.
REFERENCE_BUDGET_S = 90.0
# The GPU arm's CPU baseline: the median of this many full oracle steps, fewer
# if they take longer than the budget (at least one).
CPU_BASELINE_STEPS = 10
CPU_BASELINE_BUDGET_S = 45


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = W.WORKLOADS[args.workload]
    n_req = args.warmup + args.steps
    if w.fused:
        if args.greedy:
            w = W.replace(w, mode=W.GREEDY)
        n_seq = 4
        times = cpu_oracle_fused_times(args, n_req, n_seq, budget_s=REFERENCE_BUDGET_S)
        unit = "verify calls/s"
        sample = ("per call: the oracle forms the target logits from the hidden states and verifies %d of the "
                  "%d sequences in a single-threaded process; call time = that time x %d / %d"
                  % (n_seq, w.B, w.B, n_seq))
    elif w.verify_only:
        w = _verify_workload(args)
        n_seq = 16
        times = cpu_oracle_verify_times(args, n_req, n_seq, budget_s=REFERENCE_BUDGET_S)
        unit = "verify calls/s"
        sample = ("per call: the oracle verifies %d of the %d sequences in a single-threaded process; "
                  "call time = that time x %d / %d" % (min(n_seq, w.B), w.B, w.B, min(n_seq, w.B)))
    else:
        times = cpu_oracle_step_times(args.workload, w.k, n_req, budget_s=REFERENCE_BUDGET_S)
        unit = "steps/s"
        sample = ("per step: the oracle runs one full step of this workload (all %d draft depths and the "
                  "verification) in a single-threaded process" % w.k)
    # warm-up samples are dropped; with the time budget fewer than the requested
    # steps may have run (at least one is timed)
    skip = min(args.warmup, len(times) - 1)
    times = times[skip:]
    sample += ("; %d timed samples (%d requested, within about %d s)"
               % (len(times), args.steps, REFERENCE_BUDGET_S))
    t = float(np.mean(times))
    value = 1.0 / t
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, args),
            "cpu_baseline": dict({"value": value, "unit": unit, "cores": 1, "kind": "oracle", "sample": sample},
                                 **host_cpu()),
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_of(w, args):
    mods = getattr(args, "modules", 1)
    sp = getattr(args, "stop_p", None)
    dv = getattr(args, "draft_vocab", 0)
    name = (w.name + ("_modules%d" % mods if mods > 1 else "") + ("_stop%g" % sp if sp is not None else "")
            + ("_draftvocab%d" % dv if dv else "")
            + ("_correlated%g" % args.correlated if getattr(args, "correlated", 0) > 0 and w.mode == 0 else ""))
    return {"workload": name, "modules": mods, "stop_p": sp, "draft_vocab": dv or None, "B": w.B, "k": w.k, "d": w.d, "Hq": w.Hq, "Hkv": w.Hkv,
            "Dh": w.Dh, "F": w.F, "fused": bool(w.fused),
            "V": w.V, "ctx": w.ctx if not isinstance(w.ctx, tuple) else list(w.ctx),
            "mode": "greedy" if w.mode == 0 else "stochastic", "T": w.T,
            "launch": "cuda graph replay" if getattr(args, "graph", False) else "direct calls",
            "parallelism": "replicas%d" % args.gpus,
            "l2": ("inputs larger than L2 (the %.2f GB head streamed per call)" % (w.V * w.d * 2 / 1e9) if w.fused
                   else "inputs larger than L2 (%.2f GB of logits read per call)" % (verify_bytes(w) / 1e9) if w.verify_only
                   else "inputs larger than L2 (weights %.2f GB re-streamed per depth)"
                   % ((block_elements(w) + w.V * w.d) * 2 / 1e9))}


# ----------------------------------------------------------------------------- GPU arm

def drafts_from_q(draft_logits, u_draft, T):
    """Draft tokens drawn from q = softmax(draft / T) at u_draft by the inverse
    CDF (the smallest i whose running sum exceeds u times the total), on the
    device in float64: the verify sweep's drafts, sampled as a drafter samples
    them.  draft_logits [B, k, V] and u_draft [B, k] are CUDA tensors; returns
    int32 [B, k].  (Input preparation, outside the timed region.)"""
    import torch
    z = draft_logits.double() / T
    z = z - z.amax(dim=-1, keepdim=True)
    C = torch.cumsum(torch.exp(z), dim=-1)
    del z
    t = u_draft.double().unsqueeze(-1) * C[..., -1:]
    idx = torch.searchsorted(C, t, right=True).squeeze(-1)
    return idx.clamp_(max=draft_logits.shape[-1] - 1).to(torch.int32).contiguous()


def verify_kernel_name(w):
    """The kernel spec_verify runs: the cluster kernel for greedy mode (and
    for stochastic mode under MTP_VERIFY_SPLIT=0), else the ticketed one."""
    if w.mode == W.GREEDY or os.environ.get("MTP_VERIFY_SPLIT", "1").startswith("0"):
        return "verify_kernel"
    return "verify_split_kernel"


def verify_bytes(w):
    """Algorithmic bytes of one spec_verify: every logit row read once."""
    rows = w.B * (w.k + 1) + (w.B * w.k if w.mode == 1 else 0)
    return rows * w.V * 4


def fused_bytes(w):
    """Algorithmic bytes of one spec_verify_fused call that it certainly moves:
    the head and the hidden states read once; stochastic also writes the
    target's fp32 logits (its draw reads back only the rows it reaches, not
    counted)."""
    Na = w.B * (w.k + 1)
    return w.V * w.d * 2 + Na * w.d * 2 + (Na * w.V * 4 if w.mode == 1 else 0)


def fused_flops(w):
    return 2.0 * w.B * (w.k + 1) * w.V * w.d


def measured_tflops():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p))["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def _fused_setup(w):
    """Device inputs of the fused workload: head, hidden, the draft's logits
    (the target's own head . hidden plus the seeded noise, formed here with a
    plain float32 matmul as input preparation) and drafts drawn from q."""
    import torch
    from mtp_speculative_decoding_draft_gb300.model import FusedVerifier, to_device, to_device_bf16
    inp = W.fused_inputs(w)
    head_d, hid_d = to_device_bf16(inp["head"]), to_device_bf16(inp["hidden"])
    tl = torch.matmul(hid_d.view(-1, w.d).float(), head_d.view(w.V, w.d).float().T).view(w.B, w.k + 1, w.V)
    draft = (tl[:, :w.k] + to_device(inp["noise"])).contiguous()
    del tl
    torch.cuda.empty_cache()
    dtok = drafts_from_q(draft, to_device(inp["u_draft"]), w.T)
    ua, uf = to_device(inp["u_accept"]), to_device(inp["u_final"])
    fv = FusedVerifier(w.B, w.k, w.V, w.d, w.mode)
    return inp, head_d, hid_d, draft, dtok, ua, uf, fv


def time_fused(w, steps, warmup, peak):
    """spec_verify_fused on the fused workload, CUDA-event timed with its own
    clock samples."""
    import torch
    from mtp_speculative_decoding_draft_gb300 import binding as bd
    inp, head_d, hid_d, draft, dtok, ua, uf, fv = _fused_setup(w)
    stoch = w.mode == 1

    def call():
        fv(w.T, head_d, hid_d, draft if stoch else None, dtok, ua if stoch else None, uf if stoch else None)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        call()
    e1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / steps
    assert bd.get_status(fv.ws) == 0
    _, L, _ = fv.results()
    tf, tf_kind = measured_tflops()
    fb = fused_bytes(w)
    out = {"workload": "%s/%s" % (w.name, "stochastic" if stoch else "greedy"), "ms_per_call": ms,
           "calls_s": 1e3 / ms, "steps": steps, "warmup": warmup, "bytes_per_call": fb,
           "achieved_gbs": fb / (ms * 1e-3) / 1e9, "frac": fb / (ms * 1e-3) / 1e9 / peak,
           "tflops": fused_flops(w) / (ms * 1e-3) / 1e12, "tensor_frac": fused_flops(w) / (ms * 1e-3) / 1e12 / tf,
           "tensor_peak_kind": tf_kind, "accept_len_mean": float(L.mean()), "clocks": clk}
    return out, (inp, head_d, hid_d, draft, dtok, ua, uf, fv, call)


def run_fused_only(args, w, rank=0, world=1):
    """spec_verify_fused on the fused workload (one replica per rank)."""
    import torch
    import torch.distributed as dist
    from mtp_speculative_decoding_draft_gb300.build import build

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    if rank == 0 or world == 1:
        build()
    if world > 1:
        dist.barrier()
        build()
    if args.greedy:
        w = W.replace(w, mode=W.GREEDY)
    peak, peak_kind = measured_peaks()
    from mtp_speculative_decoding_draft_gb300 import binding as bd
    if args.trace:
        _, head_d, hid_d, draft, dtok, ua, uf, fv = _fused_setup(w)
        stoch = w.mode == 1

        def traced_call():
            fv(w.T, head_d, hid_d, draft if stoch else None, dtok, ua if stoch else None, uf if stoch else None)

        for _ in range(args.warmup):
            traced_call()
        torch.cuda.synchronize()
        return print_trace(traced_call, args.trace, torch, bd)
    n0 = bd.launch_count()
    res, (inp, head_d, hid_d, draft, dtok, ua, uf, fv, call) = time_fused(w, args.steps, args.warmup, peak)
    launches = bd.launch_count() - n0 - 2 * args.warmup
    ms = max_over_ranks(res["ms_per_call"])
    # end to end: per call the hidden states, the draft's logits and tokens and
    # the uniforms from pinned host memory (the head stays resident, like any
    # weight), the outputs read back
    stoch = w.mode == 1
    stream = torch.cuda.current_stream()
    pairs = [(hid_d.cpu().pin_memory(), hid_d), (dtok.cpu().pin_memory(), dtok)]
    if stoch:
        pairs += [(draft.cpu().pin_memory(), draft), (ua.cpu().pin_memory(), ua), (uf.cpu().pin_memory(), uf)]
    outs = [(torch.empty(t.numel(), dtype=t.dtype).pin_memory(), t) for t in (fv.out_tok, fv.accept_len, fv.num_accepted)]
    h2d = sum(h.numel() * h.element_size() for h, _ in pairs)
    d2h = sum(h.numel() * h.element_size() for h, _ in outs)

    def e2e_call():
        for h, dv in pairs:
            dv.copy_(h, non_blocking=True)
        call()
        for h, dv in outs:
            h.copy_(dv, non_blocking=True)
        stream.synchronize()

    for _ in range(max(1, args.warmup)):
        e2e_call()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_call()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps)
    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return
    fb = fused_bytes(w)
    ach = fb / (ms * 1e-3) / 1e9
    _, L, _ = fv.results()
    line = {"metric": METRIC, "value": job_rate(ms, world), "unit": "verify calls/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 head and hidden / fp32 accumulate",
            "data": "synthetic (seeded)", "config": config_of(w, args),
            "accept_len_mean": float(L.mean()), "acceptance": acceptance_metrics(L, w.k),
            "roofline": {"bound": "hbm", "kernel": "fv_gemm_kernel + fv_finish_kernel", "achieved": ach,
                         "peak": peak, "unit": "GB/s", "frac": ach / peak, "peak_kind": peak_kind,
                         "traffic": ncu_traffic("fv_gemm_kernel + fv_finish_kernel",
                                                "%s/%s" % (w.name, "stochastic" if w.mode == 1 else "greedy")),
                         "bytes_per_launch": fb, "avg_launch_ms": ms, "launches": args.steps,
                         "tflops": res["tflops"], "tensor_frac": res["tensor_frac"]},
            "e2e": {"value": job_rate(e2e_ms, world), "unit": "verify calls/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": int(launches), "clocks": res["clocks"]}
    if not args.no_cpu_baseline and world == 1:
        try:
            ts = cpu_oracle_fused_times(args, 3, 4, budget_s=60)
            t_call = float(np.median(ts))
            line["cpu_baseline"] = dict({"value": 1.0 / t_call, "unit": "verify calls/s", "cores": 1, "kind": "oracle",
                                         "sample": "median of %d calls: the oracle forms the logits and verifies 4 of "
                                                   "the %d sequences, single-threaded float64 numpy; scaled to the "
                                                   "batch" % (len(ts), w.B)}, **host_cpu())
        except Exception as e:  # report, do not hide
            line["cpu_baseline"] = {"value": None, "error": str(e)[:300]}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_verify_only(args, w, rank=0, world=1):
    """spec_verify on the verify sweep: B sequences, k drafts, V-wide rows
    (one replica per rank; rank 0 prints the line)."""
    import torch
    import torch.distributed as dist
    from mtp_speculative_decoding_draft_gb300 import binding as bd
    from mtp_speculative_decoding_draft_gb300.build import build
    from mtp_speculative_decoding_draft_gb300.model import Verifier, to_device

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    if rank == 0 or world == 1:
        build()
    if world > 1:
        dist.barrier()
        build()
    inp = W.verify_inputs(w)
    t_d, l_d = to_device(inp["target_logits"]), to_device(inp["draft_logits"])
    # drafts drawn from q at u_draft (the rejection rate the config states)
    d_d = drafts_from_q(l_d.view(w.B, w.k, w.V), to_device(inp["u_draft"]), w.T)
    d = d_d.cpu().numpy()
    ua, uf = to_device(inp["u_accept"]), to_device(inp["u_final"])
    ver = Verifier(w.B, w.k, w.V)
    stoch = w.mode == 1

    def step():
        ver(w.T, w.mode, t_d, l_d if stoch else None, d_d, ua if stoch else None, uf if stoch else None)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if args.trace:
        return print_trace(step, args.trace, torch, bd)
    if world > 1:
        dist.barrier()
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    clocks.start()
    n0 = bd.launch_count()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    launches = bd.launch_count() - n0
    clk = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps)
    assert bd.get_status(ver.ws) == 0
    _, L, _ = ver.results()

    # end to end: the call's inputs from pinned host memory, its outputs read back
    stream = torch.cuda.current_stream()
    pairs = [(torch.from_numpy(inp["target_logits"]).pin_memory(), t_d), (torch.from_numpy(d).pin_memory(), d_d)]
    if stoch:
        pairs += [(torch.from_numpy(inp["draft_logits"]).pin_memory(), l_d),
                  (torch.from_numpy(inp["u_accept"]).pin_memory(), ua), (torch.from_numpy(inp["u_final"]).pin_memory(), uf)]
    outs = [(torch.empty(t.numel(), dtype=t.dtype).pin_memory(), t)
            for t in (ver.out_tok, ver.accept_len, ver.num_accepted)]
    h2d = sum(h.numel() * h.element_size() for h, _ in pairs)
    d2h = sum(h.numel() * h.element_size() for h, _ in outs)

    def e2e_step():
        for h, dv in pairs:
            dv.copy_(h, non_blocking=True)
        step()
        for h, dv in outs:
            h.copy_(dv, non_blocking=True)
        stream.synchronize()

    for _ in range(max(1, args.warmup)):
        e2e_step()
    if world > 1:
        dist.barrier()
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps)
    assert bd.get_status(ver.ws) == 0
    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return
    peak, peak_kind = measured_peaks()
    vb = verify_bytes(w)
    ach = vb / (ms * 1e-3) / 1e9
    vkernel = verify_kernel_name(w)
    line = {"metric": METRIC, "value": job_rate(ms, world), "unit": "verify calls/s", "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32 logits", "data": "synthetic (seeded)", "config": config_of(w, args),
            "accept_len_mean": float(L.mean()),
            "acceptance": acceptance_metrics(L, w.k),
            "roofline": {"bound": "hbm", "kernel": vkernel, "achieved": ach, "peak": peak, "unit": "GB/s",
                         "frac": ach / peak, "peak_kind": peak_kind,
                         "traffic": ncu_traffic(vkernel, f"{w.name}/{'greedy' if w.mode == W.GREEDY else 'stochastic'}"),
                         "bytes_per_launch": vb,
                         "avg_launch_ms": ms, "launches": args.steps},
            "e2e": {"value": job_rate(e2e_ms, world), "unit": "verify calls/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": int(launches), "clocks": clk}
    if not args.no_cpu_baseline and world == 1:   # rank 0 at N = 1 only
        try:
            n_seq = 16
            t_call = cpu_oracle_verify_times(args, 1, n_seq)[0]
            line["cpu_baseline"] = dict({"value": 1.0 / t_call, "unit": "verify calls/s", "cores": 1, "kind": "oracle",
                                         "sample": "the oracle verifies %d of the %d sequences, single-threaded "
                                                   "float64 numpy; scaled to the batch" % (min(n_seq, w.B), w.B)},
                                        **host_cpu())
        except Exception as e:  # report, do not hide
            line["cpu_baseline"] = {"value": None, "error": str(e)[:300]}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- secondary workloads

SECONDARY_STEPS = 50


def _targets_from_own_draft(m, w, u, sd, growth):
    """Target logits = the module's own (untimed) draft logits + noise whose std
    is sd at position 0 and grows by `growth` per position; the bonus row reuses
    the last draft row.  Returns (target [B, k+1, V] float32, mean draft-logit std)."""
    import torch
    from mtp_speculative_decoding_draft_gb300.model import to_device
    stoch = w.mode == 1
    m.draft(w.T, w.mode, to_device(u["u_draft"]) if stoch else None, logits=True)
    torch.cuda.synchronize()
    dl = m.draft_logits.view(w.B, w.k, w.V).cpu().numpy()
    target = W.draft_noise(W.Workload(w.name, B=w.B, k=w.k + 1, V=w.V, seed=w.seed,
                                      draft_noise_std0=sd, noise_growth=growth), w.k + 1)
    for j in range(w.k + 1):
        target[:, j] += dl[:, min(j, w.k - 1)]
    return target, float(np.mean(dl.std(axis=2)))


def secondary_step(w, steps, warmup, peak):
    """spec_step on another workload (direct calls, inputs resident), CUDA-event
    timed with its own clock samples: steps/s, ms and the fraction of the step's
    HBM roofline."""
    import torch
    from mtp_speculative_decoding_draft_gb300 import binding as bd
    from mtp_speculative_decoding_draft_gb300.model import DraftModule, to_device
    wts = W.make_weights(w)
    ctx = W.make_context(w)
    u = W.make_uniforms(w)
    m = DraftModule(w, wts)
    m.set_context(ctx)
    target, _ = _targets_from_own_draft(m, w, u, w.draft_noise_std0, w.noise_growth)
    m.set_context(ctx)
    stoch = w.mode == 1
    td = to_device(target)
    ud, ua, uf = (to_device(u[n]) if stoch else None for n in ("u_draft", "u_accept", "u_final"))

    def step():
        m.step(w.T, w.mode, td, ud, ua, uf, logits=stoch)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / steps
    assert m.status() == 0, "device status word %d" % m.status()
    L = m.accept_len.cpu().numpy()
    sb = step_bytes(w, ctx["ctx_len"], stoch)
    out = {"workload": w.name, "value": 1e3 / ms, "unit": "steps/s", "ms_per_step": ms, "steps": steps,
           "warmup": warmup, "accepted_tok_s": 1e3 / ms * float(L.sum()), "accept_len_mean": float(L.mean()),
           "hbm_bytes_per_step": sb, "hbm_roofline_frac": sb / (ms * 1e-3) / 1e9 / peak, "clocks": clk}
    del m, td
    torch.cuda.empty_cache()
    return out


def secondary_verify(k, greedy, steps, warmup, peak):
    """spec_verify on the verify sweep at depth k (drafts drawn from q), CUDA-event
    timed with its own clock samples: ms per call and the fraction of the copy
    peak on the algorithmic bytes."""
    import torch
    from mtp_speculative_decoding_draft_gb300 import binding as bd
    from mtp_speculative_decoding_draft_gb300.model import Verifier, to_device
    w = W.with_k(W.VERIFY_SWEEP, k)
    if greedy:
        w = W.replace(w, mode=W.GREEDY)
    inp = W.verify_inputs(w)
    t_d, l_d = to_device(inp["target_logits"]), to_device(inp["draft_logits"])
    d_d = drafts_from_q(l_d.view(w.B, w.k, w.V), to_device(inp["u_draft"]), w.T)
    ua, uf = to_device(inp["u_accept"]), to_device(inp["u_final"])
    ver = Verifier(w.B, w.k, w.V)
    stoch = w.mode == 1

    def call():
        ver(w.T, w.mode, t_d, l_d if stoch else None, d_d, ua if stoch else None, uf if stoch else None)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        call()
    e1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / steps
    assert bd.get_status(ver.ws) == 0
    _, L, _ = ver.results()
    vb = verify_bytes(w)
    out = {"workload": "%s/%s" % (w.name, "greedy" if greedy else "stochastic"), "ms_per_call": ms,
           "calls_s": 1e3 / ms, "steps": steps, "warmup": warmup, "bytes_per_call": vb,
           "achieved_gbs": vb / (ms * 1e-3) / 1e9, "frac": vb / (ms * 1e-3) / 1e9 / peak,
           "accept_len_mean": float(L.mean()), "drafts": "drawn from q at u_draft", "clocks": clk}
    del ver, t_d, l_d
    torch.cuda.empty_cache()
    return out


def run_secondary(peak, steps=SECONDARY_STEPS, warmup=5):
    """The batched stochastic workload's step, the verify sweep at k = 3 and the
    verification from hidden states at the batched shape (greedy and stochastic
    each), timed in this process; failures are reported in place of the
    figures."""
    out = {}
    for key, fn in (("batched_stochastic_step", lambda: secondary_step(W.BATCHED_STOCHASTIC, steps, warmup, peak)),
                    ("verify_sweep_k3_greedy", lambda: secondary_verify(3, True, 4 * steps, warmup, peak)),
                    ("verify_sweep_k3_stochastic", lambda: secondary_verify(3, False, 4 * steps, warmup, peak)),
                    ("fused_verify_b64_k3_greedy",
                     lambda: time_fused(W.replace(W.FUSED_VERIFY, mode=W.GREEDY), steps, warmup, peak)[0]),
                    ("fused_verify_b64_k3_stochastic", lambda: time_fused(W.FUSED_VERIFY, steps, warmup, peak)[0])):
        try:
            out[key] = fn()
        except Exception as e:  # report, do not hide
            out[key] = {"error": str(e)[:300]}
    return out


def print_trace(step, n_steps, torch, bd):
    """Diagnostic (--trace N): run N steps with the launch-tracing library and
    print the live kernel timeline -- per launch its start, dependency release
    and end on the GPU's global timer -- for the last step, and per kernel kind
    the mean time it adds to the timeline (its end past everything before it)."""
    bd.trace_read()                      # drop the warm-up's records
    n0 = bd.launch_count()
    for _ in range(n_steps):
        step()
    torch.cuda.synchronize()
    per_step = (bd.launch_count() - n0) // n_steps
    recs = bd.trace_read()
    if not recs or per_step < 1:
        raise SystemExit("no trace records: run with the trace build (MTP_LIB_VARIANT=trace)")
    t_first = recs[0]["start"]
    cur = t_first
    agg = {}
    for r in recs:
        excl = max(0, r["end"] - max(r["start"], cur))
        gap = max(0, r["start"] - cur)
        cur = max(cur, r["end"])
        a = agg.setdefault(r["name"], [0, 0.0, 0.0, 0.0, 0.0])
        a[0] += 1
        a[1] += r["end"] - r["start"]
        a[2] += (r["end"] - r["dep"]) if r["dep"] else 0.0
        a[3] += excl
        a[4] += gap
    total = cur - t_first
    print("traced %d steps, %d launches, %.1f us per step" % (n_steps, len(recs), total / 1e3 / n_steps))
    print("%-28s %6s %10s %12s %12s %10s" % ("kernel", "count", "span us", "after dep us", "adds us", "gap us"))
    for name, (n, span, dep, excl, gap) in sorted(agg.items(), key=lambda kv: -kv[1][3]):
        print("%-28s %6d %10.2f %12.2f %12.2f %10.2f" % (name, n, span / n / 1e3, dep / n / 1e3, excl / n / 1e3,
                                                         gap / n / 1e3))
    last = recs[-per_step:]
    t0 = last[0]["start"]
    print("\nlast step (us from its first launch's start; marks: the kernel's intermediate points)")
    print("%-28s %9s %9s %9s %9s   %s" % ("kernel", "start", "dep", "end", "span", "marks"))

    def rel(t):
        return "%9.2f" % ((t - t0) / 1e3) if t else "%9s" % "-"
    for r in last:
        print("%-28s %s %s %s %9.2f   %s" % (r["name"], rel(r["start"]), rel(r["dep"]), rel(r["end"]),
                                            (r["end"] - r["start"]) / 1e3,
                                            " ".join(rel(m).strip() for m in r["marks"] if m)))


def run_ours(args):
    import torch
    import torch.distributed as dist
    from mtp_speculative_decoding_draft_gb300 import binding as bd
    from mtp_speculative_decoding_draft_gb300.build import build
    from mtp_speculative_decoding_draft_gb300.model import DraftModule, to_device

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    w = W.WORKLOADS[args.workload]
    if w.fused:
        return run_fused_only(args, w, rank, world)
    if w.verify_only:
        return run_verify_only(args, _verify_workload(args), rank, world)
    if rank == 0 or world == 1:
        build()
    if world > 1:
        dist.barrier()
        build()
    stoch = w.mode == 1
    wts = W.make_weights(w)
    ctx = W.make_context(w)
    u = W.make_uniforms(w)
    nm = max(1, min(args.modules, w.k))
    if (args.stop_p is not None or args.draft_vocab) and nm > 1:
        raise SystemExit("--stop-p and --draft-vocab run one module; drop --modules")
    if args.stop_p is not None and args.draft_vocab:
        raise SystemExit("--stop-p and --draft-vocab are separate calls; give one")
    extra = [W.make_module_weights(w, i, E=wts["E"]) for i in range(1, nm)]
    caches = [W.make_module_cache(w, i) for i in range(1, nm)]
    m = DraftModule(w, wts, extra_modules=extra)
    m.set_context(ctx, caches)
    draft_std = None
    if w.mode == 1 or args.correlated > 0:
        # target = the module's own draft logits + noise (growing with position
        # for the stochastic workloads; N(0, SIGMA^2) at every position with --correlated SIGMA)
        m.draft(w.T, w.mode, to_device(u["u_draft"]) if stoch else None, logits=True)
        torch.cuda.synchronize()
        dl = m.draft_logits.view(w.B, w.k, w.V).cpu().numpy()
        sd, gr = (w.draft_noise_std0, w.noise_growth) if w.mode == 1 else (args.correlated, 1.0)
        draft_std = float(np.mean(dl.std(axis=2)))
        target = W.draft_noise(W.Workload(w.name, B=w.B, k=w.k + 1, V=w.V, seed=w.seed,
                                          draft_noise_std0=sd, noise_growth=gr), w.k + 1)
        for j in range(w.k + 1):
            target[:, j] += dl[:, min(j, w.k - 1)]
        m.set_context(ctx, caches)
    else:
        target = W.target_logits(w)
    target_d = to_device(target)
    ud = to_device(u["u_draft"]) if stoch else None
    ua = to_device(u["u_accept"]) if stoch else None
    uf = to_device(u["u_final"]) if stoch else None
    logits_out = stoch

    if args.draft_vocab:
        vmap, head = W.make_draft_vocab(w, args.draft_vocab)
        m.set_draft_vocab(vmap, head)

    def step(stream=None):
        if args.draft_vocab:
            m.step_reduced(w.T, w.mode, target_d, ud, ua, uf, logits=logits_out, stream=stream)
        elif args.stop_p is not None:
            m.step_dynamic(w.T, w.mode, args.stop_p, target_d, ud, ua, uf, logits=logits_out, stream=stream)
        else:
            m.step(w.T, w.mode, target_d, ud, ua, uf, logits=logits_out, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if args.trace:
        return print_trace(step, args.trace, torch, bd)
    graph, graph_launches = None, 0
    if args.graph:
        # one step captured in a CUDA graph (after the warm-up above, on a side
        # stream first, as capture wants); the timed loop replays it
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        c0 = bd.launch_count()
        with torch.cuda.graph(graph):
            step()
        graph_launches = bd.launch_count() - c0
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()

    def run_step():
        if graph is not None:
            graph.replay()
        else:
            step()

    if world > 1:
        dist.barrier()

    clocks = ClockSampler(local)
    clocks.start()
    n0 = bd.launch_count()
    stream = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        run_step()
    e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    # a replay launches the captured kernels without passing through the host library
    launches = graph_launches * args.steps if graph is not None else bd.launch_count() - n0
    clk = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps)
    assert m.status() == 0, "device status word %d" % m.status()
    L = m.accept_len.cpu().numpy()

    # per-kernel durations: the same steps with an event pair around each launch
    bd.profiler_enable(True)
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    lm_ms, lm_n = bd.profiler_read(bd.KC_LMHEAD)
    ver_ms, _ = bd.profiler_read(bd.KC_VERIFY)
    att_ms, _ = bd.profiler_read(bd.KC_ATTN)
    gem_ms, _ = bd.profiler_read(bd.KC_GEMV)
    bd.profiler_enable(False)

    # end to end: per-step inputs from pinned host memory, results read back
    h_h = torch.from_numpy(ctx["h"].view(np.int16)).view(torch.bfloat16).pin_memory()
    h_tok = torch.from_numpy(ctx["last_tok"].astype(np.int32)).pin_memory()
    h_ctx = torch.from_numpy(ctx["ctx_len"].astype(np.int32)).pin_memory()
    h_tgt = torch.from_numpy(target).pin_memory()
    h_u = [torch.from_numpy(u[n]).pin_memory() for n in ("u_draft", "u_accept", "u_final")] if stoch else []
    d_u = [ud, ua, uf] if stoch else []
    o_out = torch.empty(m.out_tok.numel(), dtype=torch.int32).pin_memory()
    o_len = torch.empty(w.B, dtype=torch.int32).pin_memory()
    o_acc = torch.empty(w.B, dtype=torch.int32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in [h_h, h_tok, h_ctx, h_tgt] + h_u)
    d2h = sum(t.numel() * t.element_size() for t in [o_out, o_len, o_acc])

    def e2e_step():
        m.h.copy_(h_h, non_blocking=True)
        m.last_tok.copy_(h_tok, non_blocking=True)
        m.ctx_len.copy_(h_ctx, non_blocking=True)
        target_d.copy_(h_tgt.view(-1) if target_d.dim() == 1 else h_tgt, non_blocking=True)
        for hd, dd in zip(h_u, d_u):
            dd.copy_(hd, non_blocking=True)
        step()
        o_out.copy_(m.out_tok, non_blocking=True)
        o_len.copy_(m.accept_len, non_blocking=True)
        o_acc.copy_(m.num_accepted, non_blocking=True)
        stream.synchronize()

    for _ in range(max(1, args.warmup)):
        e2e_step()
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps)

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    peak, peak_kind = measured_peaks()
    depths = None
    if args.stop_p is not None:
        ke = m.k_eff.cpu().numpy()
        # weight-streaming launches of batches of up to 4 return once every sequence has stopped
        depths = min(w.k, int(ke.max()) + 1) if w.B <= 4 else w.k
    hr = args.draft_vocab or None
    sb = step_bytes(w, ctx["ctx_len"], logits_out, nm, depths, hr)
    steps_s = job_rate(ms, world)
    tokens_per_step = float(L.sum())
    lm_avg = lm_ms / max(lm_n, 1)
    lm_b = lmhead_bytes(w, logits_out, hr)
    ach = lm_b / (lm_avg * 1e-3) / 1e9
    # Batches of five or more run the LM head as a tensor-core GEMM; smaller ones as the GEMV.
    lm_kernel = "tc_gemm_kernel(LM head)" if w.B >= 5 and w.d % 64 == 0 else "lm_head_gemv"
    line = {
        "metric": METRIC, "value": steps_s, "unit": "steps/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 weights / fp32 accumulate", "data": "synthetic (seeded, random weights)",
        "config": config_of(w, args),
        "accepted_tok_s": steps_s * tokens_per_step,
        "accept_len_mean": float(L.mean()),
        "acceptance": acceptance_metrics(L, w.k),
        "draft_logit_std": draft_std,
        "k_eff_mean": float(m.k_eff.float().mean().item()) if args.stop_p is not None else None,
        "hbm_bytes_per_step": sb,
        "hbm_roofline_frac": sb / (ms * 1e-3) / 1e9 / peak,
        "roofline": {"bound": "hbm", "kernel": lm_kernel, "achieved": ach, "peak": peak, "unit": "GB/s",
                     "frac": ach / peak, "peak_kind": peak_kind,
                     "traffic": ncu_traffic(lm_kernel, w.name) if not logits_out else None,
                     "bytes_per_launch": lm_b, "avg_launch_ms": lm_avg, "launches": lm_n},
        "kernel_ms_per_step": {"lm_head": lm_ms / args.steps, "verify": ver_ms / args.steps,
                               "attention": att_ms / args.steps, "gemv_other": gem_ms / args.steps},
        "e2e": {"value": job_rate(e2e_ms, world), "unit": "steps/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": int(launches),
        "clocks": clk,
    }
    if not args.no_secondary and world == 1 and args.workload == W.SINGLE_GREEDY.name and not (
            args.graph or args.stop_p is not None or args.draft_vocab or nm > 1 or args.correlated):
        line["secondary"] = run_secondary(peak)
    if not args.no_cpu_baseline and world == 1:   # rank 0 at N = 1 only
        try:
            ts = cpu_oracle_step_times(args.workload, w.k, CPU_BASELINE_STEPS, budget_s=CPU_BASELINE_BUDGET_S)
            t_step = float(np.median(ts))
            line["cpu_baseline"] = dict({"value": 1.0 / t_step, "unit": "steps/s", "cores": 1, "kind": "oracle",
                                         "steps_timed": len(ts), "step_s_min": float(min(ts)),
                                         "step_s_max": float(max(ts)),
                                         "sample": "median of %d full steps (all %d depths + verification) of this "
                                                   "workload, single-threaded float64 numpy (up to %d steps within "
                                                   "%d s)" % (len(ts), w.k, CPU_BASELINE_STEPS, CPU_BASELINE_BUDGET_S)},
                                        **host_cpu())
        except Exception as e:  # report, do not hide
            line["cpu_baseline"] = {"value": None, "error": str(e)[:300]}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=W.SINGLE_GREEDY.name, choices=sorted(W.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the batched-stochastic step and verify-sweep figures added to the default line")
    ap.add_argument("--k", type=int, default=0, help="draft depth for the verify sweep (1..5)")
    ap.add_argument("--greedy", action="store_true", help="greedy verification for the verify sweep")
    ap.add_argument("--stop-p", type=float, default=None,
                    help="dynamic draft length: stop a sequence's chain at its first depth of draft confidence "
                         "below this (spec_step_dynamic)")
    ap.add_argument("--draft-vocab", type=int, default=0,
                    help="reduced draft vocabulary of this many ids (spec_step_reduced); 0 = the full head")
    ap.add_argument("--correlated", type=float, default=0.0, metavar="SIGMA",
                    help="greedy workloads: target logits = the draft's own logits + N(0, SIGMA^2) instead of "
                         "i.i.d. N(0, 16); 0 = off")
    ap.add_argument("--graph", action="store_true",
                    help="time replays of one step captured in a CUDA graph instead of direct calls")
    ap.add_argument("--trace", type=int, default=0, metavar="N",
                    help="diagnostic: run N steps on the launch-tracing build and print the live kernel "
                         "timeline instead of the JSON line")
    ap.add_argument("--modules", type=int, default=1,
                    help="distinct draft modules (depth j runs module min(j, modules-1)); 1 = one reused module")
    args = ap.parse_args()
    if args.trace:
        # the launch-tracing library, built and selected before the binding loads one
        from mtp_speculative_decoding_draft_gb300.build import build
        build(variant="trace")
        os.environ["MTP_LIB_VARIANT"] = "trace"
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
