"""Throughput of the chunked test-time memory update on GB300.

One step = one call of atlas_mem_forward over a whole workload (all heads,
all tokens) with its inputs resident in HBM, preceded by the reset of the
in/out state buffer to M_0.  Default workload: the linear DeltaNet-like
memory (B=8, H=16, N=4096, d=128, c=1, b=64, bf16 K/Q/V, fp32 state).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload ID]
                  [--impl atlas|reference]

Prints one JSON line (rank 0).  Under torchrun every rank runs its own copy
of the workload (heads are independent; no collective on the data path) and
the reported value is the tokens of all ranks over the slowest rank's time.
``--impl reference`` times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "memory-update tokens/sec on 1 GB300 per config; % of bf16 tensor/HBM roofline"
UNIT = "tokens/s"
L2_BYTES = 129 * 1024 * 1024  # L2 of one GB300


# ----------------------------------------------------------------- helpers

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def aggregate(tokens_per_rank: int, world: int, elapsed_max_s: float, steps: int) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * world * steps / elapsed_max_s


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p.get("hbm_gbs", 6800.0), p.get("bf16_tflops", 1900.0), \
            p.get("bf16_tflops_sustained", 1700.0), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


CSRC = os.path.join(ROOT, "test_memorization_recurrent_gb300", "csrc")


def source_hashes(files):
    """sha256 of each named file under the package's csrc/."""
    out = {}
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            out[f] = hashlib.sha256(fh.read()).hexdigest()
    return out


def profile_traffic(files, profile_name: str, units_per_launch: float):
    """DRAM bytes per call from a committed ncu summary, scaled to this call, or
    None if the summary is missing or any of the sources it was taken on (one
    `source_sha256: <hash> <file>` line each) has changed since."""
    path = os.path.join(ROOT, "profiles", profile_name)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    listed = dict((f, h) for h, f in re.findall(r"source_sha256:\s*([0-9a-f]{64})\s+(\S+)", text))
    m_b = re.search(r"dram_bytes_per_unit:\s*([0-9.eE+-]+)", text)
    if not m_b or set(listed) != set(files) or listed != source_hashes(files):
        return None
    return float(m_b.group(1)) * units_per_launch


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons.  The sampler starts
    before the warm-up; only samples stamped inside the timed region count."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 20):
        self.gpu = gpu_index
        self.interval = interval_ms
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def __enter__(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval), "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def wait_ready(self, timeout_s: float = 5.0):
        """Block until the sampler has written its first line (or timeout)."""
        t = time.time()
        while self.proc is not None and time.time() - t < timeout_s:
            if os.path.getsize(self.path) > 0:
                return
            time.sleep(0.02)

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()
        time.sleep(2.5 * self.interval / 1e3)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        import datetime
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        try:
            text = open(self.path).read()
            os.unlink(self.path)
        except OSError:
            text = ""
        for line in text.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(f[2]), float(f[3]), f[6:10]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        inside = [r for r in rows if self.t0 is not None and self.t0 - 0.01 <= r[0] <= self.t1 + 0.01]
        window = "timed region"
        if not inside:  # region shorter than the sampling interval: nearest samples
            inside = sorted(rows, key=lambda r: abs(r[0] - (self.t0 or 0)))[:3]
            window = "nearest to the timed region"
        reasons = set()
        for r in inside:
            for n, v in zip(names, r[3]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "samples": len(inside),
                "window": window, "reasons": sorted(reasons)}


# ------------------------------------------------------------------ oracle leg

def oracle_rate(w, heads, n_tokens, seed=0):
    """Time the fp64 oracle on `heads` heads x `n_tokens` tokens on all host cores."""
    import oracle
    oracle.build()
    inp = W.generate(w, seed=seed, heads=heads, n_tokens=n_tokens)
    a, b_, c_ = w.ns_coef
    cfg = oracle.make_cfg(n_tokens, w.d_k, w.d_v, w.d_h, w.mem, w.phi, w.loss, w.c, w.b,
                          w.ns_steps, a, b_, c_, w.ns_eps, loss_param=w.loss_param,
                          phi_coef=w.phi_coef)
    t = time.perf_counter()
    oracle.forward(cfg, inp["K"], inp["Q"], inp["V"], inp["alpha"], inp["eta"], inp["theta"],
                   inp["gamma"], inp["M0"])
    dt = time.perf_counter() - t
    return len(heads) * n_tokens / dt, dt


def oracle_sample(w):
    """A bounded sample of the workload for the CPU oracle (a few seconds to tens of
    seconds on the host): whole heads where affordable, else a token prefix."""
    cores = os.cpu_count() or 1
    if w.wid in (1, 2):
        return list(range(w.heads)), w.N
    if w.wid == 3:
        return list(range(min(w.heads, cores))), 512 if w.phi != W.PHI_POLY else 128
    if w.wid == 4:
        return list(range(min(w.heads, cores))), min(2048, w.N)
    return list(range(min(w.heads, cores))), 16


def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    heads, n = oracle_sample(w)
    cores = os.cpu_count() or 1
    for _ in range(args.warmup):
        oracle_rate(w, heads[:1], min(n, 64))
    # keep the whole timed run near two minutes at most: one step on the full sample
    # measures its cost, and the heads per step shrink if K steps would take longer
    _, dt0 = oracle_rate(w, heads, n)
    budget = 120.0 / max(1, args.steps)
    if dt0 > budget:  # (never fewer heads than host cores: the oracle threads over heads)
        heads = heads[:max(min(cores, len(heads)), int(len(heads) * budget / dt0))]
    rates, times = [], []
    for _ in range(args.steps):
        r, dt = oracle_rate(w, heads, n)
        rates.append(r)
        times.append(dt)
    value = len(heads) * n * len(rates) / sum(times)
    sample = f"{len(heads)} heads x {n} tokens of {w.name} per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d_k": w.d_k, "d_v": w.d_v,
                   "d_h": w.d_h, "c": w.c, "b": w.b},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- GPU leg

# Per path: the sources its kernels are compiled from (a profile summary counts
# only while all of them are unchanged) and the summary's file name.
_TC = ["tc_primitives.cuh", "common.cuh", "kernels.h"]
KERNEL_OF_PATH = {
    "linear_tc": (["linear_tc.cu", "linear_simt.cu", "linear_simt_body.cuh"] + _TC,
                  "linear_tc_{wname}.md"),
    "linear_simt": (["linear_simt.cu", "linear_simt_elastic.cu", "linear_simt_bregman.cu",
                     "linear_simt_kl.cu", "linear_simt_body.cuh", "simt_tiles.cuh", "common.cuh",
                     "kernels.h"], "linear_simt_{wname}.md"),
    "linear_wide": (["linear_wide.cu", "simt_tiles.cuh", "common.cuh", "kernels.h"],
                    "linear_wide_{wname}.md"),
    "linear_seq": (["linear_seq.cu", "common.cuh", "kernels.h"], "linear_seq_{wname}.md"),
    "linear_chunk": (["linear_chunk.cu", "tc_gemm.cu"] + _TC, "linear_chunk_{wname}.md"),
    "mlp_simt": (["mlp_simt.cu", "tc_gemm.cu", "ns_fused.cu"] + _TC, "mlp_simt_{wname}.md"),
    "mlp_tc": (["mlp_tc.cu"] + _TC, "mlp_tc_{wname}.md"),
    "linear_bwd": (["linear_bwd.cu", "common.cuh", "kernels.h"], "linear_bwd_{wname}.md"),
}

# Workloads measured beside the headline one, and the token prefix each is timed
# on (None = the whole workload).  The Newton-Schulz workload runs on a prefix of
# all 16 heads: its full million-token length is ~70 s per call at today's rate.
PER_CONFIG = ((1, None), (3, None), (4, None), (5, 1024))


def variant_workloads():
    """Variants measured beside the five workloads: the gated degree-3 polynomial
    map (input gating a = (0, 1, 1, 1)) on the wide-feature workload's shape with
    d_k = 16 (D = 968 features), window 64, momentum and decay, bounded step; the
    layer-normalised and the gated MLP memories on the MLP workload's shape (first
    1024 tokens of all 32 heads; they run on the CUDA-core MLP path); the Miras
    retention gates (elastic net lambda = 0.01, Bregman with the sigmoid link, KL of
    row mass 1, l_q with q = 3) and the robust bias (Delta = 0.5) on the DeltaNet
    workload's shape (first 1024 tokens of all 128 heads; CUDA-core linear kernel)."""
    return [W.workload(3, bounded=True, d_k=16, phi=W.PHI_POLY, phi_coef=(0.0, 1.0, 1.0, 1.0),
                       N=2048, theta_scale=0.002, name="poly3-gated-omega-c64-bf16"),
            W.workload(4, bounded=True, mem=W.MEM_MLP_LN, N=1024,
                       name="mlp-ln-momentum-b64-bf16"),
            W.workload(4, bounded=True, mem=W.MEM_MLP_GATED, N=1024,
                       name="mlp-gated-momentum-b64-bf16"),
            W.workload(2, retention=W.RET_ELASTIC, ret_param=0.01, N=1024,
                       name="linear-elastic-b64-bf16"),
            W.workload(2, retention=W.RET_BREGMAN, N=1024, name="linear-bregman-b64-bf16"),
            W.workload(2, retention=W.RET_KL, ret_param=1.0, N=1024, name="linear-kl-b64-bf16"),
            W.workload(2, retention=W.RET_LQ, ret_param=3.0, N=1024, name="linear-lq3-b64-bf16"),
            W.workload(2, loss=W.LOSS_ROBUST, loss_param=0.5, N=1024,
                       name="linear-robust-b64-bf16")]


def time_device(w, run, d, steps, warmup, stream, clk=None, world=1):
    """Device-resident timing of `steps` calls (each preceded by the reset of the
    state buffer to M_0).  A call whose data fits in L2 is preceded by a write
    of a buffer twice the L2 size, outside its events, and the step time is the
    sum of the per-step events; otherwise the steps run back to back and the
    step time is the whole loop's.  Returns (elapsed_s, kernel_s per call, flush)."""
    import torch
    import test_memorization_recurrent_gb300 as A
    bytes_launch = w.tokens * W.bytes_per_token(w) + 2 * 4 * w.heads * w.state_size
    flush = bytes_launch < 2 * L2_BYTES
    dev = run.Y.device
    scrub = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    s_start, s_end = [ev() for _ in range(steps)], [ev() for _ in range(steps)]
    k_start, k_end = [ev() for _ in range(steps)], [ev() for _ in range(steps)]
    t_start, t_end = ev(), ev()
    for _ in range(warmup):
        run(d)
    torch.cuda.synchronize()
    if clk is not None:
        clk.wait_ready()
    barrier(world)
    torch.cuda.synchronize()
    if clk is not None:
        clk.mark_start()
    t_start.record(stream)
    for i in range(steps):
        if flush:
            scrub.fill_(float(i))
        s_start[i].record(stream)
        run.M.copy_(d["M0"])
        k_start[i].record(stream)
        A.atlas_mem_forward(d["K"], d["Q"], d["V"], d["alpha"], d["eta"], d["theta"],
                            d["gamma"], run.cfg, run.Y, run.M, stream)
        k_end[i].record(stream)
        s_end[i].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    if clk is not None:
        clk.mark_end()
    barrier(world)
    if flush:
        elapsed = sum(a.elapsed_time(b) for a, b in zip(s_start, s_end)) / 1e3
    else:
        elapsed = t_start.elapsed_time(t_end) / 1e3
    kernel_s = sum(a.elapsed_time(b) for a, b in zip(k_start, k_end)) / 1e3 / steps
    status = int(run.status.item())
    if status != 0:
        raise SystemExit(f"device status {status}: {A.atlas_mem_strerror(status)}")
    return elapsed, kernel_s, flush


def roofline(w, path, kernel_s):
    """Roofline record of one launch of workload `w` taking `kernel_s`: HBM-bound
    when its arithmetic intensity is below the ridge, else against the sustained
    bf16 tensor peak.  `traffic` comes from the committed ncu summary of the
    dominant kernel when that summary was taken on the current source."""
    hbm, tf, tf_sus, peak_kind = load_peaks()
    tokens = w.tokens
    bytes_launch = tokens * W.bytes_per_token(w) + 2 * 4 * w.heads * w.state_size
    flops_launch = tokens * W.flop_per_token(w)
    ridge = tf * 1e12 / (hbm * 1e9)
    # fp32 FMAs on CUDA cores: the token-serial, CUDA-core and wide-map linear kernels
    if path in ("linear_seq", "linear_simt", "linear_wide"):
        peak = fp32_alu_peak_tflops()
        achieved = flops_launch / kernel_s / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "peak_kind": "fp32 FMA peak from unit counts and clock"}
    elif flops_launch / bytes_launch < ridge:
        achieved = bytes_launch / kernel_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "peak_kind": f"{peak_kind} hbm_gbs"}
    else:
        achieved = flops_launch / kernel_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tf_sus, "unit": "TFLOP/s",
                "frac": achieved / tf_sus, "peak_kind": f"{peak_kind} bf16_tflops_sustained"}
    files, prof = KERNEL_OF_PATH.get(path, ([], ""))
    roof["traffic"] = profile_traffic(files, prof.format(wname=w.name), tokens) if files else None
    roof["kernel"] = path
    roof["kernel_ms"] = kernel_s * 1e3
    roof["algorithmic_bytes"] = bytes_launch
    roof["algorithmic_flops"] = flops_launch
    return roof


def measure_config(wid, n_tokens, steps, warmup, dev, with_cpu):
    """One workload (an id, or a Workload) measured on its own (rank 0, one GPU):
    rate, roofline, clocks during its timed region, and the oracle on a bounded
    sample of it."""
    import torch
    import test_memorization_recurrent_gb300 as A
    from test_memorization_recurrent_gb300.harness import Runner, to_device
    w = W.workload(wid, bounded=True) if isinstance(wid, int) else wid
    if n_tokens:
        w = w.with_(N=min(n_tokens, w.N))
    inp = W.generate(w)
    d = to_device(w, inp, dev)
    run = Runner(w, w.heads, w.N, device=dev)
    path = A.atlas_mem_path(run.cfg)
    stream = torch.cuda.current_stream()
    with Clocks(torch.cuda.current_device()) as clk:
        elapsed, kernel_s, flush = time_device(w, run, d, steps, warmup, stream, clk)
    rec = {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "path": path,
           "tokens_per_call": w.tokens, "steps": steps,
           "value": w.tokens * steps / elapsed, "unit": UNIT,
           "ms_per_step": elapsed / steps * 1e3,
           "launches_per_call": A.atlas_mem_launch_count(run.cfg),
           "roofline": roofline(w, path, kernel_s), "clocks": clk.summary(),
           "l2": "flushed before every step" if flush else "inputs larger than L2"}
    if n_tokens:
        rec["sample"] = f"first {w.N} tokens of every head (all {w.heads} heads)"
    del d, run
    torch.cuda.empty_cache()
    if with_cpu:
        heads, n = oracle_sample(w)
        rate, dt = oracle_rate(w, heads, n)
        rec["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": os.cpu_count(),
                               "kind": "oracle",
                               "sample": f"{len(heads)} heads x {n} tokens of {w.name}, {dt:.1f} s"}
    return rec


def fp32_alu_peak_tflops():
    """fp32 FMA peak of one GB300 from its unit counts and clock: 152 SMs x 128
    FP32 lanes x 2 FLOP per FMA x the maximum SM clock (2070 MHz)."""
    return 152 * 128 * 2 * 2.07e9 / 1e12


def _bwd_prof(w):
    files, prof = KERNEL_OF_PATH["linear_bwd"]
    return files, prof.format(wname=w.name), w.tokens


def measure_backward(steps, warmup, dev, momentum=False):
    """The backward pass over the whole DeltaNet-like workload (every head, every
    token), or the same shape with momentum in the forward (eta ~ U(0.5, 0.9)):
    rate, and the fraction of the fp32 CUDA-core peak it reaches."""
    import torch
    from test_memorization_recurrent_gb300.harness import BackwardRunner, to_device
    w = W.workload(2, eta=(0.5, 0.9), name="linear-momentum-b64-bf16") if momentum else \
        W.workload(2)
    inp = W.generate(w)
    d = to_device(w, inp, dev)
    r = np.random.default_rng(3)
    dY = torch.from_numpy(r.standard_normal((w.heads, w.N, w.d_v)).astype(np.float32)).to(dev)
    dMN = torch.zeros((w.heads, w.state_size), dtype=torch.float32, device=dev)
    run = BackwardRunner(w, w.heads, w.N, device=dev)
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    with Clocks(torch.cuda.current_device()) as clk:
        for _ in range(warmup):
            run(d, dY, dMN)
        torch.cuda.synchronize()
        clk.wait_ready()
        clk.mark_start()
        ev[0].record(stream)
        for _ in range(steps):
            run(d, dY, dMN)
        ev[1].record(stream)
        torch.cuda.synchronize()
        clk.mark_end()
    if int(run.status.item()) != 0:
        raise SystemExit(f"backward status {int(run.status.item())}")
    s = ev[0].elapsed_time(ev[1]) / 1e3 / steps
    flops = w.tokens * W.bwd_flop_per_token(w)
    peak = fp32_alu_peak_tflops()
    rec = {"workload": w.name, "what": "backward pass (dK, dQ, dV, dalpha, deta, dtheta, dM_0)",
           "tokens_per_call": w.tokens, "steps": steps, "value": w.tokens / s, "unit": UNIT,
           "ms_per_step": s * 1e3, "launches_per_call": 4,
           "roofline": {"bound": "alu", "achieved": flops / s / 1e12, "peak": peak,
                        "unit": "TFLOP/s", "frac": flops / s / 1e12 / peak,
                        "peak_kind": "fp32 FMA peak from unit counts and clock",
                        "traffic": profile_traffic(*_bwd_prof(w)),
                        "kernel": "linear_bwd", "kernel_ms": s * 1e3,
                        "algorithmic_flops": flops,
                        "algorithmic_bytes": w.tokens * W.bwd_bytes_per_token(w)},
           "clocks": clk.summary()}
    del d, run, dY
    torch.cuda.empty_cache()
    return rec


def _packed(parts, device=None, pinned=False):
    """One contiguous byte buffer holding the tensors `parts` (name -> (shape,
    dtype)) back to back, each at a 256-byte aligned offset; returns the buffer
    and the views."""
    import torch
    offs, o = {}, 0
    for k, (shape, dt) in parts.items():
        n = int(np.prod(shape)) * torch.empty((), dtype=dt).element_size()
        offs[k] = (o, n)
        o += (n + 255) // 256 * 256
    buf = torch.empty(o, dtype=torch.uint8, device=device)
    if pinned:
        buf = buf.pin_memory()
    views = {k: buf[a:a + n].view(parts[k][1]).view(parts[k][0]) for k, (a, n) in offs.items()}
    return buf, views


def e2e_rate(w, d, run, steps, warmup, stream, world, dev, groups=8):
    """End to end through the C ABI from pinned host buffers: every step copies
    that step's inputs host -> device and the outputs (Y and M_final) back.  The
    heads are split into `groups`; a group's inputs sit in one contiguous pinned
    region and its outputs in another, so a step is one copy each way per group.
    Each group has a copy-in, a compute and a copy-out stream and two sets of
    device buffers used on alternate steps: its next copy-in overlaps its current
    update and copy-out, and the two copy directions run at once.  Events order
    each buffer's reuse.  The timed region starts before the first copy-in and
    ends after the last copy-out.  Returns (seconds for all steps, seconds for the
    same steps with the copies alone, h2d bytes per step, d2h bytes per step)."""
    import torch
    import test_memorization_recurrent_gb300 as A
    from test_memorization_recurrent_gb300.harness import cfg_for
    per_head = ("K", "Q", "V", "alpha", "eta", "theta", "M0")
    G = max(1, min(groups, w.heads))
    bounds = [w.heads * g // G for g in range(G + 1)]

    def in_parts(lo, hi):
        p = {k: ((hi - lo,) + tuple(d[k].shape[1:]), d[k].dtype) for k in per_head}
        p["gamma"] = (tuple(d["gamma"].shape), d["gamma"].dtype)
        return p

    def out_parts(lo, hi):
        return {"Y": ((hi - lo,) + tuple(run.Y.shape[1:]), torch.float32),
                "M": ((hi - lo,) + tuple(run.M.shape[1:]), torch.float32)}

    hin, hout, din, dout = [], [], [[], []], [[], []]
    for g in range(G):
        lo, hi = bounds[g], bounds[g + 1]
        buf, views = _packed(in_parts(lo, hi), pinned=True)
        for k in per_head:
            views[k].copy_(d[k][lo:hi].cpu())
        views["gamma"].copy_(d["gamma"].cpu())
        hin.append(buf)
        hout.append(_packed(out_parts(lo, hi), pinned=True)[0])
        for par in range(2):
            din[par].append(_packed(in_parts(lo, hi), device=dev))
            dout[par].append(_packed(out_parts(lo, hi), device=dev))
    h2d = sum(b.numel() for b in hin)
    d2h = sum(b.numel() for b in hout)
    s_in = [torch.cuda.Stream(device=dev) for _ in range(G)]
    s_cp = [torch.cuda.Stream(device=dev) for _ in range(G)]
    s_out = [torch.cuda.Stream(device=dev) for _ in range(G)]
    ev = lambda: [[torch.cuda.Event() for _ in range(2)] for _ in range(G)]  # noqa: E731
    ev_in, ev_cp, ev_out = ev(), ev(), ev()
    cfgs = []
    for g in range(G):
        hg = bounds[g + 1] - bounds[g]
        nb = A.atlas_mem_workspace_bytes(cfg_for(w, hg, w.N))
        ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=dev) if nb else None
        cfgs.append((cfg_for(w, hg, w.N, workspace=ws, workspace_bytes=nb, status_dev=run.status),
                     ws))
    used = [[False, False] for _ in range(G)]

    def steps_of(n, first, compute=True):
        start = torch.cuda.Event()
        start.record(stream)
        for g in range(G):
            for s_ in (s_in[g], s_cp[g], s_out[g]):
                s_.wait_event(start)
        for step in range(n):
            par = (first + step) & 1
            for g in range(G):
                (ib, iv), (ob, ov) = din[par][g], dout[par][g]
                if used[g][par]:  # this buffer's inputs were read by its last update
                    s_in[g].wait_event(ev_cp[g][par])
                with torch.cuda.stream(s_in[g]):
                    ib.copy_(hin[g], non_blocking=True)
                ev_in[g][par].record(s_in[g])
                s_cp[g].wait_event(ev_in[g][par])
                if used[g][par]:  # the outputs of this buffer have been copied out
                    s_cp[g].wait_event(ev_out[g][par])
                if compute:
                    with torch.cuda.stream(s_cp[g]):
                        ov["M"].copy_(iv["M0"])
                    A.atlas_mem_forward(iv["K"], iv["Q"], iv["V"], iv["alpha"], iv["eta"],
                                        iv["theta"], iv["gamma"], cfgs[g][0], ov["Y"], ov["M"],
                                        s_cp[g])
                ev_cp[g][par].record(s_cp[g])
                s_out[g].wait_event(ev_cp[g][par])
                with torch.cuda.stream(s_out[g]):
                    hout[g].copy_(ob, non_blocking=True)
                ev_out[g][par].record(s_out[g])
                used[g][par] = True
        for g in range(G):
            for s_ in (s_in[g], s_cp[g], s_out[g]):
                e = torch.cuda.Event()
                e.record(s_)
                stream.wait_event(e)

    def timed(compute):
        steps_of(max(2, warmup), 0, compute)
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        steps_of(steps, max(2, warmup), compute)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return e0.elapsed_time(e1) / 1e3

    t = timed(True)
    # the same copies, streams and events with no update: the rate the host link
    # allows for this step's bytes, against which the end-to-end rate is read
    t_copy = timed(False)
    return t, t_copy, h2d, d2h


def run_atlas(args, w):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    import test_memorization_recurrent_gb300 as A
    from test_memorization_recurrent_gb300 import build as B
    from test_memorization_recurrent_gb300.harness import Runner, to_device
    B.build()

    inp = W.generate(w, seed=rank)
    d = to_device(w, inp, dev)
    run = Runner(w, w.heads, w.N, device=dev)
    path = A.atlas_mem_path(run.cfg)
    launches_per_step = A.atlas_mem_launch_count(run.cfg)
    stream = torch.cuda.current_stream()

    with Clocks(torch.cuda.current_device()) as clk:
        elapsed, kernel_s, flush = time_device(w, run, d, args.steps, args.warmup, stream, clk,
                                               world)
    elapsed_max = max_over_ranks(elapsed, world, dev)
    e2e_s, copy_s, h2d, d2h = e2e_rate(w, d, run, args.steps, args.warmup, stream, world, dev)
    e2e_s = max_over_ranks(e2e_s, world, dev)
    copy_s = max_over_ranks(copy_s, world, dev)
    if int(run.status.item()) != 0:
        raise SystemExit(f"device status {int(run.status.item())} in the end-to-end leg")

    per_config = None
    if world == 1 and not args.no_per_config and not args.tokens and args.loss == "l2":
        del d
        torch.cuda.empty_cache()
        per_config = [measure_config(wid, n, min(args.steps, 10), max(3, min(args.warmup, 3)),
                                     dev, not args.no_cpu_baseline)
                      for wid, n in PER_CONFIG if wid != w.wid]

    backward = backward_momentum = variants = None
    if world == 1 and not args.no_per_config and not args.tokens and args.loss == "l2":
        backward = measure_backward(min(args.steps, 5), 2, dev)
        backward_momentum = measure_backward(min(args.steps, 5), 2, dev, momentum=True)
        variants = [measure_config(v, None, min(args.steps, 5), 3, dev, not args.no_cpu_baseline)
                    for v in variant_workloads()]

    if rank != 0:
        return
    tokens = w.tokens
    value = aggregate(tokens, world, elapsed_max, args.steps)
    bytes_launch = tokens * W.bytes_per_token(w) + 2 * 4 * w.heads * w.state_size

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        heads, n = oracle_sample(w)
        rate, dt = oracle_rate(w, heads, n)
        cpu = {"value": rate, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{len(heads)} heads x {n} tokens of {w.name}, {dt:.1f} s"}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_max / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.bf16 else "f32", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d_k": w.d_k, "d_v": w.d_v,
                   "d_h": w.d_h, "c": w.c, "b": w.b, "path": path,
                   "l2": ("L2 flushed before every step (%.2f MB per step)" if flush else
                          "inputs larger than L2 (K,Q,V,Y %.0f MB per step)")
                         % (bytes_launch / 1e6)},
        "roofline": roofline(w, path, kernel_s),
        "cpu_baseline": cpu,
        "e2e": {"value": aggregate(tokens, world, e2e_s, args.steps), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies_only": {"value": aggregate(tokens, world, copy_s, args.steps),
                                "ms_per_step": copy_s * 1e3 / args.steps,
                                "note": "the same pinned copies with no update: the "
                                        "host-link bound of the end-to-end rate"}},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if per_config is not None:
        line["per_config"] = per_config
    if backward is not None:
        line["backward"] = backward
    if backward_momentum is not None:
        line["backward_momentum"] = backward_momentum
    if variants is not None:
        line["variants"] = variants
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def profile_one_call(args, w):
    """Warm up, then run exactly one call (the forward over the workload, or the
    backward pass) between cudaProfilerStart and cudaProfilerStop, so that
    `ncu --profile-from-start off` captures that call's kernels and nothing else."""
    import torch
    import test_memorization_recurrent_gb300 as A
    from test_memorization_recurrent_gb300 import build as B
    from test_memorization_recurrent_gb300.harness import BackwardRunner, Runner, to_device
    B.build()
    torch.cuda.set_device(0)
    d = to_device(w, W.generate(w))
    if args.profile_call == "backward":
        r = np.random.default_rng(3)
        dY = torch.from_numpy(r.standard_normal((w.heads, w.N, w.d_v)).astype(np.float32)).cuda()
        dMN = torch.zeros((w.heads, w.state_size), dtype=torch.float32, device="cuda")
        run = BackwardRunner(w, w.heads, w.N)
        call = lambda: run(d, dY, dMN)  # noqa: E731
        launches = 3
    else:
        run = Runner(w, w.heads, w.N)
        call = lambda: run(d)  # noqa: E731
        launches = A.atlas_mem_launch_count(run.cfg)
    for _ in range(max(3, args.warmup)):
        call()
    if w.tokens * W.bytes_per_token(w) + 2 * 4 * w.heads * w.state_size < 2 * L2_BYTES:
        # a workload that fits in L2 is timed after an L2 scrub: profile it cold too
        torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda").fill_(1.0)
    torch.cuda.synchronize()
    torch.cuda.profiler.start()
    call()
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    if int(run.status.item()) != 0:
        raise SystemExit(f"device status {int(run.status.item())}")
    print(json.dumps({"profiled": args.profile_call, "workload": w.name, "tokens": w.tokens,
                      "launches": launches}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", type=int, default=2, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--impl", default="atlas", choices=["atlas", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-call", choices=["forward", "backward"], default=None,
                    help="warm up, then run one call between cudaProfilerStart/Stop and exit "
                         "(for ncu --profile-from-start off)")
    ap.add_argument("--variant", type=int, default=None,
                    help="with --profile-call: the variant workload of that index")
    ap.add_argument("--no-per-config", action="store_true",
                    help="measure the chosen workload only (no per_config record)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="run only the first TOKENS tokens of every head (0 = the whole workload)")
    ap.add_argument("--loss", default="l2", choices=["l2", "lp", "huber"],
                    help="attentional bias: l2 (the workloads'), or the Miras l_p / Huber variants")
    ap.add_argument("--loss-param", type=float, default=0.0,
                    help="p of the l_p bias (default 3), delta of the Huber bias (default 0.3)")
    ap.add_argument("--momentum", action="store_true",
                    help="with --profile-call backward: momentum in the forward, eta ~ U(0.5, 0.9)")
    args = ap.parse_args(argv)
    w = W.workload(args.workload, bounded=True)
    if args.momentum:
        w = w.with_(eta=(0.5, 0.9), name="linear-momentum-b64-bf16")
    if args.tokens:
        w = w.with_(N=min(args.tokens, w.N))
    if args.loss != "l2":
        kind = W.LOSS_LP if args.loss == "lp" else W.LOSS_HUBER
        prm = args.loss_param or (3.0 if args.loss == "lp" else 0.3)
        w = w.with_(loss=kind, loss_param=prm, name=f"{w.name}-{args.loss}{prm:g}")
    if args.profile_call:
        if args.variant is not None:
            w = variant_workloads()[args.variant]
        profile_one_call(args, w)
    elif args.impl == "reference":
        run_reference(args, w)
    else:
        run_atlas(args, w)


if __name__ == "__main__":
    main()
