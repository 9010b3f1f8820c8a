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


def profile_traffic(kernel_src: str, profile_name: str, units_per_launch: float):
    """DRAM bytes per launch from a committed ncu summary, scaled to this launch,
    or None if the summary is missing or was taken on another kernel source."""
    path = os.path.join(ROOT, "profiles", profile_name)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m_b = re.search(r"dram_bytes_per_unit:\s*([0-9.eE+-]+)", text)
    if not m_sha or not m_b:
        return None
    with open(kernel_src, "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != m_sha.group(1):
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
                          w.ns_steps, a, b_, c_, w.ns_eps, loss_param=w.loss_param)
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
        return list(range(min(w.heads, cores))), 512
    if w.wid == 4:
        return list(range(min(w.heads, cores))), 2048
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

KERNEL_OF_PATH = {
    "linear_tc": ("linear_tc.cu", "linear_tc_{wname}.md"),
    "linear_simt": ("linear_simt.cu", "linear_simt_{wname}.md"),
    "linear_seq": ("linear_seq.cu", "linear_seq_{wname}.md"),
    "linear_chunk": ("tc_gemm.cu", "linear_chunk_{wname}.md"),
    "mlp_simt": ("mlp_simt.cu", "mlp_simt_{wname}.md"),
    "mlp_tc": ("mlp_tc.cu", "mlp_tc_{wname}.md"),
}


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

    # -- device-resident timing.  A step whose data fits in L2 is preceded by a
    # write of a buffer twice the L2 size, outside its events, and the step
    # time is the sum of the per-step events; otherwise the steps run back to
    # back and the step time is the whole loop's.
    bytes_launch = w.tokens * W.bytes_per_token(w) + 2 * 4 * w.heads * w.state_size
    flush = bytes_launch < 2 * L2_BYTES
    scrub = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    s_start = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    s_end = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    k_start = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    k_end = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with Clocks(torch.cuda.current_device()) as clk:
        for _ in range(args.warmup):
            run(d)
        torch.cuda.synchronize()
        clk.wait_ready()
        barrier(world)
        torch.cuda.synchronize()
        clk.mark_start()
        t_start.record(stream)
        for i in range(args.steps):
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
        clk.mark_end()
        barrier(world)
    if flush:
        elapsed = sum(a.elapsed_time(b) for a, b in zip(s_start, s_end)) / 1e3
    else:
        elapsed = t_start.elapsed_time(t_end) / 1e3
    kernel_s = sum(a.elapsed_time(b) for a, b in zip(k_start, k_end)) / 1e3 / args.steps
    elapsed_max = max_over_ranks(elapsed, world, dev)
    status = int(run.status.item())
    if status != 0:
        raise SystemExit(f"device status {status}: {A.atlas_mem_strerror(status)}")

    # -- end to end through the C ABI with host buffers (pinned), copies timed
    host = {k: v.cpu().pin_memory() for k, v in d.items()}
    Yh = torch.empty(run.Y.shape, dtype=torch.float32).pin_memory()
    Mh = torch.empty(run.M.shape, dtype=torch.float32).pin_memory()
    dd = {k: torch.empty_like(v) for k, v in d.items()}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = Yh.numel() * 4 + Mh.numel() * 4

    def e2e_step():
        for k in host:
            dd[k].copy_(host[k], non_blocking=True)
        run.M.copy_(dd["M0"])
        A.atlas_mem_forward(dd["K"], dd["Q"], dd["V"], dd["alpha"], dd["eta"], dd["theta"],
                            dd["gamma"], run.cfg, run.Y, run.M, stream)
        Yh.copy_(run.Y, non_blocking=True)
        Mh.copy_(run.M, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_s = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev)

    if rank != 0:
        return
    tokens = w.tokens
    value = aggregate(tokens, world, elapsed_max, args.steps)
    hbm, tf, tf_sus, peak_kind = load_peaks()
    flops_launch = tokens * W.flop_per_token(w)
    ai = flops_launch / bytes_launch
    ridge = tf * 1e12 / (hbm * 1e9)
    src, prof = KERNEL_OF_PATH.get(path, ("", ""))
    src_path = os.path.join(ROOT, "test_memorization_recurrent_gb300", "csrc", src)
    prof_name = prof.format(wname=w.name)
    if ai < ridge:
        achieved = bytes_launch / kernel_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "peak_kind": f"{peak_kind} hbm_gbs"}
        units = tokens
    else:
        achieved = flops_launch / kernel_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tf_sus, "unit": "TFLOP/s",
                "frac": achieved / tf_sus, "peak_kind": f"{peak_kind} bf16_tflops_sustained"}
        units = tokens
    roof["traffic"] = profile_traffic(src_path, prof_name, units) if src else None
    roof["kernel"] = path
    roof["kernel_ms"] = kernel_s * 1e3
    roof["algorithmic_bytes"] = bytes_launch
    roof["algorithmic_flops"] = flops_launch

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
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": aggregate(tokens, world, e2e_s, args.steps), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", type=int, default=2, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--impl", default="atlas", choices=["atlas", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=0,
                    help="run only the first TOKENS tokens of every head (0 = the whole workload)")
    ap.add_argument("--loss", default="l2", choices=["l2", "lp", "huber"],
                    help="attentional bias: l2 (the workloads'), or the Miras l_p / Huber variants")
    ap.add_argument("--loss-param", type=float, default=0.0,
                    help="p of the l_p bias (default 3), delta of the Huber bias (default 0.3)")
    args = ap.parse_args(argv)
    w = W.workload(args.workload, bounded=True)
    if args.tokens:
        w = w.with_(N=min(args.tokens, w.N))
    if args.loss != "l2":
        kind = W.LOSS_LP if args.loss == "lp" else W.LOSS_HUBER
        prm = args.loss_param or (3.0 if args.loss == "lp" else 0.3)
        w = w.with_(loss=kind, loss_param=prm, name=f"{w.name}-{args.loss}{prm:g}")
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_atlas(args, w)


if __name__ == "__main__":
    main()
