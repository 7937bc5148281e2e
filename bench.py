"""Benchmark: 8B-class decode weight sweep at batch 1 (one step = one token).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mine|reference]

A step multiplies each of the 253 packed 1-bit matrices of an 8B-class decoder
(36 layers x {q, k, v, o, gate, up, down} + the 1-bit LM head; 1,064,263,680
weight bytes at 1.125 bits/weight) by its own bf16 activation vector, as one
grouped persistent launch (bit1_gemv_group).  The same 253 products run as a
chain of dependent launches are reported beside it ("decode_chain").  The
weights (1.06 GB) exceed the 126 MB L2, so every step streams them from HBM.
Rank 0 prints one JSON line.

--impl reference times the CPU oracle (scalar fp64, test infrastructure) on a
bounded row sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "1-bit GEMV effective weight GB/s & % of HBM peak; 8B-class decode tok/s-equiv"
WORKLOAD = "8B-class decode weight sweep, batch 1: 36 x {q,k,v,o 4096/1024x4096, gate/up 12288x4096, down 4096x12288} + LM head 151936x4096 (253 GEMVs, 1,064,263,680 weight bytes)"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """Samples SM clocks and throttle reasons while the benchmark runs: through
    NVML when the Python binding is importable, else by polling nvidia-smi."""

    REASONS = {
        "gpu_idle": 0x1, "applications_clocks_setting": 0x2, "sw_power_cap": 0x4,
        "hw_slowdown": 0x8, "sync_boost": 0x10, "sw_thermal_slowdown": 0x20,
        "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80,
        "display_clock_setting": 0x100,
    }

    def __init__(self, index: int, period_s: float = 0.005):
        self.index, self.period = index, period_s
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self._stop = threading.Event()
        self._t = None
        self.proc = None
        self.mode = None
        self.err = None
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = pynvml.nvmlDeviceGetHandleByIndex(index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.mode = "nvml"
        except Exception as e:
            self.err = f"{type(e).__name__}: {e}"
            self.mode = "nvidia-smi"

    def _run_nvml(self):
        nv = self.nv
        while not self._stop.is_set():
            try:
                self.samples.append(nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM))
                r = nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
                for k, bit in self.REASONS.items():
                    if r & bit:
                        self.reasons.add(k)
            except Exception:
                pass
            time.sleep(self.period)

    def __enter__(self):
        if self.mode == "nvml":
            self._t = threading.Thread(target=self._run_nvml, daemon=True)
            self._t.start()
        else:
            import subprocess
            q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active")
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                     "--format=csv,noheader,nounits", "-lms", "20"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                time.sleep(0.3)   # let the poller start before the timed region
            except Exception as e:
                self.err = f"{type(e).__name__}: {e}"
                self.proc = None
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._t:
            self._t.join()
        if self.proc:
            time.sleep(0.1)
            self.proc.terminate()
            out, _ = self.proc.communicate()
            for line in out.splitlines():
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 3:
                    continue
                try:
                    self.samples.append(float(parts[0]))
                    self.max_mhz = float(parts[1])
                    r = int(parts[2], 16)
                    for k, bit in self.REASONS.items():
                        if r & bit:
                            self.reasons.add(k)
                except ValueError:
                    pass

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz,
                    "reasons": [f"no clock samples ({self.mode}; {self.err})"]}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "samples": len(self.samples), "source": self.mode,
                "window": "from just before to just after the timed region",
                "reasons": sorted(self.reasons - {"gpu_idle"})}


def _traffic_for(kernel_src: str):
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu
    summary, or None when the kernel source changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        h = hashlib.sha256(open(kernel_src, "rb").read()).hexdigest()[:16]
        if d.get("kernel_src_sha256_16") != h:
            return None
        return d.get("dram_bytes_per_launch_sweep_avg")
    except Exception:
        return None


def oracle_sample(frac_den: int):
    """The first 1/frac_den rows of every matrix of the sweep (seeded, host)."""
    import numpy as np
    from bit_weight_gemv_sign_b300 import synth
    out = []
    for i, m in enumerate(synth.sweep_8b()):
        n = max(1, m.N // frac_den)
        bits, scales = synth.matrix(m.N, m.K, i)
        x = synth.x_for(1, m.K, i)
        out.append((np.ascontiguousarray(bits[:n]), np.ascontiguousarray(scales[:n]), x, n, m.K))
    return out


def time_oracle(sample, threads: int):
    """Run the oracle (as it stands) over the sample, rows spread over POSIX
    threads; returns (weight bytes, seconds)."""
    import oracle
    wbytes, secs = 0, 0.0
    for b, s, x, n, K in sample:
        t0 = time.perf_counter()
        oracle.gemv_threads(b, s, x, 1, n, K, threads)
        secs += time.perf_counter() - t0
        wbytes += n * K // 8 + 2 * n * (K // 128)
    return wbytes, secs


def cpu_baseline(frac_den: int = 8):
    threads = os.cpu_count() or 1
    sample = oracle_sample(frac_den)
    wbytes, secs = time_oracle(sample, threads)
    return {"value": wbytes / secs / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "seconds": secs, "sample": f"first 1/{frac_den} of the rows of each of the 253 sweep "
                                        f"matrices ({wbytes} weight bytes), scalar fp64 oracle, "
                                        f"{threads} threads"}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    frac = 256
    threads = os.cpu_count() or 1
    sample = oracle_sample(frac)
    for _ in range(args.warmup):
        time_oracle(sample, threads)
    wb, secs = 0, 0.0
    for _ in range(args.steps):
        b, t = time_oracle(sample, threads)
        wb += b
        secs += t
    v = wb / secs / 1e9
    desc = (f"each step: first 1/{frac} of the rows of each of the 253 sweep matrices "
            f"({wb // max(1, args.steps)} weight bytes), scalar fp64 oracle, {threads} threads")
    out = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": 1,
           "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": 1064263680 / (v * 1e9) * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": WORKLOAD, "batch": 1, "sample": desc},
           "tok_s_equiv": v * 1e9 / 1064263680,
           "cpu_baseline": {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle",
                            "sample": desc},
           "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))
    return 0


def run_mine(args):
    import torch
    import bit_weight_gemv_sign_b300 as b1
    from bit_weight_gemv_sign_b300 import synth
    from bit_weight_gemv_sign_b300.sweep import Sweep

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    b1.load()

    sw = Sweep(synth.sweep_8b(), seed0=0, batch=1, y_dtype=b1.BF16).fill()
    plan = sw.group_plan()          # one persistent launch over all 253 GEMVs
    s = torch.cuda.Stream()

    def barrier():
        if dist:
            dist.barrier()
        torch.cuda.synchronize()

    def step():
        plan.run(stream=s)

    with torch.cuda.stream(s):
        for _ in range(max(3, args.warmup)):
            step()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk, torch.cuda.stream(s):
        e0.record(s)
        for _ in range(args.steps):
            step()
        e1.record(s)
        e1.synchronize()
    barrier()
    ms = e0.elapsed_time(e1)
    if dist:
        t = torch.tensor([ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    ms_step = ms / args.steps
    gbs = ws * sw.weight_bytes / (ms_step * 1e-3) / 1e9
    timeouts = b1.bit1_device_wait_timeouts()

    # end to end through the public API with host buffers, pipelined as a
    # server would run it: two I/O slots over the same resident weights; every
    # step copies its inputs (all 253 activation vectors) from pinned host
    # memory and reads its result (the LM-head logits) back to pinned host
    # memory; step i+1's upload and step i's download overlap step i's compute.
    xs = [sw.x, torch.empty_like(sw.x)]
    ys = [sw.y, torch.empty_like(sw.y)]
    plans = [plan, sw.group_plan(xs[1], ys[1])]
    hx = torch.empty_like(sw.x, device="cpu").pin_memory()
    hx.copy_(sw.x.cpu())
    ylast = [sw.y_of(len(sw.mats) - 1, yb) for yb in ys]
    hy = [torch.empty(ylast[0].shape, dtype=ylast[0].dtype, device="cpu").pin_memory() for _ in range(2)]
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    up_done, comp_done = [ev(), ev()], [ev(), ev()]

    def e2e_steps(n):
        for i in range(n):
            k = i & 1
            up.wait_event(comp_done[k]) if i >= 2 else None
            with torch.cuda.stream(up):
                xs[k].copy_(hx, non_blocking=True)
                up_done[k].record(up)
            s.wait_event(up_done[k])
            plans[k].run(stream=s)
            comp_done[k].record(s)
            down.wait_event(comp_done[k])
            with torch.cuda.stream(down):
                hy[k].copy_(ylast[k], non_blocking=True)

    e2e_steps(4)
    torch.cuda.synchronize()
    barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(up)
    e2e_steps(args.steps)
    down.wait_stream(s)
    down.wait_stream(up)
    f1.record(down)
    f1.synchronize()
    e2e_ms = f0.elapsed_time(f1) / args.steps
    e2e_gbs = ws * sw.weight_bytes / (e2e_ms * 1e-3) / 1e9
    hy = hy[0]

    # secondary: the same 253 products as a dependent chain of separate
    # launches (CUDA graph, programmatic dependent launch; each kernel waits
    # for its predecessor before reading x, as in a real decode step)
    sw.capture(pdl=True)
    chain_steps = min(args.steps, 50)
    with torch.cuda.stream(sw.stream):
        for _ in range(3):
            sw.replay()
        sw.stream.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(sw.stream)
        for _ in range(chain_steps):
            sw.replay()
        c1.record(sw.stream)
        c1.synchronize()
    chain_ms = c0.elapsed_time(c1) / chain_steps

    hbm, src = _peaks()
    grp_src = os.path.join(ROOT, "bit_weight_gemv_sign_b300", "csrc", "gemv_group.cu")
    traffic = _traffic_for(grp_src)
    out = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": 1, "weight_bytes_per_step": sw.weight_bytes,
                   "l2": "inputs larger than L2 (1.06 GB of weights per step vs 126 MB L2)",
                   "compute": "1-bit sign weights x bf16 activations, fp32 accumulation, bf16 output",
                   "launch": "one grouped persistent launch of the 253 independent GEMVs per step",
                   "parallelism": "replicas" if ws > 1 else "single GPU"},
        "tok_s_equiv": 1e3 / ms_step,
        "hbm_frac": gbs / ws / hbm,
        "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": gbs / ws, "peak": hbm, "unit": "GB/s",
                     "frac": gbs / ws / hbm, "peak_source": src, "traffic": traffic,
                     "kernel": "k_gemv_group (one launch per step)"},
        "e2e": {"value": e2e_gbs, "unit": "GB/s", "h2d_bytes_per_step": sw.x_bytes,
                "d2h_bytes_per_step": hy.numel() * hy.element_size(), "ms_per_step": e2e_ms,
                "how": "pinned host x -> device, grouped launch, logits -> pinned host every step; "
                       "two I/O slots so step i+1's upload overlaps step i's compute"},
        "decode_chain": {"value": sw.weight_bytes / (chain_ms * 1e-3) / 1e9, "unit": "GB/s",
                         "ms_per_step": chain_ms, "tok_s_equiv": 1e3 / chain_ms,
                         "launches_per_step": sw.launches_per_step(),
                         "what": "253 dependent launches (graph + PDL, each waits before reading x)"},
        "device_wait_timeouts": timeouts,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        out["cpu_baseline"] = cpu_baseline(frac_den=8)
    if rank == 0:
        print(json.dumps(out))
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_mine(args)


if __name__ == "__main__":
    sys.exit(main())
