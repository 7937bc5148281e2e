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


def max_over_ranks(value: float, dist=None, device="cpu") -> float:
    """The largest of every rank's ``value`` (the step time a multi-GPU run
    reports: the slowest replica); the value itself without a process group."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


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
                **({"nvml_error": self.err} if self.mode != "nvml" and self.err else {}),
                "window": "from just before to just after the timed region",
                "reasons": sorted(self.reasons - {"gpu_idle"})}


# Every source the grouped kernel compiles from: a change to any of them
# invalidates the committed DRAM counters.
GROUP_KERNEL_SOURCES = ("bit_weight_gemv_sign_b300/csrc/gemv_group.cu",
                        "bit_weight_gemv_sign_b300/csrc/t6_common.cuh",
                        "bit_weight_gemv_sign_b300/csrc/common.cuh",
                        "bit_weight_gemv_sign_b300/csrc/internal.h",
                        "include/bit1.h")


def _code_only(text: str) -> str:
    """C/C++ source without comments and blank-line or trailing-space noise:
    a comment edit leaves the compiled kernel, and so its counters, unchanged."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_sources_hash(paths=GROUP_KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    for rel in paths:
        h.update(rel.encode())
        h.update(_code_only(open(os.path.join(ROOT, rel), encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def _traffic_for():
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu
    summary, or None when any of its sources changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        if d.get("kernel_sources_sha256_16") != kernel_sources_hash():
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


def cpu_baseline(frac_den: int = 1):
    threads = os.cpu_count() or 1
    sample = oracle_sample(frac_den)
    wbytes, secs = time_oracle(sample, threads)
    what = ("all rows of the 253 sweep matrices (one full decode step" if frac_den == 1 else
            f"first 1/{frac_den} of the rows of each of the 253 sweep matrices (")
    # the same oracle on one core over the first 1/256 of each matrix's rows,
    # best of three (the host cores are shared)
    import numpy as np
    sub = [(np.ascontiguousarray(b[:max(1, n // 256)]), np.ascontiguousarray(sc[:max(1, n // 256)]), x,
            max(1, n // 256), K) for b, sc, x, n, K in sample]
    runs = [time_oracle(sub, 1) for _ in range(3)]
    wb1, secs1 = runs[0][0], min(r[1] for r in runs)
    return {"value": wbytes / secs / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "seconds": secs, "tok_s_equiv": wbytes / secs / 1064263680,
            "sample": f"{what}, {wbytes} weight bytes), scalar fp64 oracle, {threads} threads",
            "single_thread": {"value": wb1 / secs1 / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": f"first 1/256 of the rows of each sweep matrix ({wb1} weight bytes), "
                                        "best of three"}}


def _timed(fn):
    t0 = time.perf_counter()
    fn()
    return time.perf_counter() - t0


def oracle_beside_extras(extras: dict) -> None:
    """The CPU oracle, as it stands, timed beside each extra row on a bounded
    sample of that row's workload (a few seconds in all); added to each row
    as "cpu_oracle".  Binary products use the oracle's row-threaded loop on
    all host cores, the ternary ones its single-threaded loops."""
    import numpy as np
    import oracle
    from bit_weight_gemv_sign_b300 import synth
    threads = os.cpu_count() or 1

    def binary(N, K, B, rows, seed):
        bits, scales = synth.matrix(N, K, seed)
        x = synth.x_for(B, K, seed)
        b, sc = np.ascontiguousarray(bits[:rows]), np.ascontiguousarray(scales[:rows])
        secs = _timed(lambda: oracle.gemv_threads(b, sc, x, B, rows, K, threads))
        return secs * N / rows            # seconds for the whole matrix

    def entry(value, unit, sample, thr):
        return {"value": value, "unit": unit, "cores": thr, "kind": "oracle", "sample": sample}

    if "c1_tiny" in extras:
        secs = binary(256, 1024, 1, 256, 0)
        extras["c1_tiny"]["cpu_oracle"] = entry(secs * 1e6, "us per GEMV", "the whole 256x1024 product", threads)
    if "c2_projections_b1" in extras:
        secs = binary(12288, 4096, 1, 768, 1)
        wb = 12288 * 4096 // 8 + 2 * 12288 * 32
        extras["c2_projections_b1"]["cpu_oracle"] = entry(wb / secs / 1e9, "GB/s",
                                                          "768 of the 12288 rows of an up/gate projection", threads)
    if "c4_mlp_crossover" in extras:
        out = {}
        for B in (16, 64):
            secs = binary(12288, 4096, B, 96, 2)
            out[f"B{B}_us_per_call"] = secs * 1e6
            out[f"B{B}_tflops"] = 2.0 * B * 12288 * 4096 / secs / 1e12
        extras["c4_mlp_crossover"]["cpu_oracle"] = {**entry(out["B16_us_per_call"], "us per call at B = 16",
                                                            "96 of the 12288 rows of up/gate at B = 16 and 64",
                                                            threads), **out}
    if "pp512_tcgen05" in extras:
        secs = binary(12288, 4096, 512, 8, 3)
        extras["pp512_tcgen05"]["cpu_oracle"] = entry(2.0 * 512 * 12288 * 4096 / secs / 1e12, "TFLOP/s",
                                                      "8 of the 12288 rows at B = 512", threads)
    if "c5_sweep_27b" in extras:
        wb = secs = 0.0
        for i, m in enumerate(synth.sweep_27b()[:7]):          # one layer's seven matrices
            rows = max(1, m.N // 64)
            secs += binary(m.N, m.K, 1, rows, 100 + i) * rows / m.N
            wb += rows * (m.K // 8 + 2 * (m.K // 128))
        extras["c5_sweep_27b"]["cpu_oracle"] = entry(wb / secs / 1e9, "GB/s",
                                                     "1/64 of the rows of one 27B-class layer's seven matrices",
                                                     threads)
    if "verify_sweep_8b_b5" in extras:
        wb = secs = 0.0
        for i, m in enumerate(synth.sweep_8b()[:7]):
            rows = max(1, m.N // 64)
            secs += binary(m.N, m.K, 5, rows, 200 + i) * rows / m.N
            wb += rows * (m.K // 8 + 2 * (m.K // 128))
        extras["verify_sweep_8b_b5"]["cpu_oracle"] = entry(wb / secs / 1e9, "GB/s (5 rows per weight read)",
                                                           "1/64 of the rows of one 8B-class layer at B = 5",
                                                           threads)
    if "fused_mlp_sweep_8b" in extras:
        N2, K, rows = 24576, 4096, 192
        bits, scales = synth.matrix(rows, K, 7)
        x = synth.x_for(1, K, 7)
        secs = _timed(lambda: oracle.gemv_swiglu(bits, scales, x, 1, rows, K))
        wb = rows * (K // 8 + 2 * (K // 128))
        extras["fused_mlp_sweep_8b"]["cpu_oracle"] = entry(wb / secs / 1e9, "GB/s",
                                                           "192 rows (96 gate/up pairs) x 4096 with SwiGLU", 1)
    if "ternary_sweep_8b" in extras:
        N, K, rows = 12288, 4096, 96
        a, b, scales = synth.ternary_matrix(rows, K, 4)
        x = synth.x_for(1, K, 4)
        secs = _timed(lambda: oracle.gemv_ternary(a, b, scales, x, 1, rows, K))
        wb = rows * (2 * K // 8 + 2 * (K // 128))
        extras["ternary_sweep_8b"]["cpu_oracle"] = entry(wb / secs / 1e9, "GB/s",
                                                         "96 rows of a 12288x4096 ternary matrix, 2-bit slots", 1)
    if "ternary_t5" in extras:
        K, rows = 4096, 96
        t = synth.ternary_codes(rows, K, synth.rng(5))
        packed = oracle.t5_pack(t, rows, K)
        scales = synth.group_scales(rows, K, synth.rng(6))
        x = synth.x_for(1, K, 5)
        secs = _timed(lambda: oracle.gemv_t5(packed, scales, x, 1, rows, K))
        wb = rows * (26 * K // 128 + 2 * (K // 128))
        extras["ternary_t5"]["cpu_oracle"] = entry(wb / secs / 1e9, "GB/s",
                                                   "96 rows x 4096, five codes per byte", 1)


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
    # ms_per_step is the wall time of the sampled step that ran; the time the
    # oracle would take for the whole sweep is reported under its own key.
    out = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": 1,
           "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": secs / max(1, args.steps) * 1e3,
           "full_sweep_ms_extrapolated": 1064263680 / (v * 1e9) * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": WORKLOAD, "batch": 1, "sample": desc},
           "tok_s_equiv": v * 1e9 / 1064263680,
           "cpu_baseline": {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle",
                            "sample": desc},
           "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))
    return 0


# ---------------------------------------------------------------- extras
# The other configurations of the workload family, measured on the same GPU
# after the headline: each shape timed as a CUDA-graph replay of REPS calls
# that rotate over enough distinct weight copies to exceed 3x the L2, so every
# call streams its weights from HBM.

L2_BYTES = 126 * 2**20
NOMINAL_HBM_GBS = 7700.0    # B300 HBM3e, nominal


def _weight_bytes(N, K):
    return N * K // 8 + 2 * N * (K // 128)


def _time_calls(torch, b1, N, K, B, variant, reps=30, ws_bytes=None, flags=0):
    """Microseconds per bit1_gemv_ex call (graph replay, L2 rotated), or None
    when the variant does not take the shape.  ``flags`` adds to FLAG_PDL
    (FLAG_SWIGLU: y is [B, N/2])."""
    if b1.bit1_gemv_launches(B, N, K, variant) == 0:
        return None
    wb = _weight_bytes(N, K)
    copies = max(2, (3 * L2_BYTES) // wb + 1)
    g = torch.Generator(device="cuda")
    g.manual_seed(N * 131 + K * 7 + B)
    bits = torch.randint(0, 256, (copies, N, K // 8), dtype=torch.uint8, device="cuda", generator=g)
    sc = (torch.randn((copies, N, K // 128), device="cuda", generator=g).abs_() * 0.02).half().view(torch.int16)
    x = torch.randn((B, K), device="cuda", generator=g).bfloat16()
    y = torch.empty((B, N // 2 if flags & b1.FLAG_SWIGLU else N), device="cuda")
    if ws_bytes is None:
        ws_bytes = b1.bit1_gemv_workspace_bytes(max(B, 16), N, K) if variant == b1.TC else 0
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for i in range(3):
            b1.bit1_gemv_ex(bits[i % copies], sc[i % copies], x, y=y, workspace=ws, variant=variant,
                            flags=b1.FLAG_PDL | flags, stream=s)
        s.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            for i in range(reps):
                b1.bit1_gemv_ex(bits[i % copies], sc[i % copies], x, y=y, workspace=ws, variant=variant,
                                flags=b1.FLAG_PDL | flags, stream=s)
        graph.replay()
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        graph.replay()
        e1.record(s)
        e1.synchronize()
    us = e0.elapsed_time(e1) / reps * 1e3
    del bits, sc, graph
    torch.cuda.empty_cache()
    return us


def _shape_entry(N, K, B, us):
    if us is None:
        return None
    return {"us": round(us, 3), "weight_gbs": round(_weight_bytes(N, K) / (us * 1e-6) / 1e9, 1),
            "tflops": round(2.0 * B * N * K / (us * 1e-6) / 1e12, 2)}


def extra_c1_tiny(torch, b1):
    """Tiny 256x1024 batch-1 GEMV and an 8-row XOR patch applied and removed."""
    from bit_weight_gemv_sign_b300 import synth
    N, K = synth.TINY.N, synth.TINY.K
    us = _time_calls(torch, b1, N, K, 1, b1.AUTO, reps=50)
    bits = torch.randint(0, 256, (N, K // 8), dtype=torch.uint8, device="cuda")
    rows = [int(r) for r in synth.distinct_rows(N, 8, 0)]
    b1.bit1_xor_patch(bits, rows)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(50):
        b1.bit1_xor_patch(bits, rows)
    e1.record()
    e1.synchronize()
    return {"shape": [N, K], "gemv": _shape_entry(N, K, 1, us),
            "xor_patch_8_rows_us": round(e0.elapsed_time(e1) / 50 * 1e3, 3),
            "note": "latency-bound sizes (36 KB of weights); reported, not a roofline case"}


def extra_c2_projections(torch, b1):
    from bit_weight_gemv_sign_b300 import synth
    out = {}
    for m in synth.PROJ_8B:
        out[m.name] = {"shape": [m.N, m.K]}
        for name, v in (("lut6", b1.LUT6), ("lut", b1.LUT), ("stream", b1.STREAM)):
            out[m.name][name] = _shape_entry(m.N, m.K, 1, _time_calls(torch, b1, m.N, m.K, 1, v))
    out["note"] = ("one bit1_gemv_ex call per projection, graph replay with PDL, L2 rotated; a 0.6-7 MB "
                   "matrix is 0.1-1.1 us of HBM time, so a single call is bound by launch and ramp latency")
    return out


def extra_c4_crossover(torch, b1):
    """CUDA-core path (6-bit tables, up to 8 batch rows per launch) vs the
    tcgen05 path on the 8B MLP shapes, with the register-MMA variant (no
    workspace) beside them."""
    out = {}
    for N, K, name in ((12288, 4096, "up_gate"), (4096, 12288, "down")):
        rows = {}
        cross = None
        for B in (1, 4, 16, 32, 64):
            cc = _time_calls(torch, b1, N, K, B, b1.LUT6)
            tc = _time_calls(torch, b1, N, K, B, b1.TC)
            mma = _time_calls(torch, b1, N, K, B, b1.MMA)
            rows[str(B)] = {"cuda_core": _shape_entry(N, K, B, cc), "tcgen05": _shape_entry(N, K, B, tc),
                            "mma_no_workspace": _shape_entry(N, K, B, mma)}
            if cross is None and cc is not None and tc is not None and tc < cc:
                cross = B
        out[name] = {"shape": [N, K], "by_batch": rows, "tcgen05_faster_from_batch": cross}
    return out


def extra_pp512(torch, b1):
    """Prompt processing: a 512-row batch through the tensor-core path on the
    8B up/gate shape (eight 64-row launches per call)."""
    N, K, B = 12288, 4096, 512
    us = _time_calls(torch, b1, N, K, B, b1.TC, reps=10, ws_bytes=b1.bit1_gemv_workspace_bytes(B, N, K))
    e = _shape_entry(N, K, B, us)
    # gate and up as one interleaved 24576-row matrix, with and without the
    # SwiGLU epilogue
    N2 = 2 * N
    ws2 = b1.bit1_gemv_workspace_bytes(B, N2, K)
    us_p = _time_calls(torch, b1, N2, K, B, b1.TC, reps=10, ws_bytes=ws2)
    us_s = _time_calls(torch, b1, N2, K, B, b1.TC, reps=10, ws_bytes=ws2, flags=b1.FLAG_SWIGLU)
    return {"shape": [N, K], "batch": B, **e,
            "gate_up_24576x4096": {"plain": _shape_entry(N2, K, B, us_p), "swiglu": _shape_entry(N2, K, B, us_s)}}


def extra_c5_sweep_27b(torch, b1, steps=20):
    """27B-class sweep (448 matrices, 2.97 GB) as one grouped launch per step,
    and the 100-entry patch applied and removed (timed on the host clock)."""
    from bit_weight_gemv_sign_b300 import synth
    from bit_weight_gemv_sign_b300.sweep import Sweep
    sw = Sweep(synth.sweep_27b(), seed0=0, batch=1, y_dtype=b1.BF16).fill_device(27)
    plan = sw.group_plan()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            plan.run(stream=s)
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(steps):
            plan.run(stream=s)
        e1.record(s)
        e1.synchronize()
    ms = e0.elapsed_time(e1) / steps
    entries = synth.patch_entries_27b(100, 0)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    sw.apply_patch(entries)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    sw.apply_patch(entries)
    torch.cuda.synchronize()
    t2 = time.perf_counter()
    hbm, _ = _peaks()
    gbs = sw.weight_bytes / (ms * 1e-3) / 1e9
    out = {"weight_bytes": sw.weight_bytes, "ms_per_step": ms, "weight_gbs": gbs, "hbm_frac": gbs / hbm,
           "tok_s_equiv": 1e3 / ms, "patch_entries": len(entries),
           "patch_apply_ms": (t1 - t0) * 1e3, "patch_remove_ms": (t2 - t1) * 1e3,
           "note": "one grouped launch per step; patch parity and bit-identical restore are "
                   "checked in tests/test_gpu_sweeps.py"}
    del sw, plan
    torch.cuda.empty_cache()
    return out


def extra_ternary_sweep_8b(torch, b1, steps=20):
    """Ternary 8B-class sweep in 2-bit slots (two sign planes per matrix,
    2.1 GB with the scales): one grouped launch over both planes of all 253
    matrices plus one combine launch per step."""
    from bit_weight_gemv_sign_b300 import synth
    from bit_weight_gemv_sign_b300.sweep import TernarySweep
    sw = TernarySweep(synth.sweep_8b(), seed0=0, y_dtype=b1.BF16).fill_device(38)
    plan = sw.group_plan()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            plan.run(stream=s)
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(steps):
            plan.run(stream=s)
        e1.record(s)
        e1.synchronize()
    ms = e0.elapsed_time(e1) / steps
    hbm, _ = _peaks()
    gbs = sw.weight_bytes / (ms * 1e-3) / 1e9
    params = sum(m.N * m.K for m in sw.mats)
    out = {"weight_bytes": sw.weight_bytes, "bits_per_weight": 8.0 * sw.weight_bytes / params,
           "ms_per_step": ms, "weight_gbs": gbs, "hbm_frac": gbs / hbm, "tok_s_equiv": 1e3 / ms,
           "launches_per_step": sw.launches_per_step(),
           "note": "algorithmic bytes count the shared scales once; the two binary passes read "
                   "them twice (2.25 bits/weight of traffic)"}
    del sw, plan
    torch.cuda.empty_cache()
    return out


def extra_t5(torch, b1, reps=20):
    """Ternary codes packed five per byte (1.75 bits/weight): the direct
    product on the 8B-class projection shapes at batch 1 (graph replay over
    copies rotated past L2), beside the same shapes in 2-bit slots through
    bit1_gemv_ternary, and the device transcode to the 2-bit-slot planes on the
    LM-head shape."""
    out = {}
    for (N, K) in ((4096, 4096), (12288, 4096), (4096, 12288)):
        pb = N * (K // 128) * 26
        wb = pb + 2 * N * (K // 128)
        copies = max(2, (3 * L2_BYTES) // wb + 1)
        g = torch.Generator(device="cuda")
        g.manual_seed(N + K)
        packed = torch.randint(0, 243, (copies, N, (K // 128) * 26), dtype=torch.uint8, device="cuda", generator=g)
        sc = (torch.randn((copies, N, K // 128), device="cuda", generator=g).abs_() * 0.02).half().view(torch.int16)
        x = torch.randn((1, K), device="cuda", generator=g).bfloat16()
        y = torch.empty((1, N), device="cuda")
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            for i in range(3):
                b1.bit1_gemv_t5(packed[i % copies], sc[i % copies], x, y=y, stream=s, N=N)
            s.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=s):
                for i in range(reps):
                    b1.bit1_gemv_t5(packed[i % copies], sc[i % copies], x, y=y, stream=s, N=N)
            graph.replay()
            s.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            graph.replay()
            e1.record(s)
            e1.synchronize()
        us = e0.elapsed_time(e1) / reps * 1e3
        # the same shape in 2-bit slots: two binary passes and a combine per call
        a = torch.randint(0, 256, (copies, N, K // 8), dtype=torch.uint8, device="cuda", generator=g)
        bpl = torch.randint(0, 256, (copies, N, K // 8), dtype=torch.uint8, device="cuda", generator=g)
        wst = torch.empty(max(b1.bit1_gemv_ternary_workspace_bytes(1, N, K), 256), dtype=torch.uint8, device="cuda")
        with torch.cuda.stream(s):
            for i in range(3):
                b1.bit1_gemv_ternary(a[i % copies], bpl[i % copies], sc[i % copies], x, y=y, workspace=wst, stream=s)
            s.synchronize()
            gs = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gs, stream=s):
                for i in range(reps):
                    b1.bit1_gemv_ternary(a[i % copies], bpl[i % copies], sc[i % copies], x, y=y, workspace=wst,
                                         stream=s)
            gs.replay()
            s.synchronize()
            e0.record(s)
            gs.replay()
            e1.record(s)
            e1.synchronize()
        us_slot = e0.elapsed_time(e1) / reps * 1e3
        out[f"gemv_{N}x{K}_b1"] = {"us": round(us, 3), "weight_gbs": round(wb / (us * 1e-6) / 1e9, 1),
                                   "gweights_s": round(N * K / (us * 1e-6) / 1e9, 1),
                                   "slot_path_us": round(us_slot, 3)}
        del packed, sc, graph, a, bpl, gs
        torch.cuda.empty_cache()
    N, K = 151936, 4096
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    packed = torch.randint(0, 243, (N, (K // 128) * 26), dtype=torch.uint8, device="cuda", generator=g)
    a = torch.empty((N, K // 8), dtype=torch.uint8, device="cuda")
    b = torch.empty_like(a)
    for _ in range(3):
        b1.bit1_t5_to_planes(packed, K, a=a, b=b)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(5):
        b1.bit1_t5_to_planes(packed, K, a=a, b=b)
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1) / 5
    moved = packed.numel() + a.numel() + b.numel()
    out["to_planes_151936x4096"] = {"ms": round(ms, 4), "gbs_in_plus_out": round(moved / (ms * 1e-3) / 1e9, 1)}
    del packed, a, b
    torch.cuda.empty_cache()
    return out


def _time_plan(torch, plan, steps, flags=0):
    """Mean ms of plan.run() over `steps` back-to-back runs on a side stream."""
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            plan.run(flags=flags, stream=s)
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(steps):
            plan.run(flags=flags, stream=s)
        e1.record(s)
        e1.synchronize()
    return e0.elapsed_time(e1) / steps


def extra_verify_sweep_8b(torch, b1, B=5, steps=20):
    """A speculative-decoding verify pass on the 8B-class sweep: every matrix
    multiplies B = 5 rows (four drafted tokens plus one), as one grouped
    table-lookup launch, as one grouped launch on register-sourced MMAs, and
    as one grouped tensor-core plan (prep + persistent tcgen05 kernel),
    against the same 253 products as per-matrix batched launches (graph +
    PDL) and the batch-1 sweep."""
    from bit_weight_gemv_sign_b300 import synth
    from bit_weight_gemv_sign_b300.sweep import Sweep
    sw = Sweep(synth.sweep_8b(), seed0=0, batch=B, y_dtype=b1.BF16).fill_device(55)
    plan = sw.group_plan()
    ms = _time_plan(torch, plan, steps)
    tc_plan = sw.group_plan(tensor_cores=True)
    ms_tc = _time_plan(torch, tc_plan, steps, flags=b1.FLAG_PDL)
    del tc_plan
    mma_plan = sw.group_plan(mma=True)
    ms_mma = _time_plan(torch, mma_plan, steps, flags=b1.FLAG_PDL)
    del mma_plan
    sw.capture(pdl=True)
    with torch.cuda.stream(sw.stream):       # graph replays run on the current stream
        for _ in range(2):
            sw.replay()
        sw.stream.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(sw.stream)
        for _ in range(5):
            sw.replay()
        c1.record(sw.stream)
        c1.synchronize()
    ms_chain = c0.elapsed_time(c1) / 5
    hbm, _ = _peaks()
    gbs = sw.weight_bytes / (ms * 1e-3) / 1e9
    gbs_tc = sw.weight_bytes / (ms_tc * 1e-3) / 1e9
    best = min(ms, ms_tc, ms_mma)
    out = {"batch_rows": B, "weight_bytes": sw.weight_bytes, "ms_per_verify_step": best,
           "ms_per_token_row": best / B, "weight_gbs": sw.weight_bytes / (best * 1e-3) / 1e9,
           "hbm_frac": sw.weight_bytes / (best * 1e-3) / 1e9 / hbm,
           "table_lookups_grouped": {"ms_per_verify_step": ms, "ms_per_token_row": ms / B, "weight_gbs": gbs,
                                     "launches_per_step": 1},
           "tensor_cores_grouped": {"ms_per_verify_step": ms_tc, "ms_per_token_row": ms_tc / B,
                                    "weight_gbs": gbs_tc, "launches_per_step": 2},
           "mma_engine_grouped": {"ms_per_verify_step": ms_mma, "ms_per_token_row": ms_mma / B,
                                  "weight_gbs": sw.weight_bytes / (ms_mma * 1e-3) / 1e9, "launches_per_step": 1},
           "ms_per_step_per_matrix_launches": ms_chain, "launches_per_step_per_matrix": sw.launches_per_step(),
           "note": "best of the three grouped plans; compare ms_per_token_row with the batch-1 sweep's ms_per_step"}
    del sw, plan
    torch.cuda.empty_cache()
    return out


def extra_batched_sweep_8b(torch, b1, batches=(16, 64), steps=10):
    """Batched decode on the 8B-class sweep: every matrix multiplies B rows in
    one grouped tensor-core plan (prep + persistent tcgen05 kernel)."""
    from bit_weight_gemv_sign_b300 import synth
    from bit_weight_gemv_sign_b300.sweep import Sweep
    hbm, _ = _peaks()
    out = {}
    for B in batches:
        sw = Sweep(synth.sweep_8b(), seed0=0, batch=B, y_dtype=b1.BF16).fill_device(60 + B)
        plan = sw.group_plan(tensor_cores=True)
        ms = _time_plan(torch, plan, steps, flags=b1.FLAG_PDL)
        gbs = sw.weight_bytes / (ms * 1e-3) / 1e9
        flops = 2.0 * B * sum(m.N * m.K for m in sw.mats)
        out[f"B{B}"] = {"ms_per_step": ms, "ms_per_token_row": ms / B, "weight_gbs": gbs, "hbm_frac": gbs / hbm,
                        "tflops": flops / (ms * 1e-3) / 1e12, "launches_per_step": 2}
        del sw, plan
        torch.cuda.empty_cache()
    out["note"] = "weight_gbs counts each weight byte once per step (B rows per read)"
    return out


def extra_fused_mlp_sweep_8b(torch, b1, steps=20):
    """The 8B-class sweep with each layer's gate and up projections in one
    interleaved matrix whose epilogue applies SwiGLU (217 matrices, the same
    weight bytes), against the plain 253-matrix sweep timed in the same way
    on the same box: the fused activation should cost nothing measurable."""
    from bit_weight_gemv_sign_b300 import synth
    from bit_weight_gemv_sign_b300.sweep import Sweep

    def timed(mats):
        sw = Sweep(mats, seed0=0, batch=1, y_dtype=b1.BF16).fill_device(66)
        plan = sw.group_plan()
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            for _ in range(3):
                plan.run(stream=s)
            s.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for _ in range(steps):
                plan.run(stream=s)
            e1.record(s)
            e1.synchronize()
        wb, yb = sw.weight_bytes, sum(2 * m.out for m in sw.mats)
        del sw, plan
        torch.cuda.empty_cache()
        return e0.elapsed_time(e1) / steps, wb, yb

    ms_f, wb, yb_f = timed(synth.sweep_8b_fused_mlp())
    ms_p, wb_p, yb_p = timed(synth.sweep_8b())
    hbm, _ = _peaks()
    gf, gp = wb / (ms_f * 1e-3) / 1e9, wb_p / (ms_p * 1e-3) / 1e9
    return {"matrices": 217, "weight_bytes": wb, "ms_per_step": ms_f, "weight_gbs": gf, "hbm_frac": gf / hbm,
            "plain_sweep_ms_per_step": ms_p, "plain_sweep_weight_gbs": gp, "output_bytes": yb_f,
            "plain_output_bytes": yb_p,
            "note": "one grouped launch per step either way; h = silu(gate) * up is written instead of gate and up"}


SETTLE_S = 0.25     # busy pre-roll before the warm-up steps (see run_mine)


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

    # The sign bits are converted once, at load, to the g128x layout (a
    # within-group bit permutation that the grouped kernel reads with fewer
    # integer operations; the same bytes, row patches unchanged).
    mats = synth.sweep_8b()
    if args.layers is not None:    # a smaller case of the same sweep, for profiling
        mats = mats[:7 * args.layers] + mats[-1:]
    sw = Sweep(mats, seed0=0, batch=1, y_dtype=b1.BF16).fill().to_g128x()
    plan = sw.group_plan()          # one persistent launch over all 253 GEMVs
    s = torch.cuda.Stream()

    def barrier():
        if dist:
            dist.barrier()
        torch.cuda.synchronize()

    # Consecutive steps are launched with programmatic dependent launch: a
    # step's kernel starts streaming its weights while the previous step
    # drains, and reads its activations only after the previous step has
    # completed (griddepcontrol.wait), as a dependent decode loop would.
    def step():
        plan.run(flags=b1.FLAG_PDL, stream=s)

    # The clock sampler starts first (the nvidia-smi poller needs a moment to
    # come up).  Then the GPU is kept busy with the same step for SETTLE_S of
    # wall time before the warm-up steps, which run directly before the timed
    # ones: on one B300, 20 steps timed after 0.3 s of idle read 4% slower
    # than hot ones, and still 1.2% slower when 5-40 warm-up steps came
    # between the idle gap and the timed region.
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    settle_steps = 0
    # The K timed steps are captured once as a CUDA graph (K launches), so
    # that the first step of the window does not wait on the host's launch
    # call after the barrier.
    with torch.cuda.stream(s):
        step()
        s.synchronize()
        g_steps = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_steps, stream=s):
            for _ in range(args.steps):
                step()
    with ClockSampler(local) as clk, torch.cuda.stream(s):
        t_end = time.perf_counter() + SETTLE_S
        while time.perf_counter() < t_end:
            for _ in range(20):
                step()
            settle_steps += 20
            s.synchronize()
        for _ in range(max(3, args.warmup)):
            step()
        barrier()
        e0.record(s)
        g_steps.replay()
        e1.record(s)
        e1.synchronize()
    barrier()
    ms = max_over_ranks(e0.elapsed_time(e1), dist, "cuda")
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
    # The same calls for E2E_WINDOW steps captured once as a CUDA graph (the
    # upload, download and compute streams fork from and join the capturing
    # stream), so that the host issues one replay per window instead of about
    # ten stream, event and copy calls per step: the measurement then shows
    # the device and the host link, not the speed of this Python loop.
    E2E_WINDOW = 10
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e, stream=s):
        up.wait_stream(s)
        down.wait_stream(s)
        e2e_steps(E2E_WINDOW)
        s.wait_stream(up)
        s.wait_stream(down)
    reps = max(1, (args.steps + E2E_WINDOW - 1) // E2E_WINDOW)
    with torch.cuda.stream(s):
        g_e2e.replay()
        s.synchronize()
        barrier()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(s)
        for _ in range(reps):
            g_e2e.replay()
        f1.record(s)
        f1.synchronize()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), dist, "cuda") / (reps * E2E_WINDOW)
    e2e_gbs = ws * sw.weight_bytes / (e2e_ms * 1e-3) / 1e9
    hy = hy[0]

    # secondary: the same 253 products as a dependent chain of separate
    # launches (CUDA graph, programmatic dependent launch; each kernel waits
    # for its predecessor before reading x, as in a real decode step)
    sw.to_canonical()               # the per-matrix kernels read the canonical layout
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
    chain_ms = max_over_ranks(c0.elapsed_time(c1), dist, "cuda") / chain_steps

    # secondary: the same weights as a fused dependent chain -- per layer q|k|v
    # as one matrix, o, gate|up interleaved with the SwiGLU epilogue, and down
    # reading that h -- 145 launches (graph + PDL)
    fz = Sweep(synth.decode_chain_8b_fused(), seed0=0, batch=1, y_dtype=b1.BF16,
               feed_swiglu=True).fill_device(77)
    fz.capture(pdl=True)
    with torch.cuda.stream(fz.stream):
        for _ in range(3):
            fz.replay()
        fz.stream.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(fz.stream)
        for _ in range(chain_steps):
            fz.replay()
        c1.record(fz.stream)
        c1.synchronize()
    fused_ms = max_over_ranks(c0.elapsed_time(c1), dist, "cuda") / chain_steps
    fused_launches, fused_bytes = fz.launches_per_step(), fz.weight_bytes
    del fz
    torch.cuda.empty_cache()

    hbm, src = _peaks()
    traffic = _traffic_for()
    out = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD if args.layers is None else
                   f"profiling case: the first {args.layers} layers of the 8B-class sweep and its LM head "
                   f"({len(mats)} GEMVs; not the benchmarked workload)",
                   "batch": 1, "weight_bytes_per_step": sw.weight_bytes,
                   "l2": "inputs larger than L2 (1.06 GB of weights per step vs 126 MB L2)",
                   "compute": "1-bit sign weights x bf16 activations, fp32 accumulation, bf16 output",
                   "launch": "one grouped persistent launch of the 253 independent GEMVs per step; the K timed "
                             "steps as one CUDA graph of K launches chained with programmatic dependent launch "
                             "(a step streams its weights while the previous one drains and reads its "
                             "activations only after it completed)",
                   "layout": "sign bits in the g128x layout (bit1_repack_g128x once at load; same bytes)",
                   "settle": f"{settle_steps} untimed steps ({SETTLE_S} s, GPU busy) before the warm-up steps",
                   "parallelism": "replicas" if ws > 1 else "single GPU"},
        "tok_s_equiv": 1e3 / ms_step,
        "hbm_frac": gbs / ws / hbm,
        "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": gbs / ws, "peak": hbm, "unit": "GB/s",
                     "frac": gbs / ws / hbm, "peak_source": src, "traffic": traffic,
                     "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": gbs / ws / NOMINAL_HBM_GBS,
                     "kernel": "k_gemv_group (one launch per step)"},
        "e2e": {"value": e2e_gbs, "unit": "GB/s", "h2d_bytes_per_step": sw.x_bytes,
                "d2h_bytes_per_step": hy.numel() * hy.element_size(), "ms_per_step": e2e_ms,
                "how": "pinned host x -> device, grouped launch, logits -> pinned host every step; "
                       "two I/O slots so step i+1's upload overlaps step i's compute; the calls of "
                       "10 steps captured as one CUDA graph and replayed"},
        "decode_chain": {"value": sw.weight_bytes / (chain_ms * 1e-3) / 1e9, "unit": "GB/s",
                         "ms_per_step": chain_ms, "tok_s_equiv": 1e3 / chain_ms,
                         "launches_per_step": sw.launches_per_step(),
                         "what": "253 dependent launches (graph + PDL, each waits before reading x)"},
        "decode_chain_fused": {"value": fused_bytes / (fused_ms * 1e-3) / 1e9, "unit": "GB/s",
                               "ms_per_step": fused_ms, "tok_s_equiv": 1e3 / fused_ms,
                               "launches_per_step": fused_launches,
                               "what": "the same weights as 145 dependent launches: per layer q|k|v, o, "
                                       "gate|up with the SwiGLU epilogue, down reading h (graph + PDL)"},
        "device_wait_timeouts": timeouts,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_extras:
        out["extras"] = {"c1_tiny": extra_c1_tiny(torch, b1),
                         "c2_projections_b1": extra_c2_projections(torch, b1),
                         "c4_mlp_crossover": extra_c4_crossover(torch, b1),
                         "pp512_tcgen05": extra_pp512(torch, b1),
                         "c5_sweep_27b": extra_c5_sweep_27b(torch, b1),
                         "ternary_sweep_8b": extra_ternary_sweep_8b(torch, b1),
                         "ternary_t5": extra_t5(torch, b1),
                         "verify_sweep_8b_b5": extra_verify_sweep_8b(torch, b1),
                         "batched_sweep_8b_tc": extra_batched_sweep_8b(torch, b1),
                         "fused_mlp_sweep_8b": extra_fused_mlp_sweep_8b(torch, b1)}
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        out["cpu_baseline"] = cpu_baseline(frac_den=1)
        if "extras" in out:
            oracle_beside_extras(out["extras"])
    if rank == 0:
        print(json.dumps(out))
    if dist:
        dist.destroy_process_group()
    return 0


def run_profile_case(args):
    """One grouped plan over the 8B-class sweep (or its first --layers layers)
    at --batch rows on --engine, run --warmup + --steps times: the small,
    short command that the ncu summaries under profiles/ capture.  Prints one
    JSON line (a profiling run, not the benchmark)."""
    import torch
    import bit_weight_gemv_sign_b300 as b1
    from bit_weight_gemv_sign_b300 import synth
    from bit_weight_gemv_sign_b300.sweep import Sweep
    b1.load()
    mats = synth.sweep_8b()
    if args.layers is not None:
        mats = mats[:7 * args.layers] + mats[-1:]
    sw = Sweep(mats, seed0=0, batch=args.batch, y_dtype=b1.BF16).fill_device(5)
    if args.engine == "tables" and args.batch == 1:
        sw.to_g128x()
    plan = sw.group_plan(tensor_cores=args.engine == "tc", mma=args.engine == "mma")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(max(1, args.warmup)):
            plan.run(flags=b1.FLAG_PDL, stream=s)
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(args.steps):
            plan.run(flags=b1.FLAG_PDL, stream=s)
        e1.record(s)
        e1.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    print(json.dumps({"profile_case": f"{len(mats)} GEMVs of the 8B-class sweep", "engine": args.engine,
                      "batch": args.batch, "ms_per_step": ms, "weight_bytes": sw.weight_bytes,
                      "weight_gbs": sw.weight_bytes / (ms * 1e-3) / 1e9,
                      "device_wait_timeouts": b1.bit1_device_wait_timeouts()}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=None,
                    help="profiling: only the first L decoder layers of the sweep and its LM head")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other configurations (tiny, projections, crossover, 27B sweep)")
    ap.add_argument("--engine", default=None, choices=["tables", "mma", "tc"],
                    help="profiling: time only one grouped plan at --batch rows on this engine")
    ap.add_argument("--batch", type=int, default=1, help="batch rows per matrix for --engine")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.engine is not None:
        return run_profile_case(args)
    return run_mine(args)


if __name__ == "__main__":
    sys.exit(main())
