#!/usr/bin/env python
"""Benchmark: attention TFLOP/s of chunked-prefill GQA attention at C=2048, P=2048.

A step is one call of the hot path (one attn_prefill launch) over the serving
chunk: q [2048][32][64] against kCache/vCache [4096][8][64], fp32, with 64
planted score-128 positions. The metric counts visible (row, key) pairs only:
flops = 4 * d * pairs * 32 heads = 51,547,996,160 per step; no credit for
tile padding or masked work.

Timing: W untimed warm-up steps, then exactly K timed steps. Before every step
a 256 MiB buffer is written to flush the 129 MB L2; each step's launch is
bracketed by CUDA events on the launching stream. The timed region is
bracketed by a barrier and torch.cuda.synchronize(); with N > 1 (torchrun)
each rank runs an independent replica and the maximum over ranks is taken.

Also reported on the same JSON line: the end-to-end number through the same
C-ABI entry point with host (pinned) buffers, copies inside the timed region;
the roofline of the kernel; the double-precision oracle timed on the host
cores on a bounded sample of rows; the SM clocks sampled during the timed
region. ``--impl reference`` times the oracle alone (the reference arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "attention TFLOP/s at C=2048,P=2048 (32q/8kv heads, d=64) and % of roofline"
METRIC_LONG = "attention TFLOP/s at C=2048,P=30720 (32q/8kv heads, d=64) and % of roofline"
UNIT = "TFLOP/s"
L2_FLUSH_BYTES = 256 << 20
NUM_SMS = 152
TRIOS = 46  # clusters of three of the prefill kernels a GB300 holds at once

# Nominal dense tensor rates (PFLOP/s per GPU) used only as ratios to carry the
# measured bf16 peak over to tf32: bf16 2.25, tf32 1.1.
NOMINAL_BF16 = 2.25
NOMINAL_TF32 = 1.1


def flops_for(C: int, P: int) -> float:
    pairs = C * P + C * (C + 1) // 2
    return 4.0 * W.D * pairs * W.HQ


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--path", default="attn_prefill",
                    choices=["attn_prefill", "attn_prefill_bf16x3", "attn_prefill_ffma", "attn_reference_prefill"])
    ap.add_argument("--kv", choices=["fp32", "bf16"], default="fp32",
                    help="bf16: the K/V cache in bf16 (attn_prefill_bf16kv)")
    ap.add_argument("--workload", choices=["serve", "long", "chunk", "decode", "matrix"], default="serve",
                    help="chunk: a chunk of --chunk rows against --prefix cached keys (uniform inputs); "
                         "decode: one decode step of 16 sequences x 16384 cached tokens (paged); "
                         "matrix: the three-kernel score-matrix pipeline at T = 512, 1024, 2048")
    ap.add_argument("--chunk", type=int, default=64, help="C of --workload chunk")
    ap.add_argument("--prefix", type=int, default=32768, help="P of --workload chunk")
    ap.add_argument("--paged", action="store_true",
                    help="time attn_prefill_paged on the same workload scattered into shuffled 16-token pages")
    ap.add_argument("--seed", type=int, default=1)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-peak", action="store_true",
                    help="skip the live tensor-pipe rate measurement (the tf32 roofline then uses "
                         "the measured bf16 peak x the nominal tf32/bf16 ratio)")
    ap.add_argument("--no-compare", action="store_true",
                    help="skip timing the FFMA path and the starter reference on the same inputs "
                         "(the page's SPEEDUP of the kernel over its starter design)")
    args = ap.parse_args()
    if args.warmup < 3:  # every timed number follows at least three warm-up steps
        print(f"bench.py: --warmup {args.warmup} raised to 3", file=sys.stderr)
        args.warmup = 3
    return args


def make_workload(name: str, seed: int, C: int = 0, P: int = 0):
    if name == "serve":
        inp = W.serve(seed)
        desc = "serving chunk C=2048 P=2048, 32q/8kv, d=64, fp32 uniform[-1,1), 64 planted 4.0 positions"
    elif name == "chunk":
        inp = W.make_inputs(C, P, seed, "uniform", name=f"chunk C={C} P={P}")
        desc = f"chunk C={C} P={P}, 32q/8kv, d=64, fp32 uniform[-1,1)"
    else:
        inp = W.long_prefix(seed)
        desc = "long cached prefix C=2048 P=30720, 32q/8kv, d=64, fp32 normal(0,0.5) clipped to [-2,2]"
    return inp, desc


def metric_for(args) -> str:
    if args.workload == "serve":
        return METRIC
    if args.workload == "long":
        return METRIC_LONG
    return f"attention TFLOP/s at C={args.chunk},P={args.prefix} (32q/8kv heads, d=64) and % of roofline"


def sample_rows_for_cpu(C: int, every: int):
    """Every ``every``-th chunk row, always including the last (the longest)."""
    rows = list(range(every - 1, C, every))
    if not rows or rows[-1] != C - 1:
        rows.append(C - 1)
    return rows


def cpu_oracle_sample(inp, rows, threads):
    import oracle
    t0 = time.perf_counter()
    oracle.prefill(inp, rows=rows, threads=threads)
    dt = time.perf_counter() - t0
    pairs = sum(inp.P + i + 1 for i in rows)
    return 4.0 * W.D * pairs * W.HQ, dt


# ----------------------------------------------------------------------------
# Clock sampling (nvidia-smi, during the timed region)
# ----------------------------------------------------------------------------

_CLOCK_FIELDS = ["timestamp", "index", "clocks.sm", "clocks.max.sm", "power.draw",
                 "clocks_event_reasons.active", "clocks_event_reasons.hw_slowdown",
                 "clocks_event_reasons.hw_thermal_slowdown",
                 "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]


class ClockSampler:
    def __init__(self, device_index: int):
        self.path = os.path.join(tempfile.mkdtemp(prefix="clk"), "clocks.csv")
        self.proc = None
        self.device_index = device_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device_index), "--query-gpu=" + ",".join(_CLOCK_FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "50", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        deadline = time.time() + 10
        while time.time() < deadline:  # wait for the first sample
            if os.path.exists(self.path) and os.path.getsize(self.path) > 0:
                break
            time.sleep(0.05)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t_begin: float, t_end: float):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != len(_CLOCK_FIELDS):
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
            except ValueError:
                continue
            rows.append((ts, parts))
        window = [p for ts, p in rows if t_begin - 0.05 <= ts <= t_end + 0.05] or [p for _, p in rows]
        if not window:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(p[2]) for p in window if p[2].replace(".", "").isdigit()]
        smax = [float(p[3]) for p in window if p[3].replace(".", "").isdigit()]
        reasons = set()
        for p in window:
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                  "sw_power_cap"), p[6:10]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(window)}


# ----------------------------------------------------------------------------
# Peaks and roofline
# ----------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"),
                "sm_max_mhz": d.get("sm_max_mhz", 2070.0), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0, "source": "fallback"}


TENSOR_PEAK_SHAPES = (("tf32", 128), ("tf32", 256), ("bf16", 128), ("bf16", 256))


def measure_tensor_peaks(cp, torch, stream, sms: int, target_ms: float = 20.0, reps: int = 10, windows=None):
    """The tensor pipe's dense rate on this GPU, measured live: every SM issues
    M = 128, N = n tcgen05.mma instructions back to back (attn_tensor_peak),
    each launch about `target_ms` long, 3 warm-up launches, then `reps` timed
    with CUDA events; the median launch gives the rate. tf32 is the split-TF32
    kernel's instruction kind (no library GEMM reports it); bf16 at N = 256
    sits beside the driver's cuBLAS bf16 figure as a check of the method; N =
    128 is the widest instruction the prefill kernels issue."""
    out = {}
    for kind, n in TENSOR_PEAK_SHAPES:
        bf16 = kind == "bf16"
        probe = 4096
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        cp.attn_tensor_peak(bf16, n, probe, sms, stream)
        e0.record(stream)
        cp.attn_tensor_peak(bf16, n, probe, sms, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        iters = int(min(1 << 22, max(probe, probe * target_ms / max(e0.elapsed_time(e1), 1e-3))))
        for _ in range(3):
            flops = cp.attn_tensor_peak(bf16, n, iters, sms, stream)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        torch.cuda.synchronize()
        w0 = time.time()
        for a, b in ev:
            a.record(stream)
            cp.attn_tensor_peak(bf16, n, iters, sms, stream)
            b.record(stream)
        torch.cuda.synchronize()
        if windows is not None:
            windows[f"{kind}_n{n}"] = (w0, time.time())
        ms = sorted(a.elapsed_time(b) for a, b in ev)
        med = statistics.median(ms)
        out[f"{kind}_n{n}"] = {"tflops": round(flops / (med * 1e-3) / 1e12, 2),
                               "tflops_best": round(flops / (ms[0] * 1e-3) / 1e12, 2),
                               "ms_median": round(med, 4), "iters": iters, "ctas": sms}
    if cp.attn_get_device_error() != 0:
        raise RuntimeError("device error in the tensor-peak measurement")
    return out


def tf32_peak_from(measured):
    """The dense kind::tf32 peak: the faster of the N = 128 and N = 256 loops."""
    return max(measured["tf32_n128"]["tflops"], measured["tf32_n256"]["tflops"])


def kernel_source_hash(path_name: str) -> str:
    """Hash of the kernel source a profile was taken on (traffic goes stale with it)."""
    fname = {"attn_prefill": "tc.cu", "attn_prefill_bf16kv": "tc_bf16.cu", "attn_prefill_bf16x3": "tc_bf16.cu",
             "attn_decode_paged": "decode.cu", "attn_naive_scores": "naive.cu", "attn_naive_softmax": "naive.cu",
             "attn_naive_weighted_sum": "naive.cu", "attn_prefill_ffma": "ffma.cu",
             "attn_reference_prefill": "reference.cu"}[path_name]
    src = os.path.join(ROOT, "chunked_prefill_gqa_gb300", "csrc", fname)
    if not os.path.exists(src):
        src = os.path.join(ROOT, "chunked_prefill_gqa_gb300", "csrc", "ffma.cu")
    return hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]


def launches_per_call(path: str, C: int, P: int) -> int:
    """Kernel launches in one call of `path` on a chunk of C rows at offset P:
    the library's own rule for its split-unit grid, on 32-row query tiles x 8
    KV heads and the device's SMs. A second grid of CTA clusters takes the
    last round's units when that round would leave at least half of the SMs
    idle and every unit sees 1024 keys or more, or when it holds more than
    half as many units as SMs but at most twice the clusters of three the
    device holds at once (46 on a GB300) and every unit sees 8192 keys or
    more. A chunk of a single round whose units are all split runs as one
    grid of clusters instead of the whole-unit grid: still one launch."""
    if path not in ("attn_prefill", "attn_prefill_bf16x3", "attn_prefill_bf16kv"):
        return 1
    units = -(-C // 32) * 8
    if units > NUM_SMS:
        rem = units % NUM_SMS
        shortest = P + min(32, C)  # the shortest unit's keys
        if rem > 0 and 2 * rem <= (NUM_SMS & ~1) and shortest >= 1024:
            return 2
        if NUM_SMS // 2 < rem <= 2 * TRIOS and shortest >= 8192:
            return 2
        return 1
    return 1  # one grid: whole units, or all split


def profiled_traffic(path_name: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source; otherwise None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(f"{path_name}:{workload}")
    if not e or e.get("source_sha256_16") != kernel_source_hash(path_name):
        return None
    return e.get("dram_bytes_per_launch")


def roofline(path_name: str, kernel: str, flops: float, ms: float, peaks, workload: str):
    achieved = flops / (ms * 1e-3) / 1e12
    if kernel.startswith("tcgen05-bf16"):
        peak = peaks["bf16_tflops"]
        r = {"bound": "tensor", "peak_dtype": "bf16",
             "peak_note": f"{peaks['source']} bf16 burst",
             "tensor_passes": 3 if kernel.startswith("tcgen05-bf16x3") else 2,
             "frac_of_split_roof": None}
        if peaks.get("bf16_n128_tflops"):
            # As for tf32: the kernel's MMAs are N <= 128; its tensor work
            # against the pipe's measured rate at N = 128.
            r["tensor_work_frac_of_n128_loop"] = round(r["tensor_passes"] * achieved / peaks["bf16_n128_tflops"], 4)
    elif kernel.startswith("tcgen05-split-tf32"):
        nominal = peaks["bf16_tflops"] * NOMINAL_TF32 / NOMINAL_BF16
        if peaks.get("tf32_tflops"):
            peak = peaks["tf32_tflops"]
            note = ("measured in this run: dense kind::tf32 tcgen05.mma loop on every SM "
                    f"(attn_tensor_peak, best of N = 128 / 256, median of 10 launches)")
        else:
            peak = nominal
            note = f"{peaks['source']} bf16 burst x {NOMINAL_TF32}/{NOMINAL_BF16} (nominal tf32/bf16)"
        r = {"bound": "tensor", "peak_dtype": "tf32", "peak_note": note,
             "tensor_passes": 3,
             "frac_of_split_roof": None,
             "peak_nominal_ratio": round(nominal, 3),
             "frac_of_nominal_ratio_peak": round(achieved / nominal, 4)}
        if peaks.get("tf32_n128_tflops"):
            # The kernel's MMAs are N <= 128 (its tensor memory holds no wider S
            # buffer); the N = 128 loop is the pipe's rate for that shape. The
            # tensor work is the three split products per algorithmic flop.
            r["tensor_work_frac_of_n128_loop"] = round(3 * achieved / peaks["tf32_n128_tflops"], 4)
    else:
        # FP32 FFMA pipe: 152 SMs x 128 lanes x 2 flop per clock at the maximum SM clock.
        peak = NUM_SMS * 128 * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12
        r = {"bound": "alu", "peak_dtype": "fp32-ffma",
             "peak_note": f"152 SMs x 128 FFMA/clk x 2 flop x {peaks['sm_max_mhz']:.0f} MHz"}
    r.update({"achieved": round(achieved, 3), "peak": round(peak, 3), "unit": UNIT,
              "frac": round(achieved / peak, 4),
              "traffic": profiled_traffic(path_name, workload)})
    if "frac_of_split_roof" in r:
        r["frac_of_split_roof"] = round(r["tensor_passes"] * achieved / peak, 4)
    return r


# ----------------------------------------------------------------------------
# Replicas: one process per GPU, each timing its own copy of the workload
# ----------------------------------------------------------------------------

def max_over_ranks(x: float, device) -> float:
    """The largest of every rank's x (the slowest replica's timed region), or
    x itself outside torch.distributed."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world: int, flops_per_step: float, slowest_ms_total: float, steps: int) -> float:
    """Whole-job TFLOP/s: every rank processed `flops_per_step` per step, and
    the job took as long as the slowest rank's timed region."""
    return world * flops_per_step / (slowest_ms_total / steps * 1e-3) / 1e12


# ----------------------------------------------------------------------------
# The reference arm: the oracle on the host cores
# ----------------------------------------------------------------------------

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    inp, desc = make_workload(args.workload, args.seed, args.chunk, args.prefix)
    threads = os.cpu_count() or 1
    # 128 rows per step (every 16th), fewer when the steps asked for would
    # take more than about a minute and a half of host time; the first
    # warm-up step is the probe that decides.
    every = 16
    rows = sample_rows_for_cpu(inp.C, every)
    _, probe_s = cpu_oracle_sample(inp, rows, threads)
    need_s = (args.steps + args.warmup) * probe_s
    if need_s > 90.0:
        every *= -(-int(need_s) // 90)
        rows = sample_rows_for_cpu(inp.C, every)
    for _ in range(args.warmup - 1):
        cpu_oracle_sample(inp, rows, threads)
    total_flops, total_s = 0.0, 0.0
    for _ in range(args.steps):
        f, dt = cpu_oracle_sample(inp, rows, threads)
        total_flops += f
        total_s += dt
    value = total_flops / total_s / 1e12
    sample = f"{len(rows)} of {inp.C} chunk rows (every {every}th + last), all 32 heads, per step"
    line = {"impl": "reference", "metric": metric_for(args),
            "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": desc, "C": inp.C, "P": inp.P, "hq": W.HQ, "hkv": W.HKV, "d": W.D,
                       "path": "oracle", "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads() if threads <= 0 else threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------
# Our arm
# ----------------------------------------------------------------------------

def run_decode(args):
    """One decode step (attn_decode_paged) for 16 sequences of 16384 cached
    tokens: bandwidth-bound, reported as K/V bytes per second against the
    measured HBM copy bandwidth."""
    import torch
    import chunked_prefill_gqa_gb300 as cp
    from chunked_prefill_gqa_gb300 import build as B
    torch.cuda.set_device(0)
    B.build()
    cp.load()
    lens = [16384] * 16
    batch = W.decode_batch(lens, seed=args.seed, spare_pages=0)
    dev = torch.device("cuda", 0)
    q = torch.from_numpy(batch.q).to(dev)
    kp = torch.from_numpy(batch.k_pages).to(dev)
    vp = torch.from_numpy(batch.v_pages).to(dev)
    tb = torch.from_numpy(batch.table).to(dev)
    cl = torch.from_numpy(batch.ctx).to(dev)
    out = torch.empty_like(q)
    nbytes = cp.attn_decode_workspace_bytes(len(lens), batch.max_context)
    ws = torch.empty(max(nbytes // 4, 4), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    kv_bytes = sum(lens) * W.HKV * W.D * 4 * 2
    flops = 4.0 * W.D * sum(lens) * W.HQ
    sampler = ClockSampler(0)
    sampler.start()
    for _ in range(args.warmup):
        cp.attn_decode_paged(q, kp, vp, tb, cl, out, batch.max_context, 0, ws, stream)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()
    t_begin = time.time()
    for i in range(args.steps):
        starts[i].record(stream)
        cp.attn_decode_paged(q, kp, vp, tb, cl, out, batch.max_context, 0, ws, stream)
        ends[i].record(stream)
    torch.cuda.synchronize()
    t_end = time.time()
    sampler.stop()
    if cp.attn_get_device_error() != 0:
        raise RuntimeError("device error in the decode bench")
    ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / args.steps
    gbs = kv_bytes / (ms * 1e-3) / 1e9
    peaks = load_peaks()
    line = {"metric": "decode K/V GB/s, 16 sequences x 16384 cached tokens (32q/8kv, d=64, paged)",
            "value": round(gbs, 1), "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": "decode step, 16 x 16384 tokens, shuffled 16-token pages",
                       "kv_bytes_per_step": kv_bytes, "tflops": round(flops / (ms * 1e-3) / 1e12, 3),
                       "l2": "K/V (1 GiB) larger than L2"},
            "roofline": {"bound": "hbm", "kernel": "decode_split_kernel + decode_merge_kernel",
                         "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4),
                         "traffic": profiled_traffic("attn_decode_paged", "decode")},
            "clocks": sampler.summary(t_begin, t_end),
            "gpu_launches": (2 if nbytes > 0 else 1) * args.steps}
    print(json.dumps(line))
    return 0


def run_matrix(args):
    """The three-kernel score-matrix pipeline on full prompts of 512, 1024 and
    2048 tokens (the sizes the full-score-matrix lab prints), each kernel timed
    with CUDA events, beside attn_full_causal on the same inputs. The line's
    value is the pipeline's time at T = 2048."""
    import torch
    import chunked_prefill_gqa_gb300 as cp
    from chunked_prefill_gqa_gb300 import build as B
    torch.cuda.set_device(0)
    B.build()
    cp.load()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    peaks = load_peaks()
    ffma_peak = NUM_SMS * 128 * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12
    table = []
    sampler = ClockSampler(0)
    sampler.start()
    t_begin = time.time()
    for T in W.FULL_T:
        inp = W.full_causal(T, seed=args.seed)
        q = torch.from_numpy(inp.q).to(dev)
        k = torch.from_numpy(inp.k).to(dev)
        v = torch.from_numpy(inp.v).to(dev)
        out = torch.empty_like(q)
        ws = torch.empty(cp.attn_naive_workspace_bytes(T, 0) // 4, dtype=torch.float32, device=dev)
        steps = [lambda: cp.attn_naive_scores(q, k, ws, 0, stream),
                 lambda: cp.attn_naive_softmax(ws, T, 0, stream),
                 lambda: cp.attn_naive_weighted_sum(ws, v, out, 0, stream),
                 lambda: cp.attn_full_causal(q, k, v, out, stream)]
        for _ in range(args.warmup):
            for f in steps:
                f()
        n = args.steps
        ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in steps]
              for _ in range(n)]
        torch.cuda.synchronize()
        for i in range(n):
            for j, f in enumerate(steps):
                flush.zero_()
                ev[i][j][0].record(stream)
                f()
                ev[i][j][1].record(stream)
        torch.cuda.synchronize()
        if cp.attn_get_device_error() != 0:
            raise RuntimeError("device error in the matrix bench")
        ms = [sum(ev[i][j][0].elapsed_time(ev[i][j][1]) for i in range(n)) / n for j in range(len(steps))]
        visible = 32 * T * (T + 1) // 2
        matrix = 32 * T * T * 4
        # What the matrix itself costs, apart from the contractions: its bytes
        # through HBM (the scores kernel writes all of it, the softmax reads
        # the visible part and writes all of it back, the weighted sum reads
        # the visible part) at the measured copy bandwidth, against the two
        # contractions (2 x 64 flop per visible pair each) at the FFMA peak.
        matrix_bytes = matrix + 4 * visible + matrix + 4 * visible
        matrix_ms = matrix_bytes / (peaks["hbm_gbs"] * 1e9) * 1e3
        contraction_ms = 2 * (2 * 64 * visible) / (ffma_peak * 1e12) * 1e3
        table.append({
            "T": T, "matrix_mib": matrix / 2**20,
            "scores_ms": round(ms[0], 4), "softmax_ms": round(ms[1], 4), "weighted_sum_ms": round(ms[2], 4),
            "pipeline_ms": round(ms[0] + ms[1] + ms[2], 4), "flash_ms": round(ms[3], 4),
            "scores_tflops": round(2 * 64 * visible / (ms[0] * 1e-3) / 1e12, 2),
            "softmax_gbs": round((4 * visible + matrix) / (ms[1] * 1e-3) / 1e9, 1),
            "weighted_sum_tflops": round(2 * 64 * visible / (ms[2] * 1e-3) / 1e12, 2),
            "matrix_traffic_bytes": matrix_bytes,
            "matrix_traffic_ms_at_hbm_peak": round(matrix_ms, 4),
            "contractions_ms_at_ffma_peak": round(contraction_ms, 4),
            "matrix_traffic_over_flash": round(matrix_ms / ms[3], 2),
            "split_note": "pipeline time = matrix traffic + contractions at best; flash_ms has no matrix"})
        del ws
        torch.cuda.empty_cache()
    t_end = time.time()
    sampler.stop()
    last = table[-1]
    dom = max(("scores", "softmax", "weighted_sum"), key=lambda name: last[name + "_ms"])
    if dom == "softmax":
        rl = {"bound": "hbm", "kernel": "naive_softmax_kernel", "achieved": last["softmax_gbs"],
              "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(last["softmax_gbs"] / peaks["hbm_gbs"], 4)}
    else:
        a = last[dom + "_tflops"]
        rl = {"bound": "alu", "kernel": f"naive_{dom}_kernel", "achieved": a, "peak": round(ffma_peak, 2),
              "unit": "TFLOP/s", "frac": round(a / ffma_peak, 4),
              "peak_note": f"152 SMs x 128 FFMA/clk x 2 flop x {peaks['sm_max_mhz']:.0f} MHz"}
    rl["traffic"] = profiled_traffic("attn_naive_" + dom, "matrix")
    line = {"metric": "score-matrix pipeline attention time, full prompt T=2048 (32q/8kv, d=64)",
            "value": last["pipeline_ms"], "unit": "ms", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": last["pipeline_ms"], "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "full causal prompts T = 512, 1024, 2048; workspace 32 x T x T fp32",
                       "l2": "flushed (256 MiB write) before every kernel", "sizes": table},
            "roofline": rl, "clocks": sampler.summary(t_begin, t_end),
            "gpu_launches": 4 * args.steps * len(W.FULL_T)}
    print(json.dumps(line))
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "decode":
        return run_decode(args)
    if args.workload == "matrix":
        return run_matrix(args)

    import torch
    import torch.distributed as dist

    import chunked_prefill_gqa_gb300 as cp
    from chunked_prefill_gqa_gb300 import build as B

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group(backend="nccl")
    else:
        torch.cuda.set_device(0)
    if rank == 0:
        B.build()
    if world > 1:
        dist.barrier()
    cp.load()

    def barrier():
        if world > 1:
            dist.barrier()

    inp, desc = make_workload(args.workload, args.seed, args.chunk, args.prefix)
    C, P = inp.C, inp.P
    flops = flops_for(C, P)
    dev = torch.device("cuda", torch.cuda.current_device())
    q = torch.from_numpy(inp.q).to(dev)
    k = torch.from_numpy(inp.k).to(dev)
    v = torch.from_numpy(inp.v).to(dev)
    out = torch.empty_like(q)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    if args.kv == "bf16":
        if args.path != "attn_prefill" or args.paged:
            raise SystemExit("--kv bf16 times attn_prefill_bf16kv on a contiguous cache only")
        args.path = "attn_prefill_bf16kv"
        kv = W.to_bf16(inp)
        k = torch.from_numpy(kv.k.view(np.int16)).to(dev).view(torch.bfloat16)
        v = torch.from_numpy(kv.v.view(np.int16)).to(dev).view(torch.bfloat16)
        desc += "; K/V cache in bf16"
    fn = getattr(cp, args.path)
    kernel = {"attn_prefill": "tcgen05-split-tf32", "attn_prefill_bf16kv": "tcgen05-bf16kv",
              "attn_prefill_bf16x3": "tcgen05-bf16x3",
              "attn_prefill_ffma": "ffma"}.get(args.path, "reference")

    if args.paged:
        if args.path != "attn_prefill":
            raise SystemExit("--paged times attn_prefill_paged only")
        pg = W.to_pages(inp, seed=args.seed + 5)
        kp = torch.from_numpy(pg.k_pages).to(dev)
        vp = torch.from_numpy(pg.v_pages).to(dev)
        tb = torch.from_numpy(pg.table).to(dev)
        kernel = "tcgen05-split-tf32-paged"
        desc += "; K/V in shuffled 16-token pages"

        def call():
            cp.attn_prefill_paged(q, kp, vp, tb, out, P, stream)
    else:
        def call():
            fn(q, k, v, out, P, stream)

    sampler = ClockSampler(dev.index if world == 1 else local)
    sampler.start()
    for _ in range(args.warmup):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    if cp.attn_get_device_error() != 0:
        raise RuntimeError("device error during warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    t_begin = time.time()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        call()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier()
    wall = time.perf_counter() - wall0
    t_end = time.time()
    sampler.stop()
    err = cp.attn_get_device_error()
    if err != 0:
        raise RuntimeError(f"device error in the timed region: {cp.strerror(err)}")
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_mean = sum(launch_ms) / len(launch_ms)
    kernel_ms_total = max_over_ranks(sum(launch_ms), dev)
    ms_per_step = kernel_ms_total / args.steps
    value = replica_throughput(world, flops, kernel_ms_total, args.steps)

    # End to end from pinned host buffers: the path's host-buffer entry point
    # where it has one (copies overlapped with compute inside the library),
    # else the device entry point between plain copies. Every step's copies
    # are inside the timed region.
    e2e = None
    if not args.no_e2e and not args.paged:
        hq = torch.from_numpy(inp.q).pin_memory()
        if args.kv == "bf16":
            hk = torch.from_numpy(kv.k.view(np.int16)).view(torch.bfloat16).pin_memory()
            hv = torch.from_numpy(kv.v.view(np.int16)).view(torch.bfloat16).pin_memory()
        else:
            hk = torch.from_numpy(inp.k).pin_memory()
            hv = torch.from_numpy(inp.v).pin_memory()
        hout = torch.empty(out.shape, dtype=torch.float32).pin_memory()
        dq, dk, dv, dout = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(out)

        host_fn = getattr(cp, args.path + "_host", None)

        def e2e_step():
            if host_fn is not None:
                host_fn(hq, hk, hv, hout, dq, dk, dv, dout, P, stream)
                return
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            fn(dq, dk, dv, dout, P, stream)
            hout.copy_(dout, non_blocking=True)

        for _ in range(max(3, args.warmup // 4)):
            flush.zero_()
            e2e_step()
        n_e2e = max(10, args.steps // 5)
        es = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
        ee = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
        barrier()
        torch.cuda.synchronize()
        for i in range(n_e2e):
            flush.zero_()
            es[i].record(stream)
            e2e_step()
            ee[i].record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in zip(es, ee)), dev) / n_e2e
        # The host path runs the chunk as sub-chunks; the device call may split
        # its last round's units over CTA pairs (another summation order), so
        # the two agree to rounding, far inside the oracle's tolerance. An
        # output is a weighted mean of V rows, so its rounding scales with
        # max |v| (here about 4), not with the output, which averaging over a
        # long prefix makes small: the bound is 1e-5 (max |v| + |out|).
        dev_out = out.cpu().numpy()
        diff = float(np.max(np.abs(hout.numpy() - dev_out)))
        vmax = float(np.max(np.abs(inp.v)))
        ok = bool(np.all(np.abs(hout.numpy() - dev_out) <= 1e-5 * (vmax + np.abs(dev_out))))
        h2d_bytes = int(hq.numel() * 4 + (hk.numel() + hv.numel()) * hk.element_size())
        d2h_bytes = int(hout.numel()) * 4
        # The link's own rates on this machine: the step's copies alone, one
        # cudaMemcpyAsync per buffer (pinned host memory), best of 5, each
        # direction alone and both directions issued together. A step can take
        # no less than its copies (as the link carries them together) and no
        # less than its compute, so the larger of the two bounds e2e.
        def copy_ms(fn_copy):
            best = float("inf")
            for _ in range(6):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn_copy()
                b.record(stream)
                torch.cuda.synchronize()
                best = min(best, a.elapsed_time(b))
            return best
        h2d_ms = copy_ms(lambda: (dq.copy_(hq, non_blocking=True), dk.copy_(hk, non_blocking=True),
                                  dv.copy_(hv, non_blocking=True)))
        d2h_ms = copy_ms(lambda: hout.copy_(dout, non_blocking=True))
        # Both directions at once (the copy-out on a second stream): whether the
        # link carries them concurrently decides the bound.
        side = torch.cuda.Stream()

        def both():
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                hout.copy_(dout, non_blocking=True)
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            stream.wait_stream(side)
        both_ms = copy_ms(both)
        copies_ms = both_ms  # the copy-in and copy-out of a step, as the link runs them together
        bound_ms, bound_by = max((copies_ms, "host-device copies (both directions at once)"),
                                 (ms_mean, "compute"))
        e2e = {"value": world * flops / (e_ms * 1e-3) / 1e12, "unit": UNIT,
               "ms_per_step": e_ms, "steps": n_e2e,
               "h2d_bytes_per_step": h2d_bytes,
               "d2h_bytes_per_step": d2h_bytes,
               "api": (args.path + "_host") if host_fn is not None else f"copies + {args.path}",
               "matches_device_timed_output": ok, "max_abs_diff_vs_device_timed_output": diff,
               "link": {"h2d_gbs": round(h2d_bytes / (h2d_ms * 1e-3) / 1e9, 1),
                        "d2h_gbs": round(d2h_bytes / (d2h_ms * 1e-3) / 1e9, 1),
                        "h2d_ms": round(h2d_ms, 4), "d2h_ms": round(d2h_ms, 4),
                        "both_directions_ms": round(both_ms, 4), "compute_ms": round(ms_mean, 4),
                        "bound_ms": round(bound_ms, 4), "bound": bound_by,
                        "frac_of_bound": round(bound_ms / e_ms, 4)}}

    compare = None
    if not args.no_compare and rank == 0 and args.kv == "fp32" and not args.paged:
        compare = {}
        for other in ("attn_prefill_ffma", "attn_reference_prefill"):
            if other == args.path:
                continue
            g = getattr(cp, other)
            reps = 3 if other == "attn_reference_prefill" else 20
            for _ in range(2):
                g(q, k, v, out, P, stream)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            tot = 0.0
            for _ in range(reps):
                flush.zero_()
                e0.record(stream)
                g(q, k, v, out, P, stream)
                e1.record(stream)
                torch.cuda.synchronize()
                tot += e0.elapsed_time(e1)
            compare[other] = {"ms": tot / reps, "tflops": flops / (tot / reps * 1e-3) / 1e12,
                              "speedup_of_measured_path": (tot / reps) / ms_mean}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        rows = sample_rows_for_cpu(C, 1)
        f, dt = cpu_oracle_sample(inp, rows, threads)
        cpu = {"value": f / dt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"all {len(rows)} of {C} chunk rows, all 32 heads (the whole step), "
                         f"{dt:.2f} s wall on {threads} threads"}
        rows1 = sample_rows_for_cpu(C, 64)
        f1, dt1 = cpu_oracle_sample(inp, rows1, 1)
        cpu["single_thread"] = {"value": f1 / dt1 / 1e12, "unit": UNIT, "cores": 1,
                                "sample": f"{len(rows1)} of {C} chunk rows (every 64th + last), {dt1:.2f} s"}

    # The tensor pipe's measured dense rate (after every timed region, so its
    # second of full-power MMAs cannot lower the clocks the path was timed at).
    tensor_peaks = None
    if rank == 0 and not args.no_peak and kernel.startswith("tcgen05"):
        psampler = ClockSampler(dev.index if world == 1 else local)
        psampler.start()
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        windows = {}
        tensor_peaks = measure_tensor_peaks(cp, torch, stream, sms, windows=windows)
        psampler.stop()
        # each shape's own clocks (a dense loop can run power-capped), and its
        # rate per clock per SM at the median clock of its timed launches
        for key, (w0, w1) in windows.items():
            clk = psampler.summary(w0, w1)
            tensor_peaks[key]["clocks"] = clk
            if clk.get("sm_mhz"):
                tensor_peaks[key]["flop_per_clk_per_sm"] = round(
                    tensor_peaks[key]["tflops"] * 1e12 / (sms * clk["sm_mhz"] * 1e6), 1)

    if rank == 0:
        peaks = load_peaks()
        if tensor_peaks is not None:
            peaks["tf32_tflops"] = tf32_peak_from(tensor_peaks)
            peaks["tf32_n128_tflops"] = tensor_peaks["tf32_n128"]["tflops"]
            peaks["bf16_n128_tflops"] = tensor_peaks["bf16_n128"]["tflops"]
        line = {
            "metric": metric_for(args),
            "value": round(value, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if args.kv == "bf16" else "f32", "data": "synthetic",
            "config": {"workload": desc, "C": C, "P": P, "hq": W.HQ, "hkv": W.HKV, "d": W.D,
                       "path": args.path, "kernel": kernel,
                       "flops_per_step": flops,
                       "launch_ms_median": round(statistics.median(launch_ms), 5),
                       "launch_ms_min": round(min(launch_ms), 5),
                       "l2": "flushed before every timed step (256 MiB write)",
                       "parallelism": f"replicas x{world}"},
            "roofline": roofline(args.path, kernel, flops, ms_mean, peaks,
                                 args.workload + ("-paged" if args.paged else "")),
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": args.steps * launches_per_call(args.path, C, P),
            "clocks": sampler.summary(t_begin, t_end),
            "wall_s_timed_region": round(wall, 4),
        }
        if compare:
            line["compare"] = compare
        if tensor_peaks is not None:
            line["tensor_peaks"] = tensor_peaks
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
