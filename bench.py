#!/usr/bin/env python3
"""Benchmark of the group-quantized weight-only GEMM on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Workload (the metric's M=1 point): the fused gate+up INT4 GEMV of an 8B-class decoder,
M=1, K=4096, N=28672, G=128, symmetric INT4 codes (zero point 8), fp16 scales, bf16
activations with 0.1% x50 outliers, bf16 output; synthetic seeded inputs (gq_synth).

One step = one decode token through CALLS_PER_STEP gate+up projections, each call reading
a different resident weight copy (COPIES copies rotated, 485 MB in total, well above the
129 MB L2, so every call streams its weights from HBM).  A step is captured once into a
CUDA graph and replayed; K replays are timed with CUDA events on the launching stream,
bracketed by a barrier and device synchronization.

Also reported: the roofline of the dominant kernel against the measured HBM copy
bandwidth, an end-to-end figure through the public C ABI with host buffers (activations
copied in, output copied out every call), the M=4096 prefill throughput against the
measured dense BF16 peak, and the float64 CPU oracle timed on a bounded sample.

With --gpus N > 1 (one process per GPU under torchrun) every rank runs an independent
replica of the same workload (the path does not need to exchange data between GPUs);
value = all ranks' bytes / the slowest rank's time.
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

import gq_synth  # noqa: E402

METRIC = "W4A16 g128 GEMM: HBM GB/s at M=1, TFLOPS at M=4096, % of roofline"
WORKLOAD = "decode_gateup"
CALLS_PER_STEP = 100
COPIES = 8
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def _kernel_traffic(kernel_file: str, summary: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current
    kernel source (the summary records the source's sha256); else None."""
    sp = os.path.join(ROOT, "profiles", summary)
    src = os.path.join(ROOT, "group_quantized_weight_gb300", "csrc", kernel_file)
    if not (os.path.exists(sp) and os.path.exists(src)):
        return None
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    txt = open(sp, encoding="utf-8").read()
    m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", txt)
    m_tr = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not (m_sha and m_tr) or m_sha.group(1) != sha:
        return None
    return float(m_tr.group(1))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _cpu_oracle_timing(cfg, n_cols: int, budget_s: float):
    """Time the float64 oracle, as it stands, on the first n_cols columns of the
    workload (a bounded sample), in a fresh process using every host core for BLAS."""
    code = f"""
import sys, time, json
sys.path.insert(0, {ROOT!r})
import numpy as np, gq_synth, oracle
cfg = gq_synth.CONFIGS[{cfg.name!r}]
inp = gq_synth.make_inputs(cfg, seed=0)
cols = np.arange({n_cols})
t0 = time.perf_counter(); n = 0
while True:
    ref, mag = oracle.reference(inp["A"], inp["codes"], inp["scales"], inp["zeros"], K=cfg.K,
                                N=cfg.N, G=cfg.G, w4=cfg.w4, act=cfg.act, sc=cfg.sc, cols=cols)
    n += 1
    if time.perf_counter() - t0 > {budget_s}:
        break
print(json.dumps({{"calls": n, "seconds": time.perf_counter() - t0}}))
"""
    cores = os.cpu_count() or 1
    env = dict(os.environ, OMP_NUM_THREADS=str(cores), OPENBLAS_NUM_THREADS=str(cores),
               MKL_NUM_THREADS=str(cores))
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    if res.returncode != 0:
        return None, cores, res.stderr[-500:]
    d = json.loads(res.stdout.strip().splitlines()[-1])
    return d, cores, None


def _constants():
    """The package's host-side constants module, loaded from its file: importing the package
    itself would map libgq.so, which the oracle-timed arm must not load."""
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_gq_constants", os.path.join(ROOT, "group_quantized_weight_gb300", "constants.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _sample_bytes(cfg, n_cols):
    return _constants().algorithmic_bytes(cfg.M, cfg.K, n_cols, cfg.G, cfg.w4, cfg.zp, cfg.act,
                                          cfg.sc, cfg.out)


def _pct(xs, q):
    """Percentile q (0..100) of xs by linear interpolation between order statistics."""
    ys = sorted(xs)
    if not ys:
        return None
    pos = (len(ys) - 1) * q / 100.0
    lo = int(pos)
    hi = min(lo + 1, len(ys) - 1)
    return ys[lo] + (ys[hi] - ys[lo]) * (pos - lo)


def _copies_for(nbytes: int, l2_bytes: int, cap: int = 16) -> int:
    """Rotated copies so that one round of them overflows L2 twice over: ceil(2·L2/bytes) + 1."""
    return int(min(cap, -(-2 * l2_bytes // max(nbytes, 1)) + 1))


def slowest_rank_ms(ms: float, world: int, dist, device="cpu") -> float:
    """The timed region's length on the slowest rank (every rank receives it)."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(world: int, bytes_per_call: int, calls: int, ms: float) -> float:
    """Whole-job throughput: the bytes of every rank's calls over the slowest rank's time."""
    return world * bytes_per_call * calls / (ms * 1e-3) / 1e9


def run_reference(args):
    """The reference arm: the float64 CPU oracle on a bounded column sample per step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    cfg = gq_synth.CONFIGS[WORKLOAD]
    n_cols = 512
    budget = 0.0   # one call per step
    import oracle
    inp = gq_synth.make_inputs(cfg, seed=0)
    cols = np.arange(n_cols)

    def step():
        oracle.reference(inp["A"], inp["codes"], inp["scales"], inp["zeros"], K=cfg.K, N=cfg.N,
                         G=cfg.G, w4=cfg.w4, act=cfg.act, sc=cfg.sc, cols=cols)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    del budget
    nbytes = _sample_bytes(cfg, n_cols)
    value = nbytes * args.steps / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD} M=1 K=4096 N=28672 G=128, first {n_cols} columns "
                               "per step (float64 CPU oracle)"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": os.cpu_count(),
                         "kind": "oracle",
                         "sample": f"one step = the oracle on the first {n_cols} of 28672 columns"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload table of the five configurations")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the M sweep against a dense BF16 GEMM")
    ap.add_argument("--calls-per-step", type=int, default=CALLS_PER_STEP,
                    help="gq_gemm calls per step (a smaller value for profiler runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")

    import group_quantized_weight_gb300 as gq
    from group_quantized_weight_gb300.constants import GQ_STATIC_W, algorithmic_bytes, gemm_flops, prec_flags

    cfg = gq_synth.CONFIGS[WORKLOAD]
    prec = prec_flags(cfg.w4, cfg.zp, cfg.act, cfg.sc, cfg.out) | GQ_STATIC_W
    inp = gq_synth.make_inputs(cfg, seed=0)
    dev = torch.device("cuda", torch.cuda.current_device())

    def to_dev(a):
        a = np.ascontiguousarray(a)
        v = a.view(np.int16) if a.dtype == np.uint16 else (a.view(np.int32) if a.dtype == np.uint32 else a)
        return torch.from_numpy(v).to(dev)

    codes = to_dev(inp["codes"])
    packed0 = gq.pack_weights_t(codes, cfg.K, cfg.N, cfg.G, prec)
    scales0 = to_dev(inp["scales"])
    W = [packed0] + [packed0.clone() for _ in range(COPIES - 1)]
    S = [scales0] + [scales0.clone() for _ in range(COPIES - 1)]
    del codes
    A = to_dev(inp["A"])
    out = torch.empty((cfg.M, cfg.N), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def call(i, a=A, o=out):
        st = gq.gq_gemm(cfg.M, cfg.K, cfg.N, cfg.G, prec, a.data_ptr(), W[i % COPIES].data_ptr(),
                        S[i % COPIES].data_ptr(), None, o.data_ptr(),
                        torch.cuda.current_stream().cuda_stream)
        if st != 0:
            raise RuntimeError(f"gq_gemm failed: {gq.gq_status_string(st)}")

    w_ptrs = [w.data_ptr() for w in W]
    s_ptrs = [x.data_ptr() for x in S]
    host_call = gq.gq_gemm_host
    e2e_ws = gq.gq_plan(cfg.M, cfg.K, cfg.N, cfg.G, prec)["workspace_bytes"]

    def call_host(i, a_host, a_dev, o_dev, o_host, s_ptr):
        # the public call on host buffers: activations in, the GEMM, the output back
        st = host_call(cfg.M, cfg.K, cfg.N, cfg.G, prec, a_host, a_dev, w_ptrs[i % COPIES],
                       s_ptrs[i % COPIES], None, o_dev, o_host, s_ptr)
        if st != 0:
            raise RuntimeError(f"gq_gemm_host failed: {gq.gq_status_string(st)}")

    call(0)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    calls_per_step = args.calls_per_step
    with torch.cuda.graph(graph):
        for i in range(calls_per_step):
            call(i)
    torch.cuda.synchronize()

    gpu_id = None
    try:
        gpu_id = str(torch.cuda.get_device_properties(dev).uuid)
        if not gpu_id.startswith("GPU-"):
            gpu_id = "GPU-" + gpu_id
    except Exception:
        gpu_id = os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0]
    sampler = ClockSampler(gpu_id)
    time.sleep(0.3)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    ev[0].record(stream)
    for i in range(args.steps):
        graph.replay()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    ms = slowest_rank_ms(ev[0].elapsed_time(ev[-1]), world, dist, dev)
    step_us = [1e3 * ev[i].elapsed_time(ev[i + 1]) / calls_per_step for i in range(args.steps)]
    # five equal blocks of the timed steps: the median block and the spread of the steps
    blocks = [statistics.fmean(step_us[i * len(step_us) // 5:(i + 1) * len(step_us) // 5])
              for i in range(5)] if len(step_us) >= 5 else step_us
    dist_us = {"median_of_5_blocks": statistics.median(blocks), "p10": _pct(step_us, 10),
               "p90": _pct(step_us, 90), "unit": "us per gq_gemm call (graph-replayed)"}
    # one host-launched call at a time (no graph, no overlap with a previous call)
    single = []
    for i in range(30):
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s0.record(stream)
        call(i)
        s1.record(stream)
        torch.cuda.synchronize()
        if i >= 5:
            single.append(1e3 * s0.elapsed_time(s1))
    dist_us["single_call_us"] = statistics.median(single)
    nbytes = algorithmic_bytes(cfg.M, cfg.K, cfg.N, cfg.G, cfg.w4, cfg.zp, cfg.act, cfg.sc, cfg.out)
    launches = args.steps * calls_per_step
    kernel_us = 1e3 * ms / launches
    value = job_gbs(world, nbytes, launches, ms)
    peaks, peak_kind = _peaks()
    achieved = nbytes / (kernel_us * 1e-6) / 1e9

    e2e = _e2e(args, torch, np, inp, A, out, call_host, world, nbytes, calls_per_step, e2e_ws)

    prefill = None
    if not args.no_prefill and rank == 0:
        prefill = _prefill(gq, torch, dev, peaks, peak_kind)
    configs = None
    if not args.no_configs and rank == 0:
        configs = _all_configs(gq, torch, dev, peaks, peak_kind)
    sweep = None
    if not args.no_sweep and rank == 0:
        sweep = _m_sweep(gq, torch, dev, peaks)

    traffic = _kernel_traffic("gq_gemv.cu", "w4_gemv_decode_gateup.md")
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{WORKLOAD}: M=1 K=4096 N=28672 G=128 W4A16 sym, fp16 scales, "
                               "bf16 act/out",
                   "step": f"{calls_per_step} gq_gemm calls replayed from one CUDA graph",
                   "weights": "static (GQ_STATIC_W): a call may start streaming its weights "
                              "before the previous call ends; activations wait for it",
                   "l2": f"inputs larger than L2: {COPIES} rotated weight copies "
                         f"({COPIES * nbytes / 1e6:.0f} MB)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "kernel": "w4_gemv_kernel", "peak_source": f"hbm_gbs of {peak_kind}",
                     "kernel_us": kernel_us, "kernel_us_distribution": dist_us},
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if configs:
        line["configs"] = configs
    if sweep:
        line["m_sweep"] = sweep
    return _finish(args, line, prefill, rank, world, cfg, dist)


def _e2e(args, torch, np, inp, A, out, call_host, world, nbytes, calls_per_step, ws_bytes):
    """End to end through the C ABI with host buffers: per call, gq_gemm_host copies the
    activations in from pinned host memory, runs the GEMM and copies the output back, all
    asynchronous on a stream; one synchronization after the last call.  The calls are
    independent requests, so they alternate between two streams, each with its own staging
    buffers (the copies of one overlap the GEMM of the other), unless the plan uses the
    shared workspace, which calls overlapping in time must not share."""
    if args.no_e2e:
        return None
    e2e_calls = 2000
    nstreams = 2 if ws_bytes == 0 else 1
    streams = [torch.cuda.Stream() for _ in range(nstreams)]
    A_h = torch.from_numpy(np.ascontiguousarray(inp["A"]).view(np.int16)).pin_memory()
    out_h = [torch.empty(tuple(out.shape), dtype=out.dtype).pin_memory() for _ in streams]
    A_d = [torch.empty_like(A) for _ in streams]
    out_d = [torch.empty_like(out) for _ in streams]
    a_h = A_h.data_ptr()
    bufs = [(A_d[j].data_ptr(), out_d[j].data_ptr(), out_h[j].data_ptr(), streams[j].cuda_stream)
            for j in range(nstreams)]
    torch.cuda.synchronize()
    for i in range(20):
        a_d, o_d, o_h, sp = bufs[i % nstreams]
        call_host(i, a_h, a_d, o_d, o_h, sp)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(e2e_calls):
        a_d, o_d, o_h, sp = bufs[i % nstreams]
        call_host(i, a_h, a_d, o_d, o_h, sp)
    t_issued = time.perf_counter()
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    return {"value": world * nbytes * e2e_calls / e2e_s / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": A_h.numel() * 2 * calls_per_step,
            "d2h_bytes_per_step": out_h[0].numel() * 2 * calls_per_step,
            "host_issue_us_per_call": (t_issued - t0) / e2e_calls * 1e6,
            "streams": nstreams,
            "note": "per call: one gq_gemm_host call (H2D of the activations from pinned host "
                    "memory, the GEMM, D2H of the output, asynchronous on the call's stream), "
                    "host-launched (no graph); independent calls alternate between the streams"}


def _finish(args, line, prefill, rank, world, cfg, dist):
    if prefill:
        line["prefill"] = prefill
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        d, cores, err = _cpu_oracle_timing(cfg, 4096, 10.0)
        if d:
            per_call = d["seconds"] / d["calls"]
            line["cpu_baseline"] = {
                "value": _sample_bytes(cfg, 4096) / per_call / 1e9, "unit": "GB/s",
                "cores": cores, "kind": "oracle",
                "sample": f"float64 oracle on the first 4096 of 28672 columns, "
                          f"{d['calls']} calls in {d['seconds']:.1f} s"}
        else:
            line["cpu_baseline"] = {"value": None, "unit": "GB/s", "cores": cores,
                                    "kind": "oracle", "sample": f"failed: {err}"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


L2_BYTES = 126 * 2 ** 20   # GB300 L2 (about 126 MiB usable)


def _dev_inputs(torch, dev, inp):
    def to_dev(a):
        if a is None:
            return None
        a = np.ascontiguousarray(a)
        v = a.view(np.int16) if a.dtype == np.uint16 else (a.view(np.int32) if a.dtype == np.uint32 else a)
        return torch.from_numpy(v).to(dev)
    return {k: to_dev(inp[k]) for k in ("codes", "scales", "zeros", "A")}


def _all_configs(gq, torch, dev, peaks, peak_kind):
    """Every workload of the benchmark set: mean time per gq_gemm call (CUDA graph of back to
    back calls, rotating weight copies so that the weights come from HBM whenever they fit
    at most a third of L2 per copy), HBM GB/s of the algorithmic bytes, TFLOPS, and the
    fraction of the roofline that bounds it (HBM below M = 128, dense BF16 above)."""
    from group_quantized_weight_gb300.constants import (GQ_ACT_F32, GQ_ACT_I8, GQ_GATE_UP,
                                                        GQ_STATIC_W, algorithmic_bytes,
                                                        gemm_flops, prec_flags)
    out = []
    side = torch.cuda.Stream()           # graph capture needs a stream other than the legacy one
    for name in ("tiny_gemv", "decode_gateup", "decode_gateup_silu", "q8_m1", "q8_m32",
                 "q8a8_m1", "q8a8_m32", "asym_m16", "asym_m16_silu", "asym_m16_zf", "prefill"):
        # decode_gateup_silu, asym_m16_silu: the gate+up shapes with the fused SiLU-and-mul
        # epilogue (GQ_GATE_UP): the same weights, an output of N/2 columns.  q8a8_*: the Q8_0 shapes
        # with int8 activation codes and per-group scales (GQ_ACT_I8), quantized on the device
        # by gq_quantize_act before the timed calls.  asym_m16_zf: the asymmetric shape with
        # bf16 float zero points subtracted after scaling (GQ_ZP_FLOAT) in place of packed ones
        fused = name.endswith("_silu")
        a8 = name.startswith("q8a8")
        if name == "asym_m16_zf":
            cfg = gq_synth.CONFIGS["asym_m16"].replace(name=name, zp=False, zf=True)
        else:
            cfg = gq_synth.CONFIGS[name[:-len("_silu")] if fused else name.replace("q8a8", "q8")]
        prec = prec_flags(cfg.w4, cfg.zp, cfg.act, cfg.sc, cfg.out, zf=cfg.zf) | GQ_STATIC_W
        if fused:
            prec |= GQ_GATE_UP
        if a8:
            prec = (prec & ~GQ_ACT_F32) | GQ_ACT_I8
        d = _dev_inputs(torch, dev, gq_synth.make_inputs(cfg, seed=0))
        packed = gq.pack_weights_t(d["codes"], cfg.K, cfg.N, cfg.G, prec)
        nbytes = algorithmic_bytes(cfg.M, cfg.K, cfg.N, cfg.G, cfg.w4, cfg.zp, cfg.act, cfg.sc,
                                   cfg.out, zf=cfg.zf)
        if fused:
            nbytes -= cfg.M * (cfg.N // 2) * 2        # half the bf16 output columns
        a_ptr, as_ptr = d["A"].data_ptr(), None
        if a8:                                        # int8 codes + fp32 scales per group
            Aq, As = gq.quantize_act_t(d["A"], cfg.K, cfg.G, GQ_ACT_F32, stream=side)
            side.synchronize()
            a_ptr, as_ptr = Aq.data_ptr(), As.data_ptr()
            nbytes += cfg.M * cfg.K * (1 - 4) + cfg.M * (cfg.K // cfg.G) * 4
        wbytes = packed.numel() + d["scales"].numel() * d["scales"].element_size()
        copies = 1 if cfg.M >= 128 else _copies_for(wbytes, L2_BYTES)
        W = [packed] + [packed.clone() for _ in range(copies - 1)]
        S = [d["scales"]] + [d["scales"].clone() for _ in range(copies - 1)]
        Z = None
        if d["zeros"] is not None:
            Z = [d["zeros"]] + [d["zeros"].clone() for _ in range(copies - 1)]
        odt = torch.float32 if cfg.out == "f32" else torch.bfloat16
        o = torch.empty((cfg.M, cfg.N // 2 if fused else cfg.N), dtype=odt, device=dev)
        big = cfg.M >= 128
        res = gq.gq_bench_calls(cfg.M, cfg.K, cfg.N, cfg.G, prec, a_ptr,
                          [w.data_ptr() for w in W], [x.data_ptr() for x in S],
                          [z.data_ptr() for z in Z] if Z else None, o.data_ptr(),
                          warmup=3, iters=10 if big else 200, use_graph=not big,
                          stream=side.cuda_stream, a_scales_ptr=as_ptr)
        us = res["us_per_call"]
        gbs = nbytes / (us * 1e-6) / 1e9
        tf = gemm_flops(cfg.M, cfg.K, cfg.N) / (us * 1e-6) / 1e12
        plan = gq.gq_plan(cfg.M, cfg.K, cfg.N, cfg.G, prec)
        row = {"workload": name, "M": cfg.M, "K": cfg.K, "N": cfg.N, "G": cfg.G,
               **({"epilogue": "silu(gate) * up, N/2 output columns"} if fused else {}),
               **({"activations": "int8 codes, fp32 scale per (row, group)"} if a8 else {}),
               **({"zero_points": "bf16 float zero points, W = q*s - zf"} if cfg.zf else {}),
               "path": plan["path"], "us": us, "GB/s": gbs, "TFLOPS": tf,
               "weight_copies": copies,
               "l2": ("from HBM (rotated copies exceed L2)" if copies * wbytes > L2_BYTES
                      else "weights fit in L2")}
        if big:
            row.update(bound="tensor", frac=tf / peaks["bf16_tflops"],
                       peak=f"bf16_tflops of {peak_kind}")
        else:
            row.update(bound="hbm", frac=gbs / peaks["hbm_gbs"], peak=f"hbm_gbs of {peak_kind}")
        out.append(row)
        del W, S, Z, d, packed, o
        torch.cuda.empty_cache()
    return out


def _m_sweep(gq, torch, dev, peaks):
    """K=4096 N=14336 G=128 W4A16 (fp16 scales, bf16 out) against the same product as a dense
    BF16 GEMM (torch.matmul on cuBLAS, weights already BF16) for M = 1 ... 4096: time per
    call of each, their ratio, and the smallest M at which the INT4 path is the slower."""
    from group_quantized_weight_gb300.constants import GQ_STATIC_W, prec_flags
    base = gq_synth.Config("sweep", M=1, K=4096, N=14336, G=128)
    prec = prec_flags(True, False, "bf16", "fp16", "bf16") | GQ_STATIC_W
    w = gq_synth.make_weights(base, seed=0)
    codes = torch.from_numpy(w["codes"].view(np.int32)).to(dev)
    packed = gq.pack_weights_t(codes, base.K, base.N, base.G, prec)
    S = torch.from_numpy(w["scales"].view(np.int16)).to(dev)
    del codes
    # both sides rotate enough copies that each round of them overflows L2 twice over, so
    # every call of either streams its weights from HBM
    copies = _copies_for(packed.numel() + S.numel() * 2, L2_BYTES)
    copies_d = _copies_for(base.N * base.K * 2, L2_BYTES)
    W = [packed] + [packed.clone() for _ in range(copies - 1)]
    Ss = [S] + [S.clone() for _ in range(copies - 1)]
    Wd = [torch.randn(base.N, base.K, device=dev).to(torch.bfloat16) for _ in range(copies_d)]
    rows = []
    crossover = None
    stream = torch.cuda.Stream()         # graph capture needs a stream other than the legacy one
    torch.cuda.synchronize()
    for M in (1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024, 2048, 4096):
        a = gq_synth.make_activations(base, seed=0, M=M)
        A = torch.from_numpy(a.view(np.int16)).to(dev)
        o = torch.empty((M, base.N), dtype=torch.bfloat16, device=dev)
        iters = 200 if M <= 64 else (50 if M <= 512 else 10)
        res = gq.gq_bench_calls(M, base.K, base.N, base.G, prec, A.data_ptr(), [x.data_ptr() for x in W],
                          [x.data_ptr() for x in Ss], None, o.data_ptr(), warmup=3, iters=iters,
                          use_graph=M < 128, stream=stream.cuda_stream)
        Ad = A.view(torch.bfloat16)
        for i in range(3):
            torch.matmul(Ad, Wd[i % copies_d].t())
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for i in range(iters):
            torch.matmul(Ad, Wd[i % copies_d].t())
        e1.record()
        torch.cuda.synchronize()
        dense_us = e0.elapsed_time(e1) * 1e3 / iters
        us = res["us_per_call"]
        if crossover is None and us > dense_us:
            crossover = M
        rows.append({"M": M, "int4_us": us, "bf16_dense_us": dense_us, "speedup": dense_us / us,
                     "path": gq.gq_plan(M, base.K, base.N, base.G, prec)["path"]})
    del W, Ss, Wd
    torch.cuda.empty_cache()
    return {"shape": "K=4096 N=14336 G=128 W4A16 sym fp16 scales vs torch.matmul bf16",
            "weights": f"rotated copies, ceil(2*L2/bytes)+1 of each: INT4 {copies} x 30.3 MB "
                       f"= {copies * 30.3:.0f} MB, BF16 {copies_d} x 117.4 MB = "
                       f"{copies_d * 117.4:.0f} MB (L2 {L2_BYTES / 2**20:.0f} MiB)",
            "crossover_M": crossover, "rows": rows}


def _prefill(gq, torch, dev, peaks, peak_kind):
    """M=4096 K=4096 N=14336 prefill: TFLOPS of gq_gemm vs the measured dense BF16 peak."""
    from group_quantized_weight_gb300.constants import GQ_STATIC_W, gemm_flops, prec_flags
    cfg = gq_synth.CONFIGS["prefill"]
    prec = prec_flags(cfg.w4, cfg.zp, cfg.act, cfg.sc, cfg.out) | GQ_STATIC_W
    w = gq_synth.make_weights(cfg, seed=0)
    a = gq_synth.make_activations(cfg, seed=0)
    codes = torch.from_numpy(w["codes"].view(np.int32)).to(dev)
    packed = gq.pack_weights_t(codes, cfg.K, cfg.N, cfg.G, prec)
    S = torch.from_numpy(w["scales"].view(np.int16)).to(dev)
    A = torch.from_numpy(a.view(np.int16)).to(dev)
    out = torch.empty((cfg.M, cfg.N), dtype=torch.bfloat16, device=dev)
    res = gq.gq_bench_calls(cfg.M, cfg.K, cfg.N, cfg.G, prec, A.data_ptr(), [packed.data_ptr()],
                      [S.data_ptr()], None, out.data_ptr(), warmup=3, iters=10,
                      use_graph=False, stream=torch.cuda.current_stream().cuda_stream)
    us = res["us_per_call"]
    flops = gemm_flops(cfg.M, cfg.K, cfg.N)
    tflops = flops / (us * 1e-6) / 1e12
    plan = gq.gq_plan(cfg.M, cfg.K, cfg.N, cfg.G, prec)
    # context: the same product as a dense BF16 GEMM in cuBLAS (weights already BF16)
    Wd = torch.randn(cfg.N, cfg.K, device=dev).to(torch.bfloat16)
    Ad = torch.randn(cfg.M, cfg.K, device=dev).to(torch.bfloat16)
    for _ in range(3):
        torch.matmul(Ad, Wd.t())
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(10):
        torch.matmul(Ad, Wd.t())
    e1.record()
    torch.cuda.synchronize()
    cublas_us = e0.elapsed_time(e1) * 100.0
    del Wd, Ad
    # the FP8 W8A8 GEMM with 128 x 128 block scales (gq_gemm_fp8_block) on the same shape:
    # E4M3 activations and weights, one fp32 scale per (row, 128-k block) and per weight block
    Af = torch.randn(cfg.M, cfg.K, device=dev).to(torch.float8_e4m3fn).view(torch.uint8)
    Wf = (0.5 * torch.randn(cfg.N, cfg.K, device=dev)).to(torch.float8_e4m3fn).view(torch.uint8)
    a_s = torch.rand(cfg.K // 128, cfg.M, device=dev) * 0.09 + 0.01
    w_s = torch.rand(-(-cfg.N // 128), cfg.K // 128, device=dev) * 0.09 + 0.01
    of = torch.empty((cfg.M, cfg.N), dtype=torch.bfloat16, device=dev)
    for _ in range(3):
        gq.gemm_fp8_t(Af, a_s, Wf, w_s, of, cfg.M, cfg.K, cfg.N)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(10):
        gq.gemm_fp8_t(Af, a_s, Wf, w_s, of, cfg.M, cfg.K, cfg.N)
    e1.record()
    torch.cuda.synchronize()
    fp8_us = e0.elapsed_time(e1) * 100.0
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    del Af, Wf, a_s, w_s, of
    return {"workload": "prefill: M=4096 K=4096 N=14336 G=128 W4A16 sym", "us": us,
            "tflops": tflops, "peak_tflops": peaks["bf16_tflops"],
            "frac": tflops / peaks["bf16_tflops"], "peak_source": f"bf16_tflops of {peak_kind}",
            "path": plan["path"], "cublas_bf16_dense_us": cublas_us,
            "cublas_bf16_dense_tflops": flops / (cublas_us * 1e-6) / 1e12,
            "fp8_block": {"workload": "FP8 E4M3 W8A8, 1x128 / 128x128 block scales, "
                                      "M=4096 K=4096 N=14336, bf16 out",
                          "us": fp8_us, "tflops": flops / (fp8_us * 1e-6) / 1e12,
                          "peak_tflops": fp8_peak,
                          "frac": flops / (fp8_us * 1e-6) / 1e12 / fp8_peak,
                          "peak_source": f"2 x bf16_tflops of {peak_kind} (nominal FP8/BF16 "
                                         "ratio)"}}


if __name__ == "__main__":
    sys.exit(main())
