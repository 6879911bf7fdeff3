#!/usr/bin/env python3
"""Benchmark of the block-quantized projection matmul on one GB300.

Headline workload: the Q4_0 decode GEMV at N=1 on the Llama-3-8B projection
shapes (M,K) = (4096,4096), (1024,4096), (14336,4096), (4096,14336); `value`
is its effective HBM bandwidth (algorithmic bytes / device time, GB/s).
One step runs the whole hot path once over one batch of synthetic input:
  decode   4 x Q4_0 GEMV, N=1                          (decode GEMV)
  lmhead   Q6_K 128256 x 4096 LM head, N=8, f32 X     (small-N GEMV)
  prefill      Q4_K 4096x4096 and 14336x4096, N=512, bf16 X (tcgen05 GEMM)
  prefill_f32  the same with f32 X (x->bf16 conversion + tcgen05 GEMM)
Weights are replicated into R device copies whose total size exceeds L2
several times, and step s uses copy s % R (rotating inputs > L2 instead of an
L2 flush).  Each op is captured in a CUDA graph over all R copies and timed
with CUDA events on the launching stream; the step time is the sum.

--impl reference runs the oracle (plain C, f64, host cores) on a bounded
sample of the same workload and prints the same JSON line with
"impl": "reference".
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_quantized_gemv_gguf_gb300 import synth  # noqa: E402

DECODE_SHAPES = [(4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336)]
LMHEAD = (128256, 4096, 8)
PREFILL_SHAPES = [(4096, 4096), (14336, 4096)]
PREFILL_N = 512
METRIC = "decode GEMV effective HBM GB/s (% of 8 TB/s); prefill N=512 GEMM TFLOP/s (% peak)"
WORKLOAD = ("Q4_0 decode GEMV N=1 on Llama-3-8B projection shapes (4096,4096) (1024,4096) (14336,4096) "
            "(4096,14336); same step also runs the Q6_K 128256x4096 LM head at N=8 and the Q4_K "
            "(4096,4096)+(14336,4096) prefill GEMM at N=512 with bf16 X and with f32 X")
NOMINAL_HBM_GBS = 8000.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# DRAM bytes (read + write) per pass of an op, summed over its kernels, from
# one ncu capture (dram__bytes_read.sum + dram__bytes_write.sum), keyed by the
# sha256 of the kernel sources they were taken on.  A source change since the
# capture turns the figure into null.
TRAFFIC = {
    # gemv_mma_kernel, Q6_K 128256x4096, N=8: 449.53 MB read + 5.59 MB written
    # (profiles/gemv_mma_q6_k_lmhead_n8.md)
    "lmhead": ("fd99067e98516dce", 455.11e6),
}


def _kernel_hash():
    import hashlib
    h = hashlib.sha256()
    cs = os.path.join(ROOT, "block_quantized_gemv_gguf_gb300", "csrc")
    for f in sorted(os.listdir(cs)):
        if f.endswith((".cu", ".cuh", ".h")):
            h.update(open(os.path.join(cs, f), "rb").read())
    return h.hexdigest()[:16]


def traffic_for(op):
    t = TRAFFIC.get(op)
    if not t or t[0] != _kernel_hash():
        return None
    return t[1]


def wbytes(wt, M, K):
    return synth.weight_bytes(wt, M, K)


def alg_bytes(wt, M, K, N, xs):
    return wbytes(wt, M, K) + N * K * xs + N * M * 4


# ---------------------------------------------------------------------------
# clocks sampler (nvidia-smi during the timed region)
# ---------------------------------------------------------------------------
class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index=0):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except FileNotFoundError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# multi-rank aggregation (each rank runs the whole step on its own GPU: weak
# scaling, no data-path collective)
# ---------------------------------------------------------------------------
def max_over_ranks(values: dict, world: int, device) -> dict:
    """Per-op times (ms per step), maximum over all ranks; unchanged when
    world == 1.  Every rank must call it with the same keys."""
    if world <= 1:
        return dict(values)
    import torch
    import torch.distributed as dist
    keys = sorted(values)
    t = torch.tensor([float(values[k]) for k in keys], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return {k: float(v) for k, v in zip(keys, t.tolist())}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_gpu(args):
    import torch
    from block_quantized_gemv_gguf_gb300 import qmm

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    qmm.load()
    # Weights are written once and then only read: let each call start
    # streaming its weights before the preceding kernel on the stream ends.
    qmm.qmm_set_static_weights(not args.no_static_weights)
    hbm_peak, bf16_peak, bf16_sus, peak_src = peaks()
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 1024 * 1024) or 126 * 1024 * 1024
    R = args.copies

    all_ops = {"decode", "lmhead", "prefill", "prefill_f32"}
    only = set(args.only.split(",")) if args.only else all_ops
    bad = only - all_ops
    if bad:
        raise SystemExit(f"unknown op(s) in --only: {sorted(bad)}")

    # ---- inputs: generated once on the host, replicated R times on device ----
    def make(wt, M, K, name):
        w = torch.from_numpy(synth.gen_weights(wt, M, K, name)).to(dev)
        return [w] + [w.clone() for _ in range(R - 1)]

    stream = torch.cuda.Stream(device=dev)

    def chk(s):
        if s != qmm.OK:
            raise RuntimeError(qmm.status_name(s))

    ops, launches_per_pass = {}, {}
    Mh, Kh, Nh = LMHEAD
    if "decode" in only:
        dec_w = [make(synth.Q4_0, M, K, f"bench-decode-{M}x{K}") for (M, K) in DECODE_SHAPES]
        dec_x = [torch.from_numpy(synth.gen_x(1, K, f"bench-decode-{K}")).to(dev) for (_, K) in DECODE_SHAPES]
        dec_y = [torch.empty(1, M, device=dev) for (M, _) in DECODE_SHAPES]

        def op_decode(r):
            for i, (M, K) in enumerate(DECODE_SHAPES):
                chk(qmm.qmm_matmul(synth.Q4_0, dec_w[i][r], M, K, dec_x[i], 1, dec_y[i], stream=stream))
        ops["decode"], launches_per_pass["decode"] = op_decode, len(DECODE_SHAPES)
    if "lmhead" in only:
        # one copy: 431 MB alone is more than three times L2
        head_w = torch.from_numpy(synth.gen_weights(synth.Q6_K, Mh, Kh, "bench-lmhead")).to(dev)
        head_x = torch.from_numpy(synth.gen_x(Nh, Kh, "bench-lmhead")).to(dev)
        head_y = torch.empty(Nh, Mh, device=dev)

        def op_lmhead(r):
            chk(qmm.qmm_matmul(synth.Q6_K, head_w, Mh, Kh, head_x, Nh, head_y, stream=stream))
        ops["lmhead"], launches_per_pass["lmhead"] = op_lmhead, 1
    if "prefill" in only or "prefill_f32" in only:
        pre_w = [make(synth.Q4_K, M, K, f"bench-prefill-{M}x{K}") for (M, K) in PREFILL_SHAPES]
        pre_x = [torch.from_numpy(synth.gen_x(PREFILL_N, K, f"bench-prefill-{K}")).to(dev)
                 for (_, K) in PREFILL_SHAPES]
        pre_y = [torch.empty(PREFILL_N, M, device=dev) for (M, _) in PREFILL_SHAPES]
    if "prefill" in only:
        # bf16 X: the GEMM alone (X in the tensor-core operand type)
        pre_xb = [torch.from_numpy(synth.f32_to_bf16_bits(x.cpu().numpy())).to(dev).view(torch.bfloat16)
                  for x in pre_x]

        def op_prefill(r):
            for i, (M, K) in enumerate(PREFILL_SHAPES):
                chk(qmm.qmm_matmul(synth.Q4_K, pre_w[i][r], M, K, pre_xb[i], PREFILL_N, pre_y[i], stream=stream))
        ops["prefill"], launches_per_pass["prefill"] = op_prefill, len(PREFILL_SHAPES)
    if "prefill_f32" in only:
        pre_ws = [qmm.workspace_for(PREFILL_N, K, x) for x, (_, K) in zip(pre_x, PREFILL_SHAPES)]

        def op_prefill_f32(r):
            for i, (M, K) in enumerate(PREFILL_SHAPES):
                chk(qmm.qmm_matmul(synth.Q4_K, pre_w[i][r], M, K, pre_x[i], PREFILL_N, pre_y[i], pre_ws[i],
                                   stream=stream))
        ops["prefill_f32"], launches_per_pass["prefill_f32"] = op_prefill_f32, 2 * len(PREFILL_SHAPES)
    rot_bytes = R * sum(wbytes(synth.Q4_0, M, K) for M, K in DECODE_SHAPES)
    torch.cuda.synchronize()

    # warm-up outside capture (also sets kernel attributes): one pass per copy
    with torch.cuda.stream(stream):
        for r in range(R):
            for f in ops.values():
                f(r)
    torch.cuda.synchronize()

    # One CUDA graph per op over all R copies (step s uses copy s % R), plus
    # one over the first K % R copies, so that exactly K steps are timed.
    K_steps = max(1, args.steps)
    full, rem = divmod(K_steps, R)

    def capture(f, passes):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for r in range(passes):
                f(r)
        return g

    graphs = {name: (capture(f, R), capture(f, rem) if rem else None) for name, f in ops.items()}
    torch.cuda.synchronize()

    def replay(g):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            g.replay()
            b.record(stream)
        return a, b

    warm_replays = max(1, -(-max(args.warmup, 3) // R))
    for _ in range(warm_replays):
        for name in graphs:
            replay(graphs[name][0])
    torch.cuda.synchronize()

    # ---- timed region: exactly K steps; each step = one pass of every op ----
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clk = Clocks(local)
    clk.start()
    time.sleep(0.3)
    events = {name: [] for name in graphs}
    t0 = time.perf_counter()
    for _ in range(full):
        for name in graphs:
            events[name].append((replay(graphs[name][0]), R))
    if rem:
        for name in graphs:
            events[name].append((replay(graphs[name][1]), rem))
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    clocks = clk.stop()
    if world > 1:
        torch.distributed.barrier()

    med = {}      # ms per pass (one step of that op), total event time / K
    for name, evs in events.items():
        med[name] = sum(a.elapsed_time(b) for (a, b), _ in evs) / K_steps
    steps_timed = K_steps
    med = max_over_ranks(med, world, dev)      # the slowest rank sets the aggregate
    ms_step = sum(med.values())

    dec_bytes = sum(alg_bytes(synth.Q4_0, M, K, 1, 4) for M, K in DECODE_SHAPES)
    head_bytes = alg_bytes(synth.Q6_K, Mh, Kh, Nh, 4)
    pre_flops = sum(2.0 * M * K * PREFILL_N for M, K in PREFILL_SHAPES)
    decode_gbs = dec_bytes / (med["decode"] * 1e-3) / 1e9 * world if "decode" in med else None
    head_gbs = head_bytes / (med["lmhead"] * 1e-3) / 1e9 * world if "lmhead" in med else None
    pre_tflops = pre_flops / (med["prefill"] * 1e-3) / 1e12 * world if "prefill" in med else None
    pre32_tflops = pre_flops / (med["prefill_f32"] * 1e-3) / 1e12 * world if "prefill_f32" in med else None

    # dominant kernel of the step -> roofline object
    shares = {k: v / sum(med.values()) for k, v in med.items()}
    dom = max(shares, key=shares.get)
    if dom in ("prefill", "prefill_f32"):
        tf = pre_tflops if dom == "prefill" else pre32_tflops
        roof = {"bound": "tensor", "achieved": round(tf, 1), "peak": bf16_peak, "unit": "TFLOP/s",
                "frac": round(tf / bf16_peak, 4), "traffic": traffic_for(dom),
                "kernel": "gemm_tc (Q4_K, N=512)" + ("" if dom == "prefill" else " + x_to_bf16"),
                "peak_source": f"bf16_tflops ({peak_src})"}
    elif dom == "lmhead":
        roof = {"bound": "hbm", "achieved": round(head_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(head_gbs / hbm_peak, 4), "traffic": traffic_for("lmhead"),
                "kernel": "gemv_mma (Q6_K 128256x4096, N=8)", "peak_source": f"hbm_gbs ({peak_src})"}
    else:
        roof = {"bound": "hbm", "achieved": round(decode_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(decode_gbs / hbm_peak, 4), "traffic": traffic_for("decode"),
                "kernel": "gemv_mma (Q4_0, N=1)", "peak_source": f"hbm_gbs ({peak_src})"}

    # ---- end to end: host X in, host Y out, through qmm_matmul_host ----
    e2e = None
    if not args.no_e2e and "decode" in ops:
        xh = [torch.from_numpy(synth.gen_x(1, K, f"bench-decode-{K}")).pin_memory() for (_, K) in DECODE_SHAPES]
        yh = [torch.empty(1, M).pin_memory() for (M, _) in DECODE_SHAPES]
        xd = [torch.empty(1, K, device=dev) for (_, K) in DECODE_SHAPES]
        yd = [torch.empty(1, M, device=dev) for (M, _) in DECODE_SHAPES]

        def e2e_pass(r):
            for i, (M, K) in enumerate(DECODE_SHAPES):
                chk(qmm.qmm_matmul_host(synth.Q4_0, dec_w[i][r], M, K, xh[i], 1, yh[i], xd[i], yd[i],
                                        stream=stream))
        with torch.cuda.stream(stream):
            for r in range(R):
                e2e_pass(r)
        stream.synchronize()
        g = capture(e2e_pass, R)
        ts = []
        for _ in range(max(3, full)):
            a, b = replay(g)
            stream.synchronize()
            ts.append(a.elapsed_time(b) / R)
        t_e2e = statistics.median(ts)
        e2e = {"value": round(dec_bytes / (t_e2e * 1e-3) / 1e9 * world, 1), "unit": "GB/s",
               "h2d_bytes_per_step": sum(K * 4 for _, K in DECODE_SHAPES),
               "d2h_bytes_per_step": sum(M * 4 for M, _ in DECODE_SHAPES),
               "ms_per_step": round(t_e2e, 5),
               "path": "qmm_matmul_host (pinned host X -> device, GEMV, device Y -> pinned host)"}

    launches = steps_timed * sum(launches_per_pass.values())
    r1 = lambda v, nd=1: None if v is None else round(v, nd)    # noqa: E731
    value = decode_gbs if decode_gbs is not None else (head_gbs if head_gbs is not None else pre_tflops)
    line = {
        "metric": METRIC,
        "value": r1(value),
        "unit": "GB/s" if (decode_gbs is not None or head_gbs is not None) else "TFLOP/s",
        "n_gpus": world,
        "steps": steps_timed,
        "warmup": max(args.warmup, 3),
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32 (GEMV); bf16 x bf16 -> f32 (GEMM)",
        "data": "synthetic (seeded random blocks and N(0,1) activations)",
        "config": {"workload": WORKLOAD if len(ops) == 3 else f"subset: {sorted(ops)}",
                   "decode_N": 1, "lmhead_N": Nh, "prefill_N": PREFILL_N,
                   "weight_copies": R, "static_weights": not args.no_static_weights, "rotating_bytes": rot_bytes, "l2_bytes": l2,
                   "l2_policy": f"inputs larger than L2: {R} rotating weight copies ({rot_bytes / 2**20:.0f} MiB "
                                f"for the decode shapes); the 431 MB LM head alone exceeds L2"},
        "step_share": {k: round(v, 4) for k, v in shares.items()},
        "roofline": roof,
        "cpu_baseline": None,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
        "wall_s_timed": round(wall, 3),
    }
    if decode_gbs is not None:
        line["decode"] = {"GBps": r1(decode_gbs), "frac_of_measured_hbm": round(decode_gbs / hbm_peak, 4),
                          "frac_of_nominal_8TBps": round(decode_gbs / NOMINAL_HBM_GBS, 4),
                          "us_per_pass": round(med["decode"] * 1e3, 3),
                          "per_shape_bytes": [alg_bytes(synth.Q4_0, M, K, 1, 4) for M, K in DECODE_SHAPES]}
    if head_gbs is not None:
        line["lmhead"] = {"GBps": r1(head_gbs), "frac_of_measured_hbm": round(head_gbs / hbm_peak, 4),
                          "us": round(med["lmhead"] * 1e3, 3), "N": Nh}
    if pre_tflops is not None:
        line["prefill"] = {"TFLOPs": r1(pre_tflops), "frac_of_measured_bf16": round(pre_tflops / bf16_peak, 4),
                           "us": round(med["prefill"] * 1e3, 3), "N": PREFILL_N, "x": "bf16",
                           "includes": "tensor-core GEMM"}
    if pre32_tflops is not None:
        line["prefill_f32"] = {"TFLOPs": r1(pre32_tflops), "frac_of_measured_bf16": round(pre32_tflops / bf16_peak, 4),
                               "us": round(med["prefill_f32"] * 1e3, 3), "N": PREFILL_N, "x": "f32",
                               "includes": "f32->bf16 conversion of X + tensor-core GEMM"}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


# ---------------------------------------------------------------------------
# Oracle arm (CPU baseline and --impl reference)
# ---------------------------------------------------------------------------
def cpu_sample_rows(M, frac):
    n = max(1, int(M * frac))
    return np.linspace(0, M - 1, n).astype(np.int64)


def cpu_baseline(seconds):
    """Time the oracle on the host cores on a bounded sample of the decode
    workload (a row subset of each shape, N=1), in the same GB/s unit."""
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    data = []
    for (M, K) in DECODE_SHAPES:
        w = synth.gen_weights(synth.Q4_0, M, K, f"bench-decode-{M}x{K}")
        x = synth.gen_x(1, K, f"bench-decode-{K}")
        data.append((M, K, w, x))
    # calibrate the row fraction so one pass takes ~seconds/3
    frac = 0.02
    t0 = time.perf_counter()
    for M, K, w, x in data:
        oracle.matmul(synth.Q4_0, w, M, K, x, rows=cpu_sample_rows(M, frac))
    t1 = time.perf_counter() - t0
    frac = min(1.0, frac * max(1.0, (seconds / 3) / max(t1, 1e-3)))
    tot_bytes, tot_t, passes = 0.0, 0.0, 0
    while tot_t < seconds and passes < 10000:
        for M, K, w, x in data:
            rows = cpu_sample_rows(M, frac)
            t0 = time.perf_counter()
            oracle.matmul(synth.Q4_0, w, M, K, x, rows=rows)
            tot_t += time.perf_counter() - t0
            tot_bytes += rows.size * synth.row_bytes(synth.Q4_0, K) + K * 4 + rows.size * 4
        passes += 1
    return {"value": round(tot_bytes / tot_t / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{passes} pass(es) over {frac * 100:.2f}% of the rows of each Q4_0 decode shape, N=1; "
                      f"{tot_t:.1f} s of oracle time (C, f64, {cores} threads)"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cpu = cpu_baseline(args.cpu_seconds)
    steps = max(args.steps, 1)
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": cpu["value"],
        "unit": "GB/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": None,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded random blocks and N(0,1) activations)",
        "config": {"workload": WORKLOAD},
        "cpu_baseline": cpu,
        "e2e": {"value": cpu["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--copies", type=int, default=8, help="rotating weight copies (inputs > L2)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-static-weights", action="store_true",
                    help="launch every call only after the preceding kernel has finished")
    ap.add_argument("--only", default="",
                    help="comma list of ops to run (decode,lmhead,prefill,prefill_f32); default all")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
