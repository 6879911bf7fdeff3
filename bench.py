#!/usr/bin/env python3
"""Benchmark of the block-quantized projection matmul on GB300.

Headline: the Q4_0 decode GEMV at N=1 on the Llama-3-8B projection shapes
(M,K) = (4096,4096), (1024,4096), (14336,4096), (4096,14336); `value` is its
effective HBM bandwidth (algorithmic bytes / device time, GB/s).

One timed step runs the whole hot path once over one batch of synthetic input:
  decode       4 x Q4_0 GEMV, N=1 (one CUDA graph per shape)   decode GEMV
  lmhead       Q6_K 128256 x 4096 LM head, N=8, f32 X          small-N GEMV
  prefill      Q4_K 4096x4096 and 14336x4096, N=512, bf16 X    tcgen05 GEMM
  prefill_f32  the same with f32 X (x -> bf16 + GEMM)
Weights are replicated into R device copies whose total exceeds L2, and
step s uses copy s % R (inputs larger than L2 instead of a flush).  Each op is
a CUDA graph over all R copies, timed with CUDA events on the launching
stream.

After the timed steps (outside the step time) the other workloads are timed
the same way and reported under "workloads": the Q8_0 256x512 GEMV, the
Q4_K prefill at N = 64 and 256, the LM head at N = 1 and 4, and the 32-layer
decoder sweep (224 projections, one graph per N, tokens/s).  Every op's
output is then checked on sampled rows against the oracle.

Multi-GPU (torchrun, one rank per GPU, NCCL): each rank owns a row slice of
every weight matrix (the LM head: a vocabulary slice), X is replicated, no
collective runs on the data path unless --allgather asks for Y to be
gathered.  --scaling weak (default): per-GPU rows fixed at the single-GPU
shapes (the global matrices have G x M rows); --scaling strong: the global
shapes are the single-GPU ones, split G ways.

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
from block_quantized_gemv_gguf_gb300.shard import row_partition  # noqa: E402

DECODE_SHAPES = [(4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336)]
LMHEAD = (128256, 4096, 8)
PREFILL_SHAPES = [(4096, 4096), (14336, 4096)]
PREFILL_N = 512
METRIC = "decode GEMV effective HBM GB/s (% of 8 TB/s); prefill N=512 GEMM TFLOP/s (% peak)"
WORKLOAD = ("Q4_0 decode GEMV N=1 on Llama-3-8B projection shapes (4096,4096) (1024,4096) (14336,4096) "
            "(4096,14336); same step also runs the Q6_K 128256x4096 LM head at N=8 and the Q4_K "
            "(4096,4096)+(14336,4096) prefill GEMM at N=512 with bf16 X and with f32 X")
NOMINAL_HBM_GBS = 8000.0
ALL_OPS = ("decode", "lmhead", "prefill", "prefill_f32")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# DRAM bytes (read + write) per launch of the dominant kernels, from one ncu
# capture each (dram__bytes_read.sum + dram__bytes_write.sum), keyed by the
# sha256 of the kernel sources they were taken on: any source change since
# the capture turns the figure into null.
TRAFFIC = {
    # kernel sources 865a33c78cf96faa: the launch list of `bench.py --steps 8 --copies 2 --no-extras` under ncu
    "decode": ("865a33c78cf96faa", 78_156_000),       # 4 launches of the streaming GEMV
    "lmhead": ("865a33c78cf96faa", 452_213_000),      # ring GEMV, Q6_K 128256x4096, N=8
    "prefill": ("865a33c78cf96faa", 55_158_000),      # 3 GEMM launches (bf16 X)
    "prefill_f32": ("865a33c78cf96faa", 71_933_000),  # 2 conversions + 3 GEMM launches
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
    """Algorithmic bytes of one call: weights + X + Y."""
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
# multi-rank helpers
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


def local_rows(M, world, rank, scaling, align=16):
    """(r0, r1) of the global matrix this rank owns, and the global M."""
    if world <= 1:
        return 0, M, M
    if scaling == "weak":
        Mg = M * world
        return rank * M, (rank + 1) * M, Mg
    r0, r1 = row_partition(M, world, rank, align)
    return r0, r1, M


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
class Timer:
    """CUDA graph of `passes` passes of f over rotating inputs; replays timed
    with CUDA events on the launching stream."""

    def __init__(self, torch, stream, f, passes, counter=None):
        self.torch, self.stream, self.passes = torch, stream, passes
        self.g = torch.cuda.CUDAGraph()
        n0 = counter() if counter else 0
        with torch.cuda.graph(self.g, stream=stream):
            for r in range(passes):
                f(r)
        # library kernels recorded into the graph, per pass
        self.launches = (counter() - n0) / passes if counter else None

    def replay(self):
        t = self.torch
        a, b = t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)
        with t.cuda.stream(self.stream):
            a.record(self.stream)
            self.g.replay()
            b.record(self.stream)
        return a, b

    def median_ms(self, reps):
        evs = [self.replay() for _ in range(reps)]
        self.torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in evs) / self.passes


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
    stream = torch.cuda.Stream(device=dev)

    only = set(args.only.split(",")) if args.only else set(ALL_OPS)
    bad = only - set(ALL_OPS)
    if bad:
        raise SystemExit(f"unknown op(s) in --only: {sorted(bad)}")

    def chk(s):
        if s != qmm.OK:
            raise RuntimeError(qmm.status_name(s))

    def gen_rows(wt, M, K, name, r0, r1, Mg):
        """Rows [r0, r1) of the global matrix (Mg rows) `name`, host bytes.
        Weak scaling: each rank's slice is its own seeded draw (the global
        matrix is the concatenation); strong: a slice of the single-GPU matrix."""
        if Mg == M and r0 == 0 and r1 == M:
            return synth.gen_weights(wt, M, K, name)
        if args.scaling == "weak":
            return synth.gen_weights(wt, r1 - r0, K, f"{name}/rows{r0}-{r1}")
        full = synth.gen_weights(wt, Mg, K, name)
        rb = synth.row_bytes(wt, K)
        return full[r0 * rb:r1 * rb].copy()

    def copies(w):
        t = torch.from_numpy(w).to(dev)
        return [t] + [t.clone() for _ in range(R - 1)]

    # ---- inputs of the timed step (this rank's rows) ----
    ops, launches_per_pass, host = {}, {}, {}
    Mh, Kh, Nh = LMHEAD
    if "decode" in only:
        dec = []
        for (M, K) in DECODE_SHAPES:
            r0, r1, Mg = local_rows(M, world, rank, args.scaling)
            w = gen_rows(synth.Q4_0, M, K, f"bench-decode-{M}x{K}", r0, r1, Mg)
            x = synth.gen_x(1, K, f"bench-decode-{K}")
            dec.append(dict(M=r1 - r0, K=K, Mg=Mg, w=w, W=copies(w), x=x, X=torch.from_numpy(x).to(dev),
                            Y=torch.empty(1, r1 - r0, device=dev)))
        for i, d in enumerate(dec):
            def op(r, d=d):
                chk(qmm.qmm_matmul(synth.Q4_0, d["W"][r], d["M"], d["K"], d["X"], 1, d["Y"], stream=stream))
            ops[f"decode{i}"] = op
        host["decode"] = dec
    if "lmhead" in only:
        r0, r1, Mg = local_rows(Mh, world, rank, args.scaling)
        w = gen_rows(synth.Q6_K, Mh, Kh, "bench-lmhead", r0, r1, Mg)
        x = synth.gen_x(Nh, Kh, "bench-lmhead")
        hd = dict(M=r1 - r0, w=w, W=torch.from_numpy(w).to(dev), x=x, X=torch.from_numpy(x).to(dev),
                  Y=torch.empty(Nh, r1 - r0, device=dev))

        def op_lmhead(r, hd=hd):   # one copy: 431 MB alone is more than three times L2
            chk(qmm.qmm_matmul(synth.Q6_K, hd["W"], hd["M"], Kh, hd["X"], Nh, hd["Y"], stream=stream))
        ops["lmhead"] = op_lmhead
        host["lmhead"] = hd
    if "prefill" in only or "prefill_f32" in only:
        pre = []
        for (M, K) in PREFILL_SHAPES:
            r0, r1, Mg = local_rows(M, world, rank, args.scaling)
            w = gen_rows(synth.Q4_K, M, K, f"bench-prefill-{M}x{K}", r0, r1, Mg)
            x = synth.gen_x(PREFILL_N, K, f"bench-prefill-{K}")
            xb = synth.f32_to_bf16_bits(x)
            X = torch.from_numpy(x).to(dev)
            pre.append(dict(M=r1 - r0, K=K, w=w, W=copies(w), x=x, X=X, xb=xb,
                            XB=torch.from_numpy(xb).to(dev).view(torch.bfloat16),
                            ws=qmm.workspace_for(PREFILL_N, K, X),
                            Y=torch.empty(PREFILL_N, r1 - r0, device=dev),
                            Y32=torch.empty(PREFILL_N, r1 - r0, device=dev)))
        host["prefill"] = pre
        if "prefill" in only:
            def op_prefill(r):
                for p in pre:
                    chk(qmm.qmm_matmul(synth.Q4_K, p["W"][r], p["M"], p["K"], p["XB"], PREFILL_N, p["Y"],
                                       stream=stream))
            ops["prefill"] = op_prefill
        if "prefill_f32" in only:
            def op_prefill_f32(r):
                for p in pre:
                    chk(qmm.qmm_matmul(synth.Q4_K, p["W"][r], p["M"], p["K"], p["X"], PREFILL_N, p["Y32"], p["ws"],
                                       stream=stream))
            ops["prefill_f32"] = op_prefill_f32
    allgather = None
    if args.allgather and world > 1 and "decode" in only:
        # the row slices of every decode output, gathered on every rank
        gat = [torch.empty(world, d["M"], device=dev) for d in host["decode"]]

        def op_gather(r):
            for d, g in zip(host["decode"], gat):
                torch.distributed.all_gather_into_tensor(g, d["Y"].view(-1))
        allgather = op_gather
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
    graphs = {name: (Timer(torch, stream, f, R, qmm.qmm_kernel_launches), Timer(torch, stream, f, rem) if rem else None)
              for name, f in ops.items()}
    # launches per pass as the library counted them while the graphs were recorded
    for name in graphs:
        n = graphs[name][0].launches
        if n != int(n) or n < 1:
            raise RuntimeError(f"{name}: {n} library launches per pass")
        launches_per_pass[name] = int(n)
    torch.cuda.synchronize()
    warm_replays = max(1, -(-max(args.warmup, 3) // R))
    for _ in range(warm_replays):
        for name in graphs:
            graphs[name][0].replay()
    torch.cuda.synchronize()

    # ---- timed region: exactly K steps; each step = one pass of every op ----
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clk = Clocks(local)
    clk.start()
    time.sleep(0.3)
    events = {name: [] for name in graphs}
    gather_ev = []
    t0 = time.perf_counter()
    for _ in range(full):
        for name in graphs:
            events[name].append(graphs[name][0].replay())
        if allgather:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(R):
                allgather(0)
            b.record()
            gather_ev.append((a, b, R))
    if rem:
        for name in graphs:
            events[name].append(graphs[name][1].replay())
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    clocks = clk.stop()
    if world > 1:
        torch.distributed.barrier()

    med = {}      # ms per step of each op (total event time / K)
    for name, evs in events.items():
        med[name] = sum(a.elapsed_time(b) for a, b in evs) / K_steps
    if gather_ev:
        med["allgather"] = sum(a.elapsed_time(b) / n for a, b, n in gather_ev) / len(gather_ev)
    med = max_over_ranks(med, world, dev)      # the slowest rank sets the aggregate
    ms_step = sum(med.values())

    # aggregate algorithmic work over all ranks (global shapes)
    dec_shape_bytes, dec_t = [], []
    if "decode" in only:
        for i, d in enumerate(host["decode"]):
            Mt = d["M"] * world if args.scaling == "weak" else d["Mg"]
            dec_shape_bytes.append(alg_bytes(synth.Q4_0, Mt, d["K"], 1, 4))
            dec_t.append(med[f"decode{i}"])
        med_decode = sum(dec_t)
    dec_bytes = sum(dec_shape_bytes)
    g_lm = Mh * (world if args.scaling == "weak" else 1)
    head_bytes = alg_bytes(synth.Q6_K, g_lm, Kh, Nh, 4)
    pre_flops = sum(2.0 * M * K * PREFILL_N for M, K in PREFILL_SHAPES) * (world if args.scaling == "weak" else 1)
    decode_gbs = dec_bytes / (med_decode * 1e-3) / 1e9 if dec_bytes else None
    head_gbs = head_bytes / (med["lmhead"] * 1e-3) / 1e9 if "lmhead" in med else None
    pre_tflops = pre_flops / (med["prefill"] * 1e-3) / 1e12 if "prefill" in med else None
    pre32_tflops = pre_flops / (med["prefill_f32"] * 1e-3) / 1e12 if "prefill_f32" in med else None

    # ---- other workloads (outside the step time) ----
    workloads = {} if (args.no_extras or world > 1) else run_workloads(torch, qmm, stream, dev, args, chk)

    # ---- output check on sampled rows against the oracle ----
    check = None if args.no_check else check_outputs(host, Nh, Kh)

    # per-op rows for the step
    step_ops = {}
    if "decode" in only:
        step_ops["decode"] = med_decode
    for k in ("lmhead", "prefill", "prefill_f32", "allgather"):
        if k in med:
            step_ops[k] = med[k]
    shares = {k: v / sum(step_ops.values()) for k, v in step_ops.items()}
    dom = max(shares, key=shares.get)
    gpu_share = {"decode": "gemv_stream_kernel (Q4_0, N=1, 4 shapes)",
                 "lmhead": "gemv_mma_kernel (Q6_K 128256x4096, N=8)",
                 "prefill": "gemm_tc_kernel (Q4_K, N=512, bf16 X)",
                 "prefill_f32": "x_to_bf16_kernel + gemm_tc_kernel (Q4_K, N=512)"}
    if dom in ("prefill", "prefill_f32"):
        tf = pre_tflops if dom == "prefill" else pre32_tflops
        roof = {"bound": "tensor", "achieved": round(tf, 1), "peak": bf16_peak, "unit": "TFLOP/s",
                "frac": round(tf / bf16_peak, 4), "traffic": traffic_for(dom), "kernel": gpu_share[dom],
                "peak_source": f"bf16_tflops ({peak_src})"}
    elif dom == "lmhead":
        roof = {"bound": "hbm", "achieved": round(head_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(head_gbs / hbm_peak, 4), "traffic": traffic_for("lmhead"),
                "kernel": gpu_share["lmhead"], "peak_source": f"hbm_gbs ({peak_src})"}
    else:
        roof = {"bound": "hbm", "achieved": round(decode_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(decode_gbs / hbm_peak, 4), "traffic": traffic_for("decode"),
                "kernel": gpu_share["decode"], "peak_source": f"hbm_gbs ({peak_src})"}

    # ---- end to end: host X in, host Y out, through qmm_matmul_host ----
    e2e = None
    if not args.no_e2e and "decode" in only:
        dd = host["decode"]
        xh = [torch.from_numpy(d["x"]).pin_memory() for d in dd]
        yh = [torch.empty(1, d["M"]).pin_memory() for d in dd]
        xd = [torch.empty(1, d["K"], device=dev) for d in dd]
        yd = [torch.empty(1, d["M"], device=dev) for d in dd]

        def e2e_pass(r):
            for i, d in enumerate(dd):
                chk(qmm.qmm_matmul_host(synth.Q4_0, d["W"][r], d["M"], d["K"], xh[i], 1, yh[i], xd[i], yd[i],
                                        stream=stream))
        with torch.cuda.stream(stream):
            for r in range(R):
                e2e_pass(r)
        stream.synchronize()
        tm = Timer(torch, stream, e2e_pass, R)
        t_e2e = tm.median_ms(max(5, full))
        t_e2e = max_over_ranks({"e2e": t_e2e}, world, dev)["e2e"]
        e2e = {"value": round(dec_bytes / (t_e2e * 1e-3) / 1e9, 1), "unit": "GB/s",
               "h2d_bytes_per_step": sum(d["K"] * 4 for d in dd),
               "d2h_bytes_per_step": sum(d["M"] * 4 for d in dd),
               "ms_per_step": round(t_e2e, 5),
               "path": "qmm_matmul_host (pinned host X -> device, GEMV, device Y -> pinned host)"}

    launches = K_steps * sum(launches_per_pass.values())
    r1 = lambda v, nd=1: None if v is None else round(v, nd)    # noqa: E731
    value = decode_gbs if decode_gbs is not None else (head_gbs if head_gbs is not None else pre_tflops)
    full_run = only == set(ALL_OPS)
    line = {
        "metric": METRIC,
        "value": r1(value),
        "unit": "GB/s" if (decode_gbs is not None or head_gbs is not None) else "TFLOP/s",
        "n_gpus": world,
        "steps": K_steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": args.scaling if world > 1 else "weak",
        "vs_baseline": None,
        "dtype": "f32 (GEMV); bf16 x bf16 -> f32 (GEMM)",
        "data": "synthetic (seeded random blocks and N(0,1) activations)",
        "config": {"workload": WORKLOAD if full_run else f"subset: {sorted(only)}",
                   "decode_N": 1, "lmhead_N": Nh, "prefill_N": PREFILL_N,
                   "weight_copies": R, "static_weights": not args.no_static_weights,
                   "l2_bytes": l2,
                   "l2_policy": f"inputs larger than L2: {R} rotating device copies of every decode and prefill "
                                f"weight matrix; the 431 MB LM head alone exceeds L2",
                   "parallelism": f"row-sharded x{world} ({args.scaling})" if world > 1 else "1 GPU",
                   "allgather": bool(allgather)},
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
                          "us_per_step": round(med_decode * 1e3, 3),
                          "per_shape": [{"M": M, "K": K, "us": round(t * 1e3, 3), "bytes": b,
                                         "GBps": round(b / (t * 1e-3) / 1e9, 1),
                                         "frac_of_measured_hbm": round(b / (t * 1e-3) / 1e9 / hbm_peak, 4)}
                                        for (M, K), t, b in zip(DECODE_SHAPES, dec_t, dec_shape_bytes)]}
    if head_gbs is not None:
        line["lmhead"] = {"GBps": r1(head_gbs), "frac_of_measured_hbm": round(head_gbs / hbm_peak, 4),
                          "us": round(med["lmhead"] * 1e3, 3), "N": Nh}
    if pre_tflops is not None:
        line["prefill"] = {"TFLOPs": r1(pre_tflops), "frac_of_measured_bf16": round(pre_tflops / bf16_peak, 4),
                           "frac_of_sustained_bf16": round(pre_tflops / bf16_sus, 4) if bf16_sus else None,
                           "us": round(med["prefill"] * 1e3, 3), "N": PREFILL_N, "x": "bf16",
                           "includes": "tensor-core GEMM"}
    if pre32_tflops is not None:
        line["prefill_f32"] = {"TFLOPs": r1(pre32_tflops), "frac_of_measured_bf16": round(pre32_tflops / bf16_peak, 4),
                               "us": round(med["prefill_f32"] * 1e3, 3), "N": PREFILL_N, "x": "f32",
                               "includes": "f32->bf16 conversion of X + tensor-core GEMM"}
    if "allgather" in med:
        line["allgather_us"] = round(med["allgather"] * 1e3, 3)
    if workloads:
        line["workloads"] = workloads
    if check is not None:
        line["output_check"] = check
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    if check is not None and not check["pass"]:
        raise SystemExit("output check against the oracle failed")


def run_workloads(torch, qmm, stream, dev, args, chk):
    """The other configurations: timed like the step (graphs over rotating
    copies), outside the step time."""
    hbm_peak, bf16_peak, _, _ = peaks()
    out = {}
    R = args.copies

    def timed(f, passes, reps=20):
        with torch.cuda.stream(stream):
            for r in range(passes):
                f(r)
        torch.cuda.synchronize()
        tm = Timer(torch, stream, f, passes)
        for _ in range(2):
            tm.replay()
        return tm.median_ms(reps)

    # Q8_0 256x512, N=1: 139 KB, latency-bound (L2-resident copies)
    wt, M, K = synth.Q8_0, 256, 512
    w = torch.from_numpy(synth.gen_weights(wt, M, K, "bench-q8")).to(dev)
    Ws = [w] + [w.clone() for _ in range(63)]
    X = torch.from_numpy(synth.gen_x(1, K, "bench-q8")).to(dev)
    Y = torch.empty(1, M, device=dev)
    t = timed(lambda r: chk(qmm.qmm_matmul(wt, Ws[r], M, K, X, 1, Y, stream=stream)), 64)
    b = alg_bytes(wt, M, K, 1, 4)
    out["q8_0_256x512_n1"] = {"us": round(t * 1e3, 3), "GBps": round(b / (t * 1e-3) / 1e9, 1),
                              "note": "latency-bound: 142 KB per call, copies stay in L2"}

    # Q4_K prefill at N = 64 and 256, bf16 X
    pre = {}
    for (M, K) in PREFILL_SHAPES:
        w = torch.from_numpy(synth.gen_weights(synth.Q4_K, M, K, f"bench-prefill-{M}x{K}")).to(dev)
        pre[(M, K)] = [w] + [w.clone() for _ in range(R - 1)]
    for N in (64, 256):
        res = []
        for (M, K) in PREFILL_SHAPES:
            x = synth.gen_x(N, K, f"bench-prefill-{K}")
            XB = torch.from_numpy(synth.f32_to_bf16_bits(x)).to(dev).view(torch.bfloat16)
            Y = torch.empty(N, M, device=dev)
            Ws = pre[(M, K)]
            t = timed(lambda r: chk(qmm.qmm_matmul(synth.Q4_K, Ws[r], M, K, XB, N, Y, stream=stream)), R)
            fl = 2.0 * M * K * N
            by = alg_bytes(synth.Q4_K, M, K, N, 2)
            res.append({"M": M, "K": K, "us": round(t * 1e3, 3), "TFLOPs": round(fl / (t * 1e-3) / 1e12, 1),
                        "frac_of_measured_bf16": round(fl / (t * 1e-3) / 1e12 / bf16_peak, 4),
                        "GBps": round(by / (t * 1e-3) / 1e9, 1),
                        "frac_of_measured_hbm": round(by / (t * 1e-3) / 1e9 / hbm_peak, 4)})
        out[f"q4_k_prefill_n{N}"] = res
    del pre

    # LM head at N = 1 and 4
    Mh, Kh, _ = LMHEAD
    w = torch.from_numpy(synth.gen_weights(synth.Q6_K, Mh, Kh, "bench-lmhead")).to(dev)
    for N in (1, 4):
        X = torch.from_numpy(synth.gen_x(N, Kh, "bench-lmhead")).to(dev)
        Y = torch.empty(N, Mh, device=dev)
        t = timed(lambda r: chk(qmm.qmm_matmul(synth.Q6_K, w, Mh, Kh, X, N, Y, stream=stream)), 1, reps=10)
        b = alg_bytes(synth.Q6_K, Mh, Kh, N, 4)
        out[f"q6_k_lmhead_n{N}"] = {"us": round(t * 1e3, 3), "GBps": round(b / (t * 1e-3) / 1e9, 1),
                                    "frac_of_measured_hbm": round(b / (t * 1e-3) / 1e9 / hbm_peak, 4)}
    del w

    out["next_rows"] = run_next_rows(torch, qmm, dev, R, chk, timed)

    if not args.no_sweep:
        out["decoder_sweep"] = run_sweep(torch, qmm, stream, dev, args, chk)
        out["gemv_gemm_crossover"] = run_crossover(torch, qmm, stream, dev, args, chk)
    return out


def run_next_rows(torch, qmm, dev, R, chk, timed):
    """The fused and alternative entry points against their unfused or
    default counterparts, timed the same way (graphs over R rotating weight
    copies; the LM head is one copy, larger than L2)."""
    def us(t):
        return round(t * 1e3, 3)

    def copies(wt, M, K, name):
        w = torch.from_numpy(synth.gen_weights(wt, M, K, name)).to(dev)
        return [w] + [w.clone() for _ in range(R - 1)]

    res = {}
    K = 4096
    x1 = torch.from_numpy(synth.gen_x(1, K, "next-x1")).to(dev)

    # F2: Q/K/V (Q4_K 4096 + 1024 + 1024 rows), N = 1, one launch vs three
    qkv = [(copies(synth.Q4_K, M, K, f"next-{n}"), M) for n, M in (("q", 4096), ("k", 1024), ("v", 1024))]
    Ys = [torch.empty(1, M, device=dev) for _, M in qkv]
    fused = timed(lambda r: chk(qmm.qmm_gemv_multi(synth.Q4_K, [(W[r], M, Y) for (W, M), Y in zip(qkv, Ys)], K, x1, 1,
                                                   stream=torch.cuda.current_stream())), R)
    sep = timed(lambda r: [chk(qmm.qmm_gemv(synth.Q4_K, W[r], M, K, x1, 1, Y, stream=torch.cuda.current_stream()))
                           for (W, M), Y in zip(qkv, Ys)], R)
    res["f2_qkv_gemv_q4_k_n1"] = {"fused_us": us(fused), "three_calls_us": us(sep)}
    del qkv

    # F2: gate/up + SwiGLU (Q4_K 2 x 14336 rows), N = 1 and N = 512
    M = 14336
    g, u = copies(synth.Q4_K, M, K, "next-gate"), copies(synth.Q4_K, M, K, "next-up")
    Y1 = torch.empty(1, M, device=dev)
    ws1 = torch.empty(2 * M, dtype=torch.float32, device=dev)
    Yg, Yu = torch.empty(1, M, device=dev), torch.empty(1, M, device=dev)
    fused = timed(lambda r: chk(qmm.qmm_gemv_swiglu(synth.Q4_K, g[r], u[r], M, K, x1, 1, Y1, ws1,
                                                    stream=torch.cuda.current_stream())), R)
    sep = timed(lambda r: (chk(qmm.qmm_gemv(synth.Q4_K, g[r], M, K, x1, 1, Yg, stream=torch.cuda.current_stream())),
                           chk(qmm.qmm_gemv(synth.Q4_K, u[r], M, K, x1, 1, Yu, stream=torch.cuda.current_stream()))), R)
    res["f2_gate_up_swiglu_gemv_q4_k_n1"] = {"fused_us": us(fused), "two_gemvs_us": us(sep)}
    N = 512
    xb = torch.from_numpy(synth.f32_to_bf16_bits(synth.gen_x(N, K, "next-x512"))).to(dev).view(torch.bfloat16)
    Yn = torch.empty(N, M, device=dev)
    wsn = torch.empty(qmm.load().qmm_gemm_swiglu_workspace_bytes(N, M, K, qmm.X_BF16), dtype=torch.uint8, device=dev)
    Ygn, Yun = torch.empty(N, M, device=dev), torch.empty(N, M, device=dev)
    fused = timed(lambda r: chk(qmm.qmm_gemm_swiglu(synth.Q4_K, g[r], u[r], M, K, xb, N, Yn, wsn,
                                                    stream=torch.cuda.current_stream())), R)
    sep = timed(lambda r: (chk(qmm.qmm_gemm(synth.Q4_K, g[r], M, K, xb, N, Ygn, stream=torch.cuda.current_stream())),
                           chk(qmm.qmm_gemm(synth.Q4_K, u[r], M, K, xb, N, Yun, stream=torch.cuda.current_stream()))), R)
    fl = 2 * 2.0 * M * K * N
    res["f2_gate_up_swiglu_gemm_q4_k_n512"] = {"fused_us": us(fused), "two_gemms_us": us(sep),
                                               "fused_TFLOPs": round(fl / (fused * 1e-3) / 1e12, 1)}
    del u

    # F4: Q8_0 activations, GEMV at N = 8 and GEMM at N = 512, against the default paths
    x8 = torch.from_numpy(synth.gen_x(8, K, "next-x8")).to(dev)
    Y8 = torch.empty(8, M, device=dev)
    ws8 = torch.empty(qmm.qmm_q8act_workspace_bytes(8, K), dtype=torch.uint8, device=dev)
    q8 = timed(lambda r: chk(qmm.qmm_gemv_q8act(synth.Q4_K, g[r], M, K, x8, 8, Y8, ws8,
                                                stream=torch.cuda.current_stream())), R)
    dflt = timed(lambda r: chk(qmm.qmm_gemv(synth.Q4_K, g[r], M, K, x8, 8, Y8, stream=torch.cuda.current_stream())), R)
    res["f4_q8act_gemv_q4_k_14336x4096_n8"] = {"q8act_us": us(q8), "f32_gemv_us": us(dflt)}
    x512 = torch.from_numpy(synth.gen_x(N, K, "next-x512")).to(dev)
    wsq = torch.empty(qmm.load().qmm_gemm_q8act_workspace_bytes(N, K), dtype=torch.uint8, device=dev)
    wsf = qmm.workspace_for(N, K, x512)
    q8 = timed(lambda r: chk(qmm.qmm_gemm_q8act(synth.Q4_K, g[r], M, K, x512, N, Yn, wsq,
                                                stream=torch.cuda.current_stream())), R)
    dflt = timed(lambda r: chk(qmm.qmm_gemm(synth.Q4_K, g[r], M, K, x512, N, Yn, wsf,
                                            stream=torch.cuda.current_stream())), R)
    res["f4_q8act_gemm_q4_k_14336x4096_n512"] = {"q8act_us": us(q8), "f32_gemm_us": us(dflt)}
    del g

    # F3: argmax-fused LM head (Q6_K 128256 x 4096), N = 1
    Mh, Kh, _ = LMHEAD
    w = torch.from_numpy(synth.gen_weights(synth.Q6_K, Mh, Kh, "bench-lmhead")).to(dev)
    xh = torch.from_numpy(synth.gen_x(1, Kh, "next-xh")).to(dev)
    idx = torch.empty(1, dtype=torch.int32, device=dev)
    val = torch.empty(1, dtype=torch.float32, device=dev)
    wsa = torch.empty(2, dtype=torch.int64, device=dev)
    Yh = torch.empty(1, Mh, device=dev)
    am = timed(lambda r: chk(qmm.qmm_gemv_argmax(synth.Q6_K, w, Mh, Kh, xh, 1, idx, val, wsa,
                                                 stream=torch.cuda.current_stream())), 1, reps=10)
    gv = timed(lambda r: chk(qmm.qmm_gemv(synth.Q6_K, w, Mh, Kh, xh, 1, Yh, stream=torch.cuda.current_stream())), 1,
               reps=10)
    res["f3_argmax_lmhead_q6_k_n1"] = {"argmax_us": us(am), "gemv_us": us(gv),
                                       "note": "the GEMV also writes 513 KB of logits that the argmax path never stores"}
    return res


def run_crossover(torch, qmm, stream, dev, args, chk):
    """qmm_gemv against qmm_gemm on the seven projections of one decoder layer
    at the token counts around the dispatcher's threshold (R rotating layer
    copies): the evidence for QMM_GEMV_MAX_N."""
    R = max(2, args.copies // 2)
    Ws = [{name: torch.from_numpy(synth.gen_weights(wt, M, K, f"layer{c}.{name}")).to(dev)
           for name, wt, M, K in synth.DECODER_LAYER} for c in range(R)]
    rows = []
    for N in (2, 4, 6, 8, 9, 10, 11, 12, 16, 24, 32):
        X = {K: torch.from_numpy(synth.gen_x(N, K, f"xover-{N}-{K}")).to(dev) for K in (4096, 14336)}
        Ys = {name: torch.empty(N, M, device=dev) for name, _, M, _ in synth.DECODER_LAYER}
        ws = torch.empty(max(qmm.qmm_gemm_workspace_bytes(N, 14336, qmm.X_F32), 16), dtype=torch.uint8, device=dev)
        row = {"N": N}
        for path in ("gemv", "gemm"):
            if path == "gemv" and N > qmm.GEMV_MAX_N:   # the GEMV's own limit
                continue

            def f(r, path=path, N=N, X=X, Ys=Ys, ws=ws):
                for name, wt, M, K in synth.DECODER_LAYER:
                    if path == "gemv":
                        chk(qmm.qmm_gemv(wt, Ws[r][name], M, K, X[K], N, Ys[name], stream=stream))
                    else:
                        chk(qmm.qmm_gemm(wt, Ws[r][name], M, K, X[K], N, Ys[name], ws, stream=stream))
            with torch.cuda.stream(stream):
                for r in range(R):
                    f(r)
            torch.cuda.synchronize()
            tm = Timer(torch, stream, f, R)
            tm.replay()
            row[f"{path}_us"] = round(tm.median_ms(10) * 1e3, 2)
        rows.append(row)
    del Ws
    torch.cuda.empty_cache()
    return {"layer": "7 projections of one decoder layer", "points": rows}


def run_sweep(torch, qmm, stream, dev, args, chk):
    """32-layer decoder sweep: 224 projections (7 per layer, independently
    seeded weights per layer) at each N, one CUDA graph per N; tokens/s =
    N / (time of the 224 matmuls).  X is one N(0,1) draw per (N, K), Y one
    buffer per projection shape."""
    hbm_peak, bf16_peak, _, _ = peaks()
    layers = args.sweep_layers
    W = {}
    for layer in range(layers):
        for name, wt, M, K in synth.DECODER_LAYER:
            W[(layer, name)] = torch.from_numpy(synth.gen_weights(wt, M, K, f"layer{layer}.{name}")).to(dev)
    wtot = sum(wbytes(wt, M, K) for _, wt, M, K in synth.DECODER_LAYER) * layers
    res = []
    for N in synth.DECODER_NS:
        X = {K: torch.from_numpy(synth.gen_x(N, K, f"sweep-{N}-{K}")).to(dev) for K in (4096, 14336)}
        Ys = {name: torch.empty(N, M, device=dev) for name, _, M, _ in synth.DECODER_LAYER}
        ws = torch.empty(max(qmm.qmm_gemm_workspace_bytes(N, 14336, qmm.X_F32), 16), dtype=torch.uint8, device=dev)

        def f(_r, N=N, X=X, Ys=Ys, ws=ws):
            for layer in range(layers):
                for name, wt, M, K in synth.DECODER_LAYER:
                    chk(qmm.qmm_matmul(wt, W[(layer, name)], M, K, X[K], N, Ys[name], ws, stream=stream))
        with torch.cuda.stream(stream):
            f(0)
        torch.cuda.synchronize()
        tm = Timer(torch, stream, f, 1)
        tm.replay()
        t = tm.median_ms(5)
        flops = 2.0 * N * sum(M * K for _, _, M, K in synth.DECODER_LAYER) * layers
        by = wtot + N * 4 * sum(K + M for _, _, M, K in synth.DECODER_LAYER) * layers
        res.append({"N": N, "ms": round(t, 4), "tokens_per_s": round(N / (t * 1e-3), 1),
                    "GBps": round(by / (t * 1e-3) / 1e9, 1), "frac_of_measured_hbm": round(by / (t * 1e-3) / 1e9 / hbm_peak, 4),
                    "TFLOPs": round(flops / (t * 1e-3) / 1e12, 1),
                    "frac_of_measured_bf16": round(flops / (t * 1e-3) / 1e12 / bf16_peak, 4)})
        del X, Ys, ws
    del W
    torch.cuda.empty_cache()
    return {"layers": layers, "projections": 7 * layers, "weight_bytes": wtot, "points": res,
            "aggregate_tokens_per_s": round(sum(p["N"] for p in res) / (sum(p["ms"] for p in res) * 1e-3), 1)}


def check_outputs(host, Nh, Kh):
    """Sampled rows of each op's last output against the oracle's exact sums
    (GEMV bar 1e-5 S + 1e-6 at N <= 16, GEMM bar 2e-3 S + 1e-5)."""
    import oracle
    oracle.build()
    rng = np.random.default_rng(20261202)
    res, ok_all = {}, True

    def one(name, wt, w, M, K, x, y, tol):
        nonlocal ok_all
        rows = np.sort(rng.choice(M, size=min(48, M), replace=False))
        Yr, S = oracle.matmul(wt, w, M, K, x, rows=rows)
        ok, ratio = oracle.within(y[:, rows], Yr, S, *tol)
        ok_all &= bool(ok)
        res[name] = {"rows": int(rows.size), "worst_err_over_tol": float(ratio), "pass": bool(ok)}

    for i, d in enumerate(host.get("decode", [])):
        one(f"decode{i}", synth.Q4_0, d["w"], d["M"], d["K"], d["x"], d["Y"].cpu().numpy(), (1e-5, 1e-6))
    if "lmhead" in host:
        hd = host["lmhead"]
        one("lmhead", synth.Q6_K, hd["w"], hd["M"], Kh, hd["x"], hd["Y"].cpu().numpy(), (1e-5, 1e-6))
    for i, p in enumerate(host.get("prefill", [])):
        one(f"prefill{i}", synth.Q4_K, p["w"], p["M"], p["K"], p["xb"], p["Y"].cpu().numpy(), (2e-3, 1e-5))
        one(f"prefill_f32_{i}", synth.Q4_K, p["w"], p["M"], p["K"], p["x"], p["Y32"].cpu().numpy(), (2e-3, 1e-5))
    return {"pass": ok_all, "ops": res}


# ---------------------------------------------------------------------------
# Oracle arm (CPU baseline and --impl reference)
# ---------------------------------------------------------------------------
def cpu_sample_rows(M, frac):
    n = max(1, int(M * frac))
    return np.linspace(0, M - 1, n).astype(np.int64)


def cpu_baseline(seconds):
    """Time the oracle on the host cores on a bounded sample of the decode
    workload (a row subset of each shape, N=1), in the same GB/s unit, plus a
    short timing of each other workload on a row sample."""
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
    other = {}
    # the other workloads on small row samples (rates per unit of work)
    for name, wt, M, K, N in (("q8_0_256x512_n1", synth.Q8_0, 256, 512, 1),
                              ("q4_k_prefill_4096x4096_n64", synth.Q4_K, 4096, 4096, 64),
                              ("q6_k_lmhead_n8", synth.Q6_K, 128256, 4096, 8)):
        rows = cpu_sample_rows(M, min(1.0, 128 / M))
        w = synth.gen_weights(wt, M, K, "cpu-sample") if M * K <= 4096 * 4096 else \
            synth.gen_weights(wt, 2048, K, "cpu-sample")
        Mw = M if M * K <= 4096 * 4096 else 2048
        rows = rows[rows < Mw]
        x = synth.gen_x(N, K, "cpu-sample")
        t0 = time.perf_counter()
        oracle.matmul(wt, w, Mw, K, x, rows=rows)
        dt = time.perf_counter() - t0
        other[name] = {"rows": int(rows.size), "s": round(dt, 4),
                       "GBps": round(rows.size * synth.row_bytes(wt, K) / dt / 1e9, 4),
                       "GFLOPs": round(2.0 * rows.size * K * N / dt / 1e9, 3)}
    return {"value": round(tot_bytes / tot_t / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{passes} pass(es) over {frac * 100:.2f}% of the rows of each Q4_0 decode shape, N=1; "
                      f"{tot_t:.1f} s of oracle time (C, f64, {cores} threads)",
            "other_workloads_on_row_samples": other}


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
    ap.add_argument("--copies", type=int, default=32, help="rotating weight copies (inputs > L2)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-sweep", action="store_true", help="skip the 32-layer decoder sweep")
    ap.add_argument("--sweep-layers", type=int, default=synth.DECODER_LAYERS)
    ap.add_argument("--no-check", action="store_true", help="skip the output check against the oracle")
    ap.add_argument("--no-static-weights", action="store_true",
                    help="launch every call only after the preceding kernel has finished")
    ap.add_argument("--only", default="",
                    help="comma list of ops to run (decode,lmhead,prefill,prefill_f32); default all")
    ap.add_argument("--scaling", choices=["weak", "strong"], default="weak",
                    help="multi-GPU: per-GPU rows fixed (weak) or global rows fixed (strong)")
    ap.add_argument("--allgather", action="store_true", help="multi-GPU: gather the decode outputs (NCCL)")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus != world:
        if world == 1 and args.gpus > 1 and "RANK" not in os.environ:
            # launched without torchrun: start one rank per GPU ourselves
            cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
                   "--master-addr", "127.0.0.1", "--master-port", os.environ.get("MASTER_PORT", "29517"),
                   os.path.abspath(__file__)] + sys.argv[1:]
            raise SystemExit(subprocess.call(cmd))
        raise SystemExit(f"--gpus {args.gpus} does not match WORLD_SIZE {world}")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
