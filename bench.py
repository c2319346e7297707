"""Benchmark of the sparse top-k MoE layer forward on GB300.

One step = one moe_layer_forward (router + top-k, permutation, grouped
SwiGLU GEMMs, combine) over one batch of seeded synthetic tokens of the
Mixtral-8x7B-shaped prefill layer (T=4096, d_model=4096, 8 experts, top-2,
d_ff=14336, bf16). Prints one JSON line; see ``--help``.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the plain fp64 definition) on the
host cores on a bounded sample of the same workload instead.
With N > 1 (torchrun) every rank runs an independent replica on its own
tokens (the layer is per-token; no collective on the data path); the
barrier and the max-over-ranks of the elapsed time use a gloo group.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s; grouped-GEMM % bf16 tensor peak; decode % HBM BW"
# fp32 FMA peak from unit counts and the maximum clock: 152 SMs x 128 lanes x 2 flop x 2.07 GHz
FP32_ALU_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
UNIT = "tokens/s"
AUX_ALPHA = 0.01  # the balance loss's weight alpha
L2_BYTES = 129 * 1024 * 1024  # GB300 L2
DECODE_MAX_T = 64  # batches up to this size stream the expert weights (decode)
# Nominal dense tensor rates relative to bf16 (2.25 PFLOP/s): fp8 4.5, fp4 13.5.
QUANT_PEAK_RATIO = {None: 1.0, "fp8": 4.5 / 2.25, "nvfp4": 13.5 / 2.25}
SPIN_CYCLES = 200_000  # ~0.1 ms at 2 GHz: covers the host's call latency of a decode step


# ----------------------------------------------------------------- helpers --
def world():
    """(rank, world_size, local_rank) from the torchrun environment."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def init_group(ws):
    if ws > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group("gloo")


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(v: float, ws: int) -> float:
    """Max of a host float over all ranks (gloo)."""
    if ws == 1:
        return float(v)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def kernel_source_key():
    """First 16 hex digits of the sha256 of the code lines of the grouped GEMM
    sources (csrc/grouped_sm103.cu then csrc/sm103_ptx.cuh; blank lines and
    lines that are only a // comment left out, so a comment edit keeps the
    key). None if the sources cannot be read."""
    import hashlib
    csrc = os.path.join(ROOT, "sparse_mixture_experts_router_gb300", "csrc")
    h = hashlib.sha256()
    try:
        for f in ("grouped_sm103.cu", "sm103_ptx.cuh"):
            for line in open(os.path.join(csrc, f), encoding="utf-8"):
                t = line.strip()
                if t and not t.startswith("//"):
                    h.update((t + "\n").encode())
    except OSError:
        return None
    return h.hexdigest()[:16]


# DRAM bytes per gate/up launch from ncu captures, keyed on the operand kind
# and workload (profiles/traffic.json; each entry names its summary file)
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def traffic_entries():
    """The recorded gate/up DRAM figures: {(quant, workload): entry}."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return {}
    return {(None if e["quant"] == "bf16" else e["quant"], e["workload"]): e
            for e in d.get("entries", []) if e.get("kernel") == "gate_up"}


def recorded_traffic(quant, workload):
    """DRAM bytes per gate/up launch recorded for this operand kind and
    workload, or None when there is none or the kernel code changed since
    that capture (kernel_source_key differs from the one recorded)."""
    e = traffic_entries().get((quant, workload))
    key = kernel_source_key()
    if e is None or key is None or e.get("kernel_source_sha256") != key:
        return None
    try:
        return float(e["dram_bytes_per_launch"])
    except (KeyError, TypeError, ValueError):
        return None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi clock / throttle samples every 50 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [s.strip() for s in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        # Samples while the GPU is loaded: the highest-power half of the run.
        pw = sorted((num(r[3]) or 0.0, i) for i, r in enumerate(rows))
        loaded = [rows[i] for _, i in pw[len(pw) // 2:]] or rows
        sm_loaded = [num(r[1]) for r in loaded if num(r[1]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in loaded:
            for name, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm_loaded) if sm_loaded else None,
                "sm_max_mhz": max(num(r[2]) or 0 for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(num(r[3]) or 0 for r in rows)}


# ---------------------------------------------------------- work accounting --
def capacity_of(w):
    if w.capacity_factor <= 0:
        return 0
    return max(1, math.ceil(w.capacity_factor * w.T * w.top_k / w.n_experts))


def gemm_flops(w, counts=None):
    """Algorithmic flops of the two grouped GEMMs: 4·d·d_ff and 2·d·d_ff per
    row that runs (routed pairs kept by the capacity, plus T shared rows per
    shared expert)."""
    routed = w.T * w.top_k
    cap = capacity_of(w)
    if cap and counts is not None:
        routed = sum(min(int(c), cap) for c in counts)
    rows = routed + w.n_shared * w.T
    return 4.0 * rows * w.d_model * w.d_ff, 2.0 * rows * w.d_ff * w.d_model


def expert_rows(moe, w, cfg, inp, counts, dev, stream):
    """Rows each routed expert ran in the last step, and a summary of the
    capacity reroute (None without one). Without a reroute these are the
    router's counts (gemm_flops and gemm_bytes apply the cut); with one, an
    untimed pass of the router (scores out) and moe_reroute on the same
    inputs gives the experts the pairs ran on."""
    import numpy as np
    import torch
    c = counts.cpu().tolist()
    if not (w.overflow and capacity_of(w)):
        return c, None
    T, N, k = w.T, w.n_experts, w.top_k
    logits = torch.empty(T, N, dtype=torch.float32, device=dev)
    idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    tw = torch.empty(T, k, dtype=torch.float32, device=dev)
    cnt = torch.empty(N, dtype=torch.int32, device=dev)
    ps = torch.empty(N, dtype=torch.float32, device=dev)
    rws = moe.workspace(cfg, "router", dev)
    moe.moe_router_topk(cfg, inp["x"], inp["w_router"], inp["logit_bias"], inp["sel_bias"], None,
                        logits, idx, tw, cnt, ps, rws, stream)
    assign = torch.empty(T, k, dtype=torch.int32, device=dev)
    rounds = torch.empty(1, dtype=torch.int32, device=dev)
    ws = moe.workspace(cfg, "reroute", dev)
    moe.moe_reroute(cfg, logits, inp["sel_bias"], idx, assign, rounds, ws, stream)
    if moe.moe_stream_status(ws, stream) != 0:
        raise RuntimeError(f"{w.name}: moe_reroute failed on the device")
    a, i0 = assign.cpu().numpy(), idx.cpu().numpy()
    loads = np.bincount(a[a >= 0], minlength=N).tolist()
    summary = {"capacity": capacity_of(w), "rounds": int(rounds.item()),
               "pairs_over_capacity": int(sum(max(0, v - capacity_of(w)) for v in c)),
               "pairs_rerouted": int(((a != i0) & (a >= 0)).sum()),
               "pairs_dropped": int((a < 0).sum())}
    return loads, summary


def gemm_bytes(w, counts, quant=None):
    """Algorithmic HBM bytes of the two grouped GEMMs: the weights (and
    scales) of every expert with a row, the A rows read once and the output
    rows written once. Operand bytes per element: bf16 2, E4M3 1 (+ an fp32
    row scale), NVFP4 1/2 (+ an E4M3 scale per 16 and an fp32 row scale); H
    is written in bf16 by gate/up in every case."""
    cap = capacity_of(w)
    routed = sum(min(int(c), cap) if cap else int(c) for c in counts)
    rows = routed + w.n_shared * w.T
    active = sum(1 for c in counts if c > 0) + w.n_shared
    d, f = w.d_model, w.d_ff

    def mat(r, cols):  # bytes of an r x cols operand in the GEMM's format
        if quant == "fp8":
            return r * cols + 4 * r
        if quant == "nvfp4":
            return r * cols // 2 + r * nvfp4_scale_stride(cols) + 4 * r
        return r * cols * eb
    eb = 4 if w.dtype == "f32" else 2  # activations and unquantized weights
    gu = active * 2 * mat(f, d) + mat(rows, d) + rows * f * eb
    dn = active * mat(d, f) + mat(rows, f) + rows * d * eb
    return gu, dn


def nvfp4_scale_stride(cols):
    """Bytes of one row of NVFP4 block scales (cols / 16 rounded up to 16)."""
    return (cols // 16 + 15) // 16 * 16


def touched_weight_bytes(w, counts, quant=None):
    """Expert weight bytes a forward must read: every expert with a row (E4M3:
    one byte a weight plus an fp32 scale per output channel; NVFP4: half a
    byte a weight, one E4M3 block scale per 16 weights and an fp32 scale per
    output channel)."""
    if quant == "fp8":
        per = 3 * w.d_model * w.d_ff + 4 * (2 * w.d_ff + w.d_model)
    elif quant == "nvfp4":
        per = (3 * w.d_model * w.d_ff // 2 + 2 * w.d_ff * nvfp4_scale_stride(w.d_model)
               + w.d_model * nvfp4_scale_stride(w.d_ff) + 4 * (2 * w.d_ff + w.d_model))
    else:
        per = 3 * w.d_model * w.d_ff * (2 if w.dtype == "bf16" else 4)
    active = sum(1 for c in counts if c > 0) + w.n_shared
    return active * per, active


class Forward:
    """One layer forward through the C ABI: moe_layer_forward, or with --fp8
    moe_layer_forward_fp8 on weights quantized once by moe_quantize_fp8, or
    with --nvfp4 moe_layer_forward_nvfp4 on weights quantized once by
    moe_quantize_nvfp4."""

    def __init__(self, moe, cfg, inp, quant, dev, q=None):
        import torch
        self.moe, self.cfg, self.inp, self.quant = moe, cfg, inp, quant
        self.ws = moe.workspace(cfg, {None: "layer", "fp8": "layer_fp8",
                                      "nvfp4": "layer_nvfp4"}[quant], dev)
        self.q = q if q is not None else []
        if quant and not self.q:
            for n in ("w_gate", "w_up", "w_down"):
                t = inp[n]
                rows, cols = t.shape[0] * t.shape[1], t.shape[2]
                sc = torch.empty(rows, dtype=torch.float32, device=dev)
                if quant == "fp8":
                    q = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
                    moe.moe_quantize_fp8(t.reshape(rows, cols), q, sc)
                    self.q.append((q, sc))
                else:
                    q = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
                    sf = torch.empty((rows, nvfp4_scale_stride(cols)), dtype=torch.uint8,
                                     device=dev)
                    moe.moe_quantize_nvfp4(t.reshape(rows, cols), q, sf, sc)
                    self.q.append((q, sf, sc))
            torch.cuda.synchronize(dev)

    def __call__(self, x, y, idx, tw, counts, ps, stream):
        i = self.inp
        if self.quant == "fp8":
            (gq, gs), (uq, us), (dq, ds) = self.q
            self.moe.moe_layer_forward_fp8(self.cfg, x, i["w_router"], i["logit_bias"],
                                           i["sel_bias"], gq, gs, uq, us, dq, ds, y, idx, tw,
                                           counts, ps, self.ws, stream)
        elif self.quant == "nvfp4":
            (gq, gf, gs), (uq, uf, us), (dq, df, ds) = self.q
            self.moe.moe_layer_forward_nvfp4(self.cfg, x, i["w_router"], i["logit_bias"],
                                             i["sel_bias"], gq, gf, gs, uq, uf, us, dq, df, ds,
                                             y, idx, tw, counts, ps, self.ws, stream)
        else:
            self.moe.moe_layer_forward(self.cfg, x, i["w_router"], i["logit_bias"], i["sel_bias"],
                                       i["w_gate"], i["w_up"], i["w_down"], y, idx, tw, counts,
                                       ps, self.ws, stream)


# ----------------------------------------------------------------- our arm --
def run_ours(args):
    import torch

    import sparse_mixture_experts_router_gb300 as moe
    from sparse_mixture_experts_router_gb300 import synth

    rank, ws, local = world()
    init_group(ws)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pk = peaks()
    w = shaped(WORKLOADS[args.workload](synth), args)
    if w.dtype == "f32" and args.quant:
        raise SystemExit("--fp8 / --nvfp4 take bf16 workloads")
    inp = synth.make_inputs(w, dev, seed=w.seed + 1000 * rank)
    eb = 4 if w.dtype == "f32" else 2
    cfg = moe.config(T=w.T, d_model=w.d_model, n_experts=w.n_experts, top_k=w.top_k, d_ff=w.d_ff,
                     n_shared=w.n_shared, dtype=moe.MOE_F32 if w.dtype == "f32" else moe.MOE_BF16,
                     gate_mode=w.gate_mode, capacity=capacity_of(w), tiles=args.tiles,
                     gather=args.gather, overflow=w.overflow)
    y = torch.empty(w.T, w.d_model, dtype=w.torch_dtype, device=dev)
    # Inputs that fit in L2 (the tiny fp32 layer) are timed step by step with
    # L2 flushed (a 256 MB write) before each step; larger ones stream their
    # weights from HBM every step anyway.
    in_bytes = sum(t.numel() * t.element_size() for t in inp.values() if t is not None)
    flush_l2 = in_bytes < 2 * L2_BYTES
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev) if flush_l2 else None
    idx = torch.empty(w.T, w.top_k, dtype=torch.int32, device=dev)
    tw = torch.empty(w.T, w.top_k, dtype=torch.float32, device=dev)
    counts = torch.empty(w.n_experts, dtype=torch.int32, device=dev)
    ps = torch.empty(w.n_experts, dtype=torch.float32, device=dev)
    fwd = Forward(moe, cfg, inp, args.quant, dev)
    wsp = fwd.ws
    stream = torch.cuda.current_stream(dev)

    def step(x):
        fwd(x, y, idx, tw, counts, ps, stream)

    default = args.workload == DEFAULT_WORKLOAD and not reshaped(args)
    # The decode sweep runs before the prefill timing and the end-to-end
    # loop: measured after them, in the same process, the single-token step
    # took ~14 us more (0.160 against 0.146 ms, its one kernel unchanged at
    # 143 us); run first it matches a process that runs it alone.
    decode = run_decode(moe, synth, dev, stream, pk, args) if default and not args.no_decode else None
    for _ in range(args.warmup):
        step(inp["x"])
    torch.cuda.synchronize(dev)
    st = moe.moe_stream_status(wsp, stream)
    if st != 0:
        raise RuntimeError(f"warm-up step failed on the device: {moe.status_string(st)}")

    # ---- device-timed region: inputs resident in HBM -------------------------
    clocks = ClockSampler(local)
    clocks.start()
    # Events only around the dominant kernel: an event between two launches
    # costs the programmatic-dependent-launch overlap at that boundary.
    moe.profile_enable(True, kernels=["gate_up", "decode_fused"])
    moe.profile_collect()  # drop anything recorded before
    launches0 = moe.launch_count()
    barrier(ws)
    torch.cuda.synchronize(dev)
    clocks.mark("t0")
    if flush_l2:
        ms_local = 0.0
        for _ in range(args.steps):
            flush.fill_(1)
            torch.cuda._sleep(SPIN_CYCLES)  # the host's call latency stays outside the events
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step(inp["x"])
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ms_local += e0.elapsed_time(e1)
    else:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step(inp["x"])
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms_local = e0.elapsed_time(e1)
    clocks.mark("t1")
    barrier(ws)
    launches = moe.launch_count() - launches0
    kern_timed = moe.profile_collect()
    moe.profile_enable(False)
    clk = clocks.stop()
    ms_total = reduce_max(ms_local, ws)
    ms_step = ms_total / args.steps
    value = ws * w.T * args.steps / (ms_total / 1e3)

    # ---- end to end through the C ABI with host buffers ----------------------
    # Every step copies its tokens from pinned host memory to the device, runs
    # moe_layer_forward and copies y back to pinned host memory. The copies of
    # step i+1 / i-1 overlap the forward of step i (separate copy streams,
    # two device buffers each, ordered with events), as a serving loop does.
    x_host = inp["x"].cpu().pin_memory()
    y_host = [torch.empty(w.T, w.d_model, dtype=w.torch_dtype).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(inp["x"]) for _ in range(2)]
    y_dev = [torch.empty_like(y) for _ in range(2)]
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    x_ready, x_free = [ev(), ev()], [ev(), ev()]
    y_ready, y_free = [ev(), ev()], [ev(), ev()]
    for e_ in x_free + y_free:
        e_.record(stream)

    def e2e_step(i):
        b = i % 2
        h2d.wait_event(x_free[b])
        with torch.cuda.stream(h2d):
            x_dev[b].copy_(x_host, non_blocking=True)
        x_ready[b].record(h2d)
        stream.wait_event(x_ready[b])
        stream.wait_event(y_free[b])
        fwd(x_dev[b], y_dev[b], idx, tw, counts, ps, stream)
        x_free[b].record(stream)
        y_ready[b].record(stream)
        d2h.wait_event(y_ready[b])
        with torch.cuda.stream(d2h):
            y_host[b].copy_(y_dev[b], non_blocking=True)
        y_free[b].record(d2h)

    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier(ws)
    t0 = time.perf_counter()
    for i in range(args.steps):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e2e_s = time.perf_counter() - t0
    barrier(ws)
    e2e_ms = reduce_max(e2e_s * 1e3, ws)
    e2e_value = ws * w.T * args.steps / (e2e_ms / 1e3)
    bytes_io = w.T * w.d_model * eb

    # ---- every kernel bracketed by events, in a separate pass ------------------
    # (shares and per-kernel rates; the step time above is taken without them)
    moe.profile_enable(True)
    step(inp["x"])         # the first step waits on the host; leave it out
    moe.profile_collect()
    for _ in range(min(args.steps, 5)):
        step(inp["x"])
    kern = moe.profile_collect()
    moe.profile_enable(False)

    # ---- roofline of the dominant kernel ---------------------------------------
    # rows each expert ran: the router's counts, cut by the capacity, or
    # after the capacity reroute
    loads, rerouted = expert_rows(moe, w, cfg, inp, counts, dev, stream)
    f_gu, f_dn = gemm_flops(w, loads)
    per_kernel = {}
    for name, (ms, n) in kern.items():
        per_kernel[name] = {"ms_per_launch": ms / n, "launches": n,
                            "share": ms / sum(v[0] for v in kern.values())}
    # the dominant kernel's duration comes from the timed region itself
    # E4M3 / NVFP4: the measured bf16 peaks times the nominal dense ratio of
    # the operand type to bf16 (4.5 / 2.25 for fp8, 13.5 / 2.25 for fp4)
    ratio = QUANT_PEAK_RATIO[args.quant]
    tpk = pk["bf16"] * ratio
    tpk_s = pk["bf16_sustained"] * ratio
    if "gate_up" not in kern_timed:  # a single token: the whole layer is one kernel
        fused_ms = kern_timed["decode_fused"][0] / kern_timed["decode_fused"][1]
        per_kernel["decode_fused"]["ms_per_launch"] = fused_ms
        wbytes, _ = touched_weight_bytes(w, loads, args.quant)
        total = wbytes + w.n_experts * w.d_model * 2 + 2 * w.T * w.d_model * 2
        gbs = total / (fused_ms / 1e3) / 1e9
        per_kernel["decode_fused"]["gbs"] = round(gbs, 1)
        gemm_tflops = (f_gu + f_dn) / (fused_ms / 1e3) / 1e12
        roofline = {"bound": "hbm", "kernel": "decode_fused (routing, both projections and the "
                                              "gated sum in one kernel)",
                    "achieved": round(gbs, 1), "peak": round(pk["hbm"], 1), "unit": "GB/s",
                    "frac": round(gbs / pk["hbm"], 4), "traffic": None,
                    "peak_source": f"{pk['source']} HBM copy",
                    "algorithmic_bytes_per_launch": total}
    else:
        per_kernel["gate_up"]["ms_per_launch"] = kern_timed["gate_up"][0] / kern_timed["gate_up"][1]
    gu_ms = per_kernel["gate_up"]["ms_per_launch"] if "gate_up" in kern_timed else None
    if gu_ms is not None:
        dn_ms = per_kernel["down"]["ms_per_launch"]
        per_kernel["gate_up"]["tflops"] = f_gu / (gu_ms / 1e3) / 1e12
        per_kernel["down"]["tflops"] = f_dn / (dn_ms / 1e3) / 1e12
        # the same launches against HBM: algorithmic bytes / time
        b_gu, b_dn = gemm_bytes(w, loads, args.quant)
        for name, b, ms in (("gate_up", b_gu, gu_ms), ("down", b_dn, dn_ms)):
            per_kernel[name]["algorithmic_bytes"] = b
            per_kernel[name]["gbs"] = round(b / (ms / 1e3) / 1e9, 1)
            per_kernel[name]["hbm_frac"] = round(b / (ms / 1e3) / 1e9 / pk["hbm"], 4)
        gemm_tflops = (f_gu + f_dn) / ((gu_ms + dn_ms) / 1e3) / 1e12
        ach = per_kernel["gate_up"]["tflops"]
    if gu_ms is not None and w.dtype == "f32":
        # fp32 layers run their expert products on the CUDA cores (tcgen05 has
        # no fp32-operand kind): the peak is the fp32 FMA rate
        roofline = {"bound": "alu", "kernel": "gate_up (fp32 CUDA-core expert GEMM, stage 1)",
                    "achieved": round(ach, 3), "peak": round(FP32_ALU_PEAK_TFLOPS, 1),
                    "unit": "TFLOP/s", "frac": round(ach / FP32_ALU_PEAK_TFLOPS, 5),
                    "traffic": None,
                    "peak_source": "152 SMs x 128 fp32 lanes x 2 flop x 2.07 GHz",
                    "algorithmic_flops_per_launch": f_gu,
                    "note": "a few thousand tokens' worth of work: bound by launch and "
                            "memory latency, reported for its latency"}
    elif gu_ms is not None and w.T <= DECODE_MAX_T:
        # decode-sized batches stream the weights: the bound is HBM
        gbs_gu = per_kernel["gate_up"]["gbs"]
        roofline = {"bound": "hbm", "kernel": "gate_up (grouped SwiGLU gate+up GEMM, decode tiles)",
                    "achieved": gbs_gu, "peak": round(pk["hbm"], 1), "unit": "GB/s",
                    "frac": round(gbs_gu / pk["hbm"], 4),
                    "traffic": (args.traffic if args.traffic is not None
                                else recorded_traffic(args.quant, w.name)),
                    "peak_source": f"{pk['source']} HBM copy",
                    "algorithmic_bytes_per_launch": per_kernel["gate_up"]["algorithmic_bytes"],
                    "tflops": round(ach, 1)}
    elif gu_ms is not None:
        roofline = {"bound": "tensor", "kernel": "gate_up (grouped SwiGLU gate+up GEMM)",
                    "achieved": round(ach, 1), "peak": round(tpk, 1), "unit": "TFLOP/s",
                    "frac": round(ach / tpk, 4),
                    "traffic": (args.traffic if args.traffic is not None
                                else recorded_traffic(args.quant, w.name)),
                    "peak_source": (f"{pk['source']} bf16 burst x {ratio:g} (nominal "
                                    f"{args.quant}/bf16 dense ratio)"
                                    if args.quant else f"{pk['source']} bf16 burst"),
                    "frac_of_sustained": round(ach / tpk_s, 4),
                    "algorithmic_flops_per_launch": f_gu,
                    "grouped_gemm_both_kernels_tflops": round(gemm_tflops, 1),
                    "grouped_gemm_both_kernels_frac": round(gemm_tflops / tpk, 4)}
    # HBM-bound kernels of the step against the copy bandwidth
    P = w.T * w.top_k
    # permute_gather: each token row is read from HBM once (a token's second
    # and later copies hit L2), every routed row written once, plus the row
    # indices: the unique bytes, not 2 P d
    hb = {"router_topk": w.T * w.d_model * eb + w.n_experts * w.d_model * eb + P * 8,
          "permute_gather": (w.T + P) * w.d_model * eb + P * 4,
          "combine": (P + w.n_shared * w.T) * w.d_model * eb + w.T * w.d_model * eb + P * 4}
    if "router_topk" in per_kernel:  # the router's score contraction
        fl = 2.0 * w.T * w.n_experts * w.d_model
        tf = fl / (per_kernel["router_topk"]["ms_per_launch"] / 1e3) / 1e12
        if w.dtype == "bf16":  # tensor cores (tcgen05 for N > 32, mma.sync up to 32)
            per_kernel["router_topk"]["tensor_tflops"] = round(tf, 2)
            per_kernel["router_topk"]["tensor_frac"] = round(tf / pk["bf16"], 4)
        else:  # CUDA-core FMA router kernels
            per_kernel["router_topk"]["fp32_tflops"] = round(tf, 2)
            per_kernel["router_topk"]["fp32_alu_frac"] = round(tf / FP32_ALU_PEAK_TFLOPS, 4)
    for name, b in hb.items():
        if name in per_kernel:
            gbs = b / (per_kernel[name]["ms_per_launch"] / 1e3) / 1e9
            per_kernel[name]["gbs"] = round(gbs, 1)
            per_kernel[name]["hbm_frac"] = round(gbs / pk["hbm"], 4)

    # the other layer shapes and operand types, measured in the same run
    others = {}
    if default and not args.quant and not args.no_others:
        for key, ow, q in (("deepseek_v3_moe", synth.DEEPSEEK_V3, None),
                           ("zipf_imbalanced", synth.ZIPF, None),
                           ("zipf_imbalanced_capacity_reroute", synth.ZIPF_REROUTE, None),
                           ("mixtral_8x7b_prefill_fp8", synth.MIXTRAL_PREFILL, "fp8"),
                           ("mixtral_8x7b_prefill_nvfp4", synth.MIXTRAL_PREFILL, "nvfp4")):
            others[key] = run_layer_summary(moe, synth, dev, stream, pk, ow, q, args)
    backward = (run_backward(moe, dev, stream, pk, w, inp, cfg, args)
                if default and not args.quant and not args.no_backward else None)
    E = w.n_experts + w.n_shared
    wb = touched_weight_bytes(w, [1] * w.n_experts, args.quant)[0]
    # balance statistics of the last step's routing, by the library's own kernel:
    # f_i = counts_i / (T*k), P_i = prob_sum_i / T, aux = alpha * N * sum_i f_i P_i
    bf = torch.empty(w.n_experts, dtype=torch.float32, device=dev)
    bP = torch.empty(w.n_experts, dtype=torch.float32, device=dev)
    baux = torch.empty(1, dtype=torch.float32, device=dev)
    moe.moe_balance_stats(w.n_experts, w.T, w.top_k, counts, ps, AUX_ALPHA, bf, bP, baux, stream)
    torch.cuda.synchronize(dev)
    routing = {"max_over_mean_expert_load": round(float(counts.max()) / max(1e-9, float(counts.float().mean())), 3),
               "experts_with_tokens": int((counts > 0).sum()),
               "aux_loss": {"alpha": AUX_ALPHA, "value": round(float(baux.item()), 6),
                            "balanced_value": AUX_ALPHA,
                            "f": [round(v, 5) for v in bf.cpu().tolist()],
                            "P": [round(v, 5) for v in bP.cpu().tolist()]}}
    if rerouted is not None:
        routing["capacity_reroute"] = rerouted
    elif capacity_of(w):
        routing["pairs_dropped_by_capacity"] = int(sum(max(0, int(c) - capacity_of(w))
                                                       for c in counts.cpu().tolist()))

    if rank == 0:
        cpu = None if (args.no_cpu_baseline or not default) else cpu_baseline(inp, w, args)
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("f32" if w.dtype == "f32" else
                      {None: "bf16", "fp8": "e4m3 experts (row scales), bf16 tokens and router",
                       "nvfp4": "nvfp4 experts (e2m1, e4m3 scales of 16-element blocks, row "
                                "scales), bf16 tokens and router"}[args.quant]),
            "data": "synthetic (seeded N(0,1) tokens, N(0,0.02^2) random-init weights)",
            "config": {"workload": w.name, "T": w.T, "d_model": w.d_model,
                       "n_experts": w.n_experts, "top_k": w.top_k, "d_ff": w.d_ff,
                       "n_shared": w.n_shared,
                       "gate": ["softmax over the kept top-k scores",
                                "softmax over all scores, kept ones renormalised"][w.gate_mode],
                       "selection_bias": w.sel_bias, "zipf_offset_s": w.zipf_s or None,
                       "capacity": capacity_of(w) or None,
                       "overflow": (("rerouted" if w.overflow else "dropped")
                                    if capacity_of(w) else None),
                       "tiles": {0: "library's choice", 1: "1-CTA", 2: "256-row CTA pairs",
                                 3: "weight-stationary CTA pairs"}[args.tiles],
                       "gather": {0: "library's choice", 1: "a kernel of its own",
                                  2: "fused into the gate/up GEMM"}[args.gather],
                       "parallelism": f"replicas x{ws} (per-token layer, no collective)",
                       "l2": (f"inputs ({in_bytes / 1e6:.2f} MB) fit in L2: L2 flushed (256 MB "
                              "write) before every timed step, each step timed on its own"
                              if flush_l2 else
                              f"inputs larger than L2: {wb / 1e9:.2f} GB of expert weights read "
                              "every step")},
            "routing": routing,
            "tflops_grouped_gemm": round(gemm_tflops, 1),
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": bytes_io,
                    "d2h_bytes_per_step": bytes_io,
                    "path": "per step: pinned host x -> H2D (copy stream) -> moe_layer_forward"
                            + {None: " ", "fp8": "_fp8 ", "nvfp4": "_nvfp4 "}[args.quant] +
                            "(C ABI, compute stream) -> D2H y (copy stream) -> pinned host; "
                            "copies overlap neighbouring steps' forwards; host wall clock"},
            "gpu_launches": int(launches),
            "clocks": clk,
            "kernels": per_kernel,
            "decode": decode,
            "backward": backward,
        }
        line.update(others)
        print(json.dumps(line))


def run_layer_summary(moe, synth, dev, stream, pk, w, quant, args):
    """A compact measurement of one more workload for the default run: the
    layer step (device time, CUDA events, inputs resident in HBM; the expert
    weights exceed L2), tokens/s, and both grouped GEMMs against their
    rooflines (algorithmic flops against the bf16 burst peak times the
    operand type's nominal ratio, algorithmic bytes against the measured HBM
    copy bandwidth), from a second, profiled pass. The tiling is the
    library's choice."""
    import torch
    inp = synth.make_inputs(w, dev)
    cfg = moe.config(T=w.T, d_model=w.d_model, n_experts=w.n_experts, top_k=w.top_k, d_ff=w.d_ff,
                     n_shared=w.n_shared, dtype=moe.MOE_BF16, gate_mode=w.gate_mode,
                     capacity=capacity_of(w), overflow=w.overflow)
    y = torch.empty(w.T, w.d_model, dtype=torch.bfloat16, device=dev)
    idx = torch.empty(w.T, w.top_k, dtype=torch.int32, device=dev)
    tw = torch.empty(w.T, w.top_k, dtype=torch.float32, device=dev)
    counts = torch.empty(w.n_experts, dtype=torch.int32, device=dev)
    ps = torch.empty(w.n_experts, dtype=torch.float32, device=dev)
    fwd = Forward(moe, cfg, inp, quant, dev)

    def step():
        fwd(inp["x"], y, idx, tw, counts, ps, stream)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if moe.moe_stream_status(fwd.ws, stream) != 0:
        raise RuntimeError(f"{w.name}: warm-up step failed on the device")
    reps = max(5, min(args.steps, 20))
    # the dominant kernel's duration inside the timed region, as in the headline
    moe.profile_enable(True, kernels=["gate_up"])
    moe.profile_collect()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / reps
    gu_timed = moe.profile_collect()
    moe.profile_enable(True)
    moe.profile_collect()
    for _ in range(3):
        step()
    kern = moe.profile_collect()
    moe.profile_enable(False)
    c, rerouted = expert_rows(moe, w, cfg, inp, counts, dev, stream)
    f_gu, f_dn = gemm_flops(w, c)
    b_gu, b_dn = gemm_bytes(w, c, quant)
    ratio = QUANT_PEAK_RATIO[quant]
    tpk = pk["bf16"] * ratio
    gu_ms = gu_timed["gate_up"][0] / gu_timed["gate_up"][1]
    dn_ms = kern["down"][0] / kern["down"][1]
    out = {"workload": w.name, "T": w.T, "d_model": w.d_model, "n_experts": w.n_experts,
           "n_shared": w.n_shared, "top_k": w.top_k, "d_ff": w.d_ff,
           "operands": {None: "bf16", "fp8": "e4m3 experts (row scales)",
                        "nvfp4": "nvfp4 experts (e2m1, e4m3 16-element block scales, row scales)"}[quant],
           "ms_per_step": round(ms, 4), "steps": reps,
           "tokens_per_s": round(w.T / (ms / 1e3), 1),
           "peak_tflops": round(tpk, 1),
           "peak_source": (f"{pk['source']} bf16 burst x {ratio:g}" if quant
                           else f"{pk['source']} bf16 burst")}
    for name, f, by, t in (("gate_up", f_gu, b_gu, gu_ms), ("down", f_dn, b_dn, dn_ms)):
        tf = f / (t / 1e3) / 1e12
        gbs = by / (t / 1e3) / 1e9
        out[name] = {"ms": round(t, 4), "tflops": round(tf, 1), "tensor_frac": round(tf / tpk, 4),
                     "algorithmic_bytes": by, "gbs": round(gbs, 1),
                     "hbm_frac": round(gbs / pk["hbm"], 4),
                     # the floor is whichever of the tensor and HBM times is larger
                     "roofline_ms": round(max(f / (tpk * 1e12), by / (pk["hbm"] * 1e9)) * 1e3, 4)}
    out["kernel_ms"] = {k: round(v[0] / v[1], 4) for k, v in kern.items()}
    if rerouted is not None:
        out["capacity_reroute"] = rerouted
    out["experts_with_tokens"] = int(sum(1 for v in c if v > 0))
    out["max_over_mean_expert_load"] = round(max(c) / max(1e-9, sum(c) / len(c)), 3)
    if w.zipf_s:
        bf = torch.empty(w.n_experts, dtype=torch.float32, device=dev)
        bP = torch.empty(w.n_experts, dtype=torch.float32, device=dev)
        baux = torch.empty(1, dtype=torch.float32, device=dev)
        moe.moe_balance_stats(w.n_experts, w.T, w.top_k, counts, ps, AUX_ALPHA, bf, bP, baux,
                              stream)
        torch.cuda.synchronize(dev)
        out["aux_loss"] = {"alpha": AUX_ALPHA, "value": round(float(baux.item()), 6),
                           "balanced_value": AUX_ALPHA}
    del inp, fwd
    torch.cuda.empty_cache()
    return out


def reshaped(args):
    return any(v is not None for v in (args.tokens, args.experts, args.d_ff))


def shaped(w, args):
    """The workload with --tokens / --experts / --d-ff applied (a smaller case
    of the same layer shape, for profiling); its name says so."""
    if not reshaped(args):
        return w
    n = args.experts or w.n_experts
    w2 = w.replace(T=args.tokens or w.T, n_experts=n, top_k=min(w.top_k, n),
                   d_ff=args.d_ff or w.d_ff)
    return w2.replace(name=f"{w.name} (T={w2.T}, {w2.n_experts} experts, d_ff={w2.d_ff})")


def run_backward_only(args):
    """The backward alone, on the workload or a smaller case of the same shape
    (--tokens, --experts): one JSON line with the backward object."""
    import torch

    import sparse_mixture_experts_router_gb300 as moe
    from sparse_mixture_experts_router_gb300 import synth
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.workload](synth)
    w = w.replace(T=args.tokens or w.T, n_experts=args.experts or w.n_experts,
                  top_k=min(w.top_k, args.experts or w.n_experts))
    inp = synth.make_inputs(w, dev)
    cfg = moe.config(T=w.T, d_model=w.d_model, n_experts=w.n_experts, top_k=w.top_k, d_ff=w.d_ff,
                     n_shared=w.n_shared, dtype=moe.MOE_BF16, gate_mode=w.gate_mode,
                     capacity=capacity_of(w))
    out = run_backward(moe, dev, torch.cuda.current_stream(dev), peaks(), w, inp, cfg, args)
    print(json.dumps({"workload": w.name, "T": w.T, "n_experts": w.n_experts, "top_k": w.top_k,
                      "d_model": w.d_model, "d_ff": w.d_ff, "backward": out}))


def run_backward(moe, dev, stream, pk, w, inp, cfg, args):
    """The layer's backward (moe_layer_backward: forward recomputed, then the
    activation and weight gradients) on the same workload, dL/dy ~ N(0, 1):
    device time per step with CUDA events (operands and gradients far larger
    than L2), a per-kernel breakdown from a separate profiled step, and the
    tensor-core work against the bf16 peak. Algorithmic work: the forward's
    two projections again (6 d d_ff flop per row), the activation gradients
    dH and dA (6 d d_ff), the weight gradients (6 d d_ff); the router's
    products (2 x 2 T N d) are counted too."""
    import torch
    from sparse_mixture_experts_router_gb300 import synth
    E = w.n_experts + w.n_shared
    dy = synth.make_grad_output(w, dev)
    dx = torch.empty(w.T, w.d_model, device=dev)
    dwr = torch.empty(w.n_experts, w.d_model, device=dev)
    dwg = torch.empty(E, w.d_ff, w.d_model, device=dev)
    dwu = torch.empty_like(dwg)
    dwd = torch.empty(E, w.d_model, w.d_ff, device=dev)
    ws = moe.workspace(cfg, "backward", dev)

    def step():
        moe.moe_layer_backward(cfg, inp["x"], inp["w_router"], inp["logit_bias"], inp["sel_bias"],
                               inp["w_gate"], inp["w_up"], inp["w_down"], dy, 0.01, 1.0, dx, dwr,
                               dwg, dwu, dwd, ws, stream)
    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    if moe.moe_stream_status(ws, stream) != 0:
        raise RuntimeError("backward warm-up failed on the device")
    reps = max(3, min(args.steps, 20))
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / reps
    moe.profile_enable(True)
    moe.profile_collect()
    step()
    kern = moe.profile_collect()
    moe.profile_enable(False)
    R = w.T * (w.top_k + w.n_shared)
    flops = 18.0 * w.d_model * w.d_ff * R + 4.0 * w.T * w.n_experts * w.d_model
    tf = flops / (ms / 1e3) / 1e12
    out = {"ms_per_step": round(ms, 4), "steps": reps,
           "tokens_per_s": round(w.T / (ms / 1e3), 1),
           "algorithmic_tflop": round(flops / 1e12, 3), "tflops": round(tf, 1),
           "frac_of_bf16_sustained": round(tf / pk["bf16_sustained"], 4),
           "kernels": {k: {"ms": round(v[0], 4), "launches": v[1],
                           "share": round(v[0] / sum(x[0] for x in kern.values()), 4)}
                       for k, v in kern.items()},
           "outputs": "fp32 dx, dW_r, dW_g, dW_u, dW_d; dy bf16; alpha 0.01, aux_grad 1"}
    if "bwd_wgrad" in kern:  # the three expert weight-gradient launches
        wms = kern["bwd_wgrad"][0] / kern["bwd_wgrad"][1]
        wfl = 2.0 * w.d_model * w.d_ff * R
        out["wgrad_tflops"] = round(wfl / (wms / 1e3) / 1e12, 1)
        out["wgrad_gbs_written"] = round(E * w.d_model * w.d_ff * 4 / (wms / 1e3) / 1e9, 1)
    return out


def run_decode(moe, synth, dev, stream, pk, args):
    """Decode steps (T = 1, 8, 32, 64) of the same layer: weight streaming,
    reported as algorithmic bytes / time against the HBM copy bandwidth, for
    plain launches and for the same call replayed from a CUDA graph. L2 is
    flushed (a 256 MB write) before every timed step."""
    import torch
    out = {}
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    base = synth.make_inputs(synth.MIXTRAL_DECODE[-1], dev)
    qcache = None
    for w in synth.MIXTRAL_DECODE:
        x = base["x"][: w.T].contiguous()
        cfg = moe.config(T=w.T, d_model=w.d_model, n_experts=w.n_experts, top_k=w.top_k,
                         d_ff=w.d_ff, dtype=moe.MOE_BF16)
        y = torch.empty(w.T, w.d_model, dtype=torch.bfloat16, device=dev)
        counts = torch.empty(w.n_experts, dtype=torch.int32, device=dev)
        fwd = Forward(moe, cfg, base, args.quant, dev, qcache)
        qcache = fwd.q  # the expert weights are quantized once for all batch sizes

        def step(st=None):
            fwd(x, y, None, None, counts, None,
                st if st is not None else torch.cuda.current_stream(dev))
        for _ in range(3):
            step()
        torch.cuda.synchronize(dev)
        reps = max(5, min(args.steps, 50))

        def timed(fn):
            # A ~0.1 ms spin kernel after the L2 flush keeps the GPU busy while
            # the host makes the call (Python marshalling of the step's
            # arguments takes tens of microseconds, longer than a T = 1 step's
            # first kernel); the events then bracket the step's own GPU time
            # and not the host's call latency.
            out = []
            for _ in range(reps):
                flush.fill_(1)
                torch.cuda._sleep(SPIN_CYCLES)
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record()
                fn()
                b.record()
                torch.cuda.synchronize(dev)
                out.append(a.elapsed_time(b))
            return statistics.median(out)

        ms = timed(step)
        # The same forward captured once in a CUDA graph and replayed (what a
        # serving loop does for decode-sized steps): no launch gaps.
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(cap):
            step(cap)  # warm the capture stream
        torch.cuda.current_stream(dev).wait_stream(cap)
        torch.cuda.synchronize(dev)
        with torch.cuda.graph(graph, stream=cap):
            step(cap)
        graph.replay()
        torch.cuda.synchronize(dev)
        ms_graph = timed(graph.replay)
        # per-kernel breakdown in separate steps (the events add a little time)
        moe.profile_enable(True)
        moe.profile_collect()
        for _ in range(5):
            flush.fill_(1)
            step()
        kern = moe.profile_collect()
        moe.profile_enable(False)
        wbytes, active = touched_weight_bytes(w, counts.cpu().tolist(), args.quant)
        total = wbytes + w.n_experts * w.d_model * 2 + 2 * w.T * w.d_model * 2
        gbs = total / (ms / 1e3) / 1e9
        gbs_g = total / (ms_graph / 1e3) / 1e9
        out[f"T{w.T}"] = {"ms": round(ms, 4), "experts_touched": active,
                          "algorithmic_bytes": total, "gbs": round(gbs, 1),
                          "hbm_frac": round(gbs / pk["hbm"], 4),
                          "tokens_per_s": round(w.T / (ms / 1e3), 1),
                          "graph_ms": round(ms_graph, 4), "graph_gbs": round(gbs_g, 1),
                          "graph_hbm_frac": round(gbs_g / pk["hbm"], 4),
                          "kernel_us": {k: round(1e3 * v[0] / v[1], 1) for k, v in kern.items()}}
    return out


# ------------------------------------------------------------- CPU oracle ----
def _oracle_sample(o, inp_host, w, rows):
    """Oracle forward: routing of every token, layer output of `rows`."""
    x, Wr, wg, wu, wd = inp_host
    _, r32 = o.router_logits(x, Wr, None)
    idx, tw, _, _ = o.route(r32, w.top_k, w.gate_mode, None)
    need = sorted(set(idx[rows].ravel().tolist()))
    experts = {e: (wg[e], wu[e], wd[e]) for e in need}
    return o.layer_rows(x, experts, idx, tw, rows, w.n_experts, w.n_shared)


def _host_inputs(inp):
    from sparse_mixture_experts_router_gb300 import synth
    return tuple(synth.bf16_bits(inp[k]) for k in ("x", "w_router", "w_gate", "w_up", "w_down"))


def cpu_baseline(inp, w, args):
    """The oracle as it stands, on this host's cores, on a bounded sample:
    routing of all T tokens plus the layer output of n sampled tokens, timed
    and scaled to tokens/s (tokens are independent, so per-token time
    extrapolates)."""
    import oracle
    o = oracle.Oracle()
    host = _host_inputs(inp)
    n = args.cpu_tokens
    rows = list(range(0, w.T, max(1, w.T // n)))[:n]
    t0 = time.perf_counter()
    _oracle_sample(o, host, w, rows)
    dt = time.perf_counter() - t0
    return {"value": round(len(rows) / dt, 3), "unit": UNIT, "cores": o.num_threads(),
            "kind": "oracle",
            "sample": f"routing of all {w.T} tokens + layer output of {len(rows)} of {w.T} tokens "
                      f"(fp64 C oracle, OpenMP), {dt:.1f} s; tokens/s = {len(rows)} / time"}


def run_reference(args):
    """The CPU oracle timed on the host cores (rank 0 only)."""
    rank, ws, local = world()
    if rank != 0:
        return
    import torch

    import oracle
    from sparse_mixture_experts_router_gb300 import synth
    w = synth.MIXTRAL_PREFILL
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    inp = synth.make_inputs(w, dev)
    host = _host_inputs(inp)
    del inp
    o = oracle.Oracle()
    n = args.ref_tokens
    times = []
    for i in range(args.warmup + args.steps):
        rows = [((i * 997) + j * (w.T // n)) % w.T for j in range(n)]
        t0 = time.perf_counter()
        _oracle_sample(o, host, w, rows)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = n * len(times) / total
    sample = (f"per step: routing of all {w.T} tokens + layer output of {n} of {w.T} tokens "
              f"(fp64 C oracle, OpenMP); tokens/s = sampled tokens / time")
    line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * total / len(times), 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "T": w.T, "d_model": w.d_model, "n_experts": w.n_experts,
                       "top_k": w.top_k, "d_ff": w.d_ff},
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "kind": "oracle",
                             "cores": o.num_threads(), "sample": sample},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


DEFAULT_WORKLOAD = "mixtral_8x7b_prefill"
WORKLOADS = {
    "tiny_fp32": lambda synth: synth.TINY,
    "mixtral_8x7b_prefill": lambda synth: synth.MIXTRAL_PREFILL,
    "deepseek_v3_moe": lambda synth: synth.DEEPSEEK_V3,
    "zipf_imbalanced": lambda synth: synth.ZIPF,
    "zipf_imbalanced_capacity": lambda synth: synth.ZIPF_CAPACITY,
    "zipf_imbalanced_capacity_reroute": lambda synth: synth.ZIPF_REROUTE,
    **{f"mixtral_8x7b_decode_T{t}": (lambda t_: lambda synth: [w for w in synth.MIXTRAL_DECODE if w.T == t_][0])(t)
       for t in (1, 8, 32, 64)},
}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD,
                    help="layer shape to time (the default is the one the metric is quoted on)")
    ap.add_argument("--cpu-tokens", type=int, default=48,
                    help="sampled tokens of the CPU-oracle baseline")
    ap.add_argument("--ref-tokens", type=int, default=4,
                    help="sampled tokens per step of --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--no-others", action="store_true",
                    help="skip the DeepSeek-V3, Zipf, FP8 and NVFP4 objects of the default run")
    ap.add_argument("--backward-only", action="store_true",
                    help="time only the layer's backward and print its object (for profiling)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="tokens T instead of the workload's (a smaller case, for profiling)")
    ap.add_argument("--experts", type=int, default=None,
                    help="routed experts N instead of the workload's (for profiling)")
    ap.add_argument("--d-ff", type=int, default=None,
                    help="expert width d_ff instead of the workload's (for profiling)")
    ap.add_argument("--fp8", action="store_true",
                    help="E4M3 expert weights (moe_layer_forward_fp8); not the headline, which is bf16")
    ap.add_argument("--nvfp4", action="store_true",
                    help="NVFP4 expert weights (moe_layer_forward_nvfp4); not the headline, which "
                         "is bf16")
    ap.add_argument("--tiles", type=int, choices=[0, 1, 2, 3], default=0,
                    help="grouped-GEMM tiling (moe_config.tiles): 0 the library's choice, 1 1-CTA, "
                         "2 256-row CTA pairs, 3 weight-stationary CTA pairs")
    ap.add_argument("--gather", type=int, choices=[0, 1, 2], default=0,
                    help="row gather (moe_config.gather): 0 the library's choice, 1 a kernel of its "
                         "own, 2 fused into the gate/up GEMM")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per gate_up launch from an ncu capture of this build")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.fp8 and args.nvfp4:
        ap.error("--fp8 and --nvfp4 exclude each other")
    args.quant = "fp8" if args.fp8 else "nvfp4" if args.nvfp4 else None
    if args.impl == "reference":
        run_reference(args)
    elif args.backward_only:
        run_backward_only(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
