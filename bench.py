#!/usr/bin/env python3
"""Benchmark of the SiTU routed-MoE expert layer on GB300.

The headline line is the Kimi-K3 TP8 decode layer, w4a16 (T=64 tokens,
hidden 3584, intermediate 384, 896 local experts, top-16 uniform routing,
bf16 activations, MXFP4 weights); the same JSON line carries a second
record, ``prefill_w4a8_8192``, for the Kimi-K3 TP8 prefill layer, w4a8
(T=8192, top-16 Zipf(1.0), MXFP8 activations quantised from bf16 inside the
step).  One step = one pass of the whole layer (permute -> gather -> FC1 +
SiTU -> FC2 -> combine; for MXFP8 / NVFP4 activations also their
quantisation) over one batch already resident in HBM.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload decode]
  python bench.py --impl reference ...     # the CPU oracle as reference arm
  python bench.py --peaks-only             # just the tensor-core peaks (JSON)

Timing: CUDA events on the launching stream around each step, a 256 MiB
write between steps flushes L2 (the events exclude it), max over ranks.
Under torchrun each rank runs its own replica of the layer (its own seed);
the layer needs no collective (each EP/TP rank produces a partial output
the caller all-reduces), so scaling is weak.

Roofline peaks: HBM from MEASURED_PEAKS.json; the tensor-core peak of each
GEMM is that of the MMA kind it runs (kind::mxf8f6f4 for the MXFP4 GEMMs,
kind::mxf4nvf4 for the NVFP4 FC1, kind::f16 bf16 for the NVFP4 FC2),
measured in the same run by the library's MMA-throughput kernel
(situ_tc_peak, one CTA per SM issuing back-to-back M=128 N=256 MMAs).
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "K3-shape MoE layer tokens/s and % of roofline (HBM or block-scaled TC), T=64/8192"
WORKLOAD_NAMES = {
    "decode": "Kimi-K3 TP8 decode layer, w4a16: T=64 H=3584 I=384 E=896 local, top-16 uniform, "
              "bf16 activations x MXFP4 weights",
    "prefill_w4a8": "Kimi-K3 TP8 prefill layer, w4a8: T=8192 H=3584 I=384 E=896, top-16 Zipf(1.0), "
                    "MXFP8 activations x MXFP4 weights",
    "ep_shard": "Kimi-K3 EP8 shard 3/8: T=4096 H=3584 I=3072 E_loc=112 offset 336, top-16 uniform, w4a16",
    "nvfp4": "Kimi-K3 NVFP4 layer: T=256 H=3584 I=384 E=896, top-16 Zipf(0.8), NVFP4 x NVFP4",
    "tiny": "tiny MoE: T=16 H=256 I=128 E=8 top-2, w4a16",
}
L2_FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0


FALLBACK_BF16_TFLOPS = 1900.0
TC_PEAKS_FILE = os.path.join(ROOT, "profiles", "tc_peaks.json")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def measure_tc_peaks(dev, reps: int = 8, target_ms: float = 20.0):
    """Dense TFLOP/s of each MMA kind on this GPU: ``reps`` launches of the
    library's MMA-throughput kernel, each sized to about ``target_ms``; the
    best launch is the burst peak, the median is reported beside it."""
    import torch
    from block_scaled_fp4_permute_gb300 import binding
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)

    def timed(kind, m):
        e0.record(stream)
        f = binding.situ_tc_peak(kind, m, status)
        e1.record(stream)
        e1.synchronize()
        return f, e0.elapsed_time(e1)

    out = {}
    for kind, name in binding.TC_KIND_NAMES.items():
        m = 4096
        timed(kind, m)                       # first launch: attributes, module load
        _, ms = timed(kind, m)
        m = int(max(4, min(1 << 30, m * target_ms / max(ms, 1e-3)))) // 4 * 4
        rates, times = [], []
        for _ in range(reps):
            f, ms = timed(kind, m)
            rates.append(f / (ms * 1e-3) / 1e12)
            times.append(ms)
        if int(status.item()) != 0:
            raise RuntimeError(f"situ_tc_peak({name}): device status {int(status.item())}")
        out[name] = {"tflops": max(rates), "tflops_median": float(np.median(rates)),
                     "mmas_per_sm": m, "launch_ms": float(np.median(times))}
    return out


def load_tc_peaks():
    """The committed microbenchmark result (used when no live measurement)."""
    if os.path.exists(TC_PEAKS_FILE):
        with open(TC_PEAKS_FILE) as f:
            return json.load(f).get("kinds")
    return None


def gemm_kinds(wl, h1_nvfp4=False):
    """The tensor-core MMA kind each GEMM of the layer runs on, by the path
    the shapes take (mirrors the library's host-side path choice)."""
    rows_per_expert = wl.T * wl.K / max(wl.E_total, 1)
    if wl.wt == 0 and wl.H % 128 == 0 and wl.I % 128 == 0:
        return {"fc1": "mxf8f6f4", "fc2": "mxf8f6f4"}
    if wl.wt == 1 and wl.act == 2 and rows_per_expert <= 512.0 and wl.H % 256 == 0 and wl.I % 128 == 0:
        return {"fc1": "mxf4nvf4", "fc2": "mxf4nvf4" if h1_nvfp4 else "bf16"}
    return {"fc1": "f16", "fc2": "f16"}


def tensor_peak_of(kind, tc):
    """(TFLOP/s, source) of one MMA kind: the live (or committed)
    microbenchmark for the block-scaled kinds, MEASURED_PEAKS.json's cuBLAS
    bf16 GEMM for bf16 / f16."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    bf16, bsrc = FALLBACK_BF16_TFLOPS, "fallback 1.9 PFLOP/s bf16"
    if os.path.exists(p):
        with open(p) as f:
            bf16 = float(json.load(f)["bf16_tflops"])
        bsrc = "measured bf16_tflops (MEASURED_PEAKS.json, cuBLAS bf16 GEMM burst)"
    if kind in ("bf16", "f16"):
        return bf16, bsrc
    if tc and kind in tc:
        return float(tc[kind]["tflops"]), f"measured kind::{kind} (situ_tc_peak microbenchmark, {tc.get('_source', 'this run')})"
    return 2.0 * bf16, bsrc + " x 2 (nominal fp8 : bf16 ratio; no microbenchmark result)"


def routing_stats(wl):
    ids = wl.host("topk_ids")
    kept = (ids >= wl.off) & (ids < wl.off + wl.E_loc)
    R = int(kept.sum())
    touched = int(np.unique(ids[kept]).size)
    return R, touched


def algorithmic_bytes(wl, R, touched, h1_nvfp4=False):
    """Bytes each stage must move at minimum (weights of touched experts
    once, activations and outputs once)."""
    H, I, T, K = wl.H, wl.I, wl.T, wl.K
    bs = 16 if wl.wt == 1 else 32
    w1 = touched * (2 * I * H // 2 + 2 * I * H // bs) + (touched * 8 if wl.wt == 1 else 0)
    w2 = touched * (H * I // 2 + H * I // bs) + (touched * 4 if wl.wt == 1 else 0)
    act_in = {0: T * H * 2, 1: T * H + T * H // 32, 2: T * H // 2 + T * H // 16 + 4 * T}[wl.act]
    # one token row as the GEMMs read it: the FC1 input in its contract format
    # (bf16, MXFP8 with its scale bytes, NVFP4 with its scales and global
    # scale) and H1 (MXFP8 for w4a8, bf16 otherwise)
    x_row = act_in / max(T, 1)
    h_row = I + I / 32 if wl.act == 1 else 2 * I
    # FC2 reads H1 as FC1 writes it, or as its NVFP4 requantisation
    h_in = I / 2 + I / 16 + 4 if h1_nvfp4 else h_row
    route = T * K * 8
    out = T * H * 2
    # bytes per element of the FC2 rows Y the combine reads: f16 + a scale byte
    # per 32 on the block-scaled prefill tiles, fp32 elsewhere
    blk_prefill = (wl.act in (0, 1) and wl.wt == 0 and H % 128 == 0 and I % 128 == 0
                   and T * K / max(wl.E_total, 1) > 6.0)
    y_bytes = 2 + 1 / 32 if blk_prefill else 4
    return {
        "permute": T * K * 4 + 2 * T * K * 4 + 2 * wl.E_loc * 4,
        # the input read once, the expert-ordered rows written once
        "gather": act_in + R * x_row,
        "fc1": w1 + R * x_row + R * h_row,
        "fc2": w2 + R * h_in + R * H * y_bytes,
        "combine": R * H * y_bytes + route + out,
        "quant": T * H * 2 + (T * H + T * H // 32 if wl.act == 1 else T * H // 2 + T * H // 16 + 4 * T),
        "layer": w1 + w2 + act_in + route + out,
    }


def layer_dtype(wl, h1_nvfp4=False):
    """The operand types the layer computes in (what the contract's formats
    are, not the tensor-core containers): bf16 or MXFP8 or NVFP4 activations
    times MXFP4 / NVFP4 weights, fp32 accumulation."""
    act = {0: "bf16", 1: "mxfp8", 2: "nvfp4"}[wl.act]
    w = {0: "mxfp4", 1: "nvfp4"}[wl.wt]
    h1 = "mxfp8" if wl.act == 1 else "nvfp4" if h1_nvfp4 else "bf16"
    return f"{act}x{w}->f32 (FC1), {h1}x{w}->f32 (FC2)"


def mma_containers(wl, h1_nvfp4=False):
    """How the tensor cores see the operands, per GEMM."""
    k = gemm_kinds(wl, h1_nvfp4)
    if k["fc1"] == "mxf8f6f4":
        rows = "bf16 rows as E4M3 hi + lo pairs (two MMAs per K block)" if wl.act == 0 else "E4M3 rows"
        return {"fc1": f"kind::mxf8f6f4, {rows} x E2M1 weights", "fc2": f"kind::mxf8f6f4, H1 as "
                + ("E4M3 hi + lo pairs" if wl.act == 0 else "E4M3 rows") + " x E2M1 weights"}
    if k["fc1"] == "mxf4nvf4":
        return {"fc1": "kind::mxf4nvf4, E2M1 x E2M1, E4M3 scales per 16",
                "fc2": ("kind::mxf4nvf4, requantised NVFP4 H1 x NVFP4 weights" if h1_nvfp4 else
                        "kind::f16, bf16 H1 x bf16-expanded NVFP4 weights")}
    return {"fc1": "kind::f16 / mma.sync on f16-expanded operands", "fc2": "same"}


def layer_flops(wl, R):
    return 2.0 * R * (wl.H * 2 * wl.I + wl.I * wl.H)


class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.dev)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
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
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(smax)) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def oracle_tokens_per_s(wl, budget_s: float, host_kw=None, max_tokens=None):
    """Time the oracle on a bounded token sample; returns (tok/s, n_tok, seconds, threads)."""
    import oracle
    from block_scaled_fp4_permute_gb300 import workloads as W
    if host_kw is None:
        host_kw = host_oracle_kwargs(wl)
    T = wl.T
    cap = min(max_tokens or T, T)
    # the oracle works expert by expert, so a small sample's time per token
    # overstates a large one's: size the sample in two steps
    n = min(T, 2)
    t0 = time.perf_counter()
    _oracle_run(oracle, W, wl, host_kw, n)
    dt = time.perf_counter() - t0
    for _ in range(2):
        if dt >= 0.5 * budget_s or n >= cap:
            break
        n = int(max(1, min(cap, round(n * budget_s / max(dt, 1e-6)))))
        t0 = time.perf_counter()
        _oracle_run(oracle, W, wl, host_kw, n)
        dt = time.perf_counter() - t0
    return n / dt, n, dt, oracle.get_threads()


def host_oracle_kwargs(wl):
    from block_scaled_fp4_permute_gb300 import workloads as W
    if wl.act in (W.ACT_MXFP8, W.ACT_NVFP4):
        return W.oracle_kwargs(wl), wl.host("x_bf16")
    return W.oracle_kwargs(wl), None


def _oracle_run(oracle, W, wl, host_kw, n):
    kw, xbits = host_kw
    toks = np.arange(n, dtype=np.int32)
    if xbits is not None and wl.act == W.ACT_MXFP8:   # the oracle's own quantisation is part of the step
        q, s = oracle.quant_mxfp8(xbits[:n])
        kw = dict(kw)
        qf = np.zeros((wl.T, wl.H), np.uint8)
        sf = np.zeros((wl.T, wl.H // 32), np.uint8)
        qf[:n], sf[:n] = q, s
        kw["hidden_states_q"], kw["hidden_states_scale"] = qf, sf
    elif xbits is not None:
        q, s, g = oracle.quant_nvfp4(xbits[:n])
        kw = dict(kw)
        qf = np.zeros((wl.T, wl.H // 2), np.uint8)
        sf = np.zeros((wl.T, wl.H // 16), np.uint8)
        gf = np.ones((wl.T,), np.float32)
        qf[:n], sf[:n], gf[:n] = q, s, g
        kw["hidden_states_q"], kw["hidden_states_scale"], kw["hidden_states_gscale"] = qf, sf, gf
    return oracle.moe_forward(**kw, tokens=toks)


def max_over_ranks(x: float, device) -> float:
    """The largest of every rank's x (the job's time is its slowest rank's);
    x itself on one rank or without a process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def make_workload(name, device, seed, tokens=None):
    from block_scaled_fp4_permute_gb300 import workloads as W
    return W.make(name, device=device, seed=seed, T=tokens)


def run_reference(args):
    """The oracle (CPU, as it stands) as the reference arm."""
    import torch
    ws, rank, _ = dist_env()
    if ws > 1 and rank != 0:
        return 0
    import oracle
    oracle.build()
    dev = "cuda:0" if torch.cuda.is_available() else "cpu"
    wl = make_workload(args.workload, dev, args.seed, args.tokens)
    host_kw = host_oracle_kwargs(wl)
    per_step = max(0.5, 120.0 / max(1, args.steps + args.warmup))
    _, n, _, threads = oracle_tokens_per_s(wl, per_step, host_kw)
    from block_scaled_fp4_permute_gb300 import workloads as W
    for _ in range(args.warmup):
        _oracle_run(oracle, W, wl, host_kw, n)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_run(oracle, W, wl, host_kw, n)
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    value = n / dt
    sample = f"{n} of {wl.T} tokens per step ({wl.name} workload), all local experts"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_NAMES[args.workload], "T": wl.T},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def pack_inputs(wl):
    """Rebinds the workload's per-step inputs (x_bf16, topk_ids,
    topk_weights) as views into one uint8 device buffer, each at a 256-byte
    aligned offset, and returns the buffer."""
    import torch
    ts = [wl.x_bf16, wl.topk_ids, wl.topk_weights]
    offs, o = [], 0
    for t in ts:
        offs.append(o)
        o += -(-t.numel() * t.element_size() // 256) * 256
    buf = torch.empty(max(o, 256), dtype=torch.uint8, device=wl.x_bf16.device)
    views = []
    for t, off in zip(ts, offs):
        n = t.numel() * t.element_size()
        v = buf[off:off + n].view(t.dtype).view(t.shape)
        v.copy_(t)
        views.append(v)
    wl.x_bf16, wl.topk_ids, wl.topk_weights = views
    return buf


def measure_workload(name, args, dev, rank, ws, tc, sampler_dev, cpu_budget):
    """Times one workload: the plain C-ABI forward for ``args.steps`` steps
    (events around each), per-stage times from the profiled call, and the
    end-to-end call with host buffers.  Returns the record (dict)."""
    import torch
    from block_scaled_fp4_permute_gb300 import binding

    wl = make_workload(name, dev, args.seed + rank, args.tokens if name == args.workload else None)
    # a step's inputs (activations, top-k IDs and weights) as views into one
    # device buffer, so that the end-to-end step moves them in one copy
    packed = pack_inputs(wl)
    layer = binding.Layer(wl, fuse_combine=args.fuse_combine, h1_nvfp4=args.h1_nvfp4 and wl.act == 2)
    R, touched = routing_stats(wl)
    h1nv = bool(args.h1_nvfp4 and wl.act == 2)
    nbytes = algorithmic_bytes(wl, R, touched, h1nv)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    nst = len(binding.PROFILE_STAGES)
    is_q = wl.act != binding.SITU_ACT_BF16   # the step includes the activation quantisation
    qname = "quant_mxfp8" if wl.act == binding.SITU_ACT_MXFP8 else "quant_nvfp4"

    def new_events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record(stream)     # creates the underlying cudaEvent_t
        return evs

    # the timed steps are the plain forward call (events only around it); the
    # per-stage times come from a second pass of the profiled call, whose
    # events between the kernels keep them from overlapping
    bounds = [new_events(2) for _ in range(args.steps)]
    n_prof = min(args.steps, 50)
    steps = [new_events(nst + 1) for _ in range(n_prof)]
    qevs = [new_events(2) for _ in range(n_prof)] if is_q else None
    for _ in range(args.warmup):
        flush.zero_()
        layer()
    torch.cuda.synchronize()

    sampler = ClockSampler(sampler_dev)
    sampler.start()
    time.sleep(0.25)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    graph = layer.capture() if args.graph else None
    for i in range(args.steps):
        flush.zero_()
        bounds[i][0].record(stream)
        if graph is not None:
            graph.replay()
        else:
            layer()
        bounds[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    clocks = sampler.stop()
    if layer.device_status() != 0:
        raise RuntimeError(f"{name}: a kernel gave up a bounded wait (device status {layer.device_status()})")
    for i in range(n_prof):
        flush.zero_()
        layer.profiled(steps[i], qevs[i] if is_q else None)
    torch.cuda.synchronize()

    stage_ms = np.zeros(nst)
    quant_ms = 0.0
    for i, evs in enumerate(steps):
        for s_ in range(nst):
            stage_ms[s_] += evs[s_].elapsed_time(evs[s_ + 1])
        if is_q:
            quant_ms += qevs[i][0].elapsed_time(qevs[i][1])
    stage_ms /= n_prof
    quant_ms /= n_prof
    step_ms = np.array([b[0].elapsed_time(b[1]) for b in bounds])
    ms = max_over_ranks(float(step_ms.mean()), dev)

    # end to end: pinned host inputs -> device (one copy of the packed
    # buffer), layer, output -> pinned host
    dev_in = [packed]
    host_in = [t.cpu().pin_memory() for t in dev_in]
    host_out = torch.empty(layer.out.shape, dtype=layer.out.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host_in)   # the packed inputs, with their alignment gaps
    d2h = host_out.numel() * host_out.element_size()
    e_ms = []
    for i in range(max(args.warmup, 1) + args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for d, h in zip(dev_in, host_in):
            d.copy_(h, non_blocking=True)
        layer()
        host_out.copy_(layer.out, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        if i >= max(args.warmup, 1):
            e_ms.append(e0.elapsed_time(e1))
    e2e_ms = max_over_ranks(float(np.mean(e_ms)), dev)

    hbm, peak_kind = peaks()
    stages = {}
    for s_, sname in enumerate(binding.PROFILE_STAGES):
        gbs = nbytes[sname] / (stage_ms[s_] * 1e-3) / 1e9 if stage_ms[s_] > 0 else None
        stages[sname] = {"ms": float(stage_ms[s_]), "alg_bytes": int(nbytes[sname]),
                         "gbs": gbs, "frac_hbm": gbs / hbm if gbs else None}
    if is_q:
        gbs = nbytes["quant"] / (quant_ms * 1e-3) / 1e9
        stages[qname] = {"ms": quant_ms, "alg_bytes": int(nbytes["quant"]), "gbs": gbs, "frac_hbm": gbs / hbm}
    kinds = gemm_kinds(wl, h1nv)
    kflops = {"fc1": 2.0 * R * wl.H * 2 * wl.I, "fc2": 2.0 * R * wl.I * wl.H}
    for g in ("fc1", "fc2"):
        pk, _ = tensor_peak_of(kinds[g], tc)
        stages[g]["tflops"] = kflops[g] / (stage_ms[binding.PROFILE_STAGES.index(g)] * 1e-3) / 1e12 \
            if stages[g]["ms"] > 0 else None
        stages[g]["mma_kind"] = kinds[g]
        stages[g]["frac_tensor"] = stages[g]["tflops"] / pk if stages[g]["tflops"] else None
    dom = max(stages, key=lambda k: stages[k]["ms"])
    traffic = None
    tpath = os.path.join(ROOT, "profiles", f"traffic_{name}.json")
    if os.path.exists(tpath):
        with open(tpath) as f:
            tj = json.load(f)
        # counters of a capture at this token count, of the current kernels only
        if tj.get("T") == wl.T and not tj.get("stale"):
            traffic = tj.get(dom)
    # the bound of the dominant kernel and of the layer: the larger of the
    # HBM time of its algorithmic bytes and the tensor time of its FLOPs (each
    # GEMM against the peak of its own MMA kind)
    hbm_src = (f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
               else "fallback 6.8 TB/s")
    kf = kflops.get(dom, 0.0)
    if dom in kinds:
        tc_peak, tc_src = tensor_peak_of(kinds[dom], tc)
    else:
        tc_peak, tc_src = float("inf"), "-"
    if kf / (tc_peak * 1e12) > nbytes[dom] / (hbm * 1e9):
        ach = kf / (stages[dom]["ms"] * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": dom, "achieved": ach, "peak": tc_peak,
                "unit": "TFLOP/s", "frac": ach / tc_peak, "traffic": traffic, "peak_source": tc_src,
                "mma_kind": kinds[dom]}
    else:
        roof = {"bound": "hbm", "kernel": dom, "achieved": stages[dom]["gbs"], "peak": hbm,
                "unit": "GB/s", "frac": stages[dom]["frac_hbm"], "traffic": traffic,
                "peak_source": hbm_src}
    layer_gbs = nbytes["layer"] / (ms * 1e-3) / 1e9
    flops = layer_flops(wl, R)
    t_hbm = nbytes["layer"] / (hbm * 1e9)
    t_tc = sum(kflops[g] / (tensor_peak_of(kinds[g], tc)[0] * 1e12) for g in ("fc1", "fc2"))
    # one number for "the" tensor peak of the layer: its FLOPs over the
    # per-kind tensor time
    layer_tc_peak = flops / t_tc / 1e12

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        tps, n, dt, threads = oracle_tokens_per_s(wl, cpu_budget)
        cpu = {"value": tps, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"{n} of {wl.T} tokens of the same workload, {dt:.1f} s"}

    rec = {
        "value": ws * wl.T / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
        "dtype": layer_dtype(wl, h1nv), "mma": mma_containers(wl, h1nv),
        "config": {"workload": WORKLOAD_NAMES[name], "T": wl.T, "H": wl.H, "I": wl.I,
                   "E_total": wl.E_total, "E_loc": wl.E_loc, "offset": wl.off, "top_k": wl.K,
                   "kept_pairs": R, "touched_experts": touched,
                   "l2": "flushed between steps (256 MiB write, outside the step events)",
                   "parallelism": f"replicas x{ws}, no collective",
                   "launch": "CUDA graph replay of the layer call" if args.graph else "eager C-ABI call",
                   "combine": "fused into FC2 (fp32 reductions)" if args.fuse_combine
                   else "separate kernel, ascending slot order",
                   "h1": ("NVFP4, requantised per token (opt-in)" if args.h1_nvfp4 and wl.act == 2 else
                          "MXFP8" if wl.act == 1 else "bf16"),
                   "step": ("MXFP8 quantisation of the bf16 input + " if wl.act == 1 else
                            "NVFP4 quantisation of the bf16 input + " if wl.act == 2 else "")
                   + "the whole layer"},
        "roofline": roof,
        "layer_roofline": {"bound": "tensor" if t_tc > t_hbm else "hbm", "alg_bytes": int(nbytes["layer"]),
                           "flops": flops, "roofline_ms": max(t_hbm, t_tc) * 1e3,
                           "frac": max(t_hbm, t_tc) / (ms * 1e-3),
                           "gbs": layer_gbs, "frac_hbm": layer_gbs / hbm,
                           "tflops": flops / (ms * 1e-3) / 1e12, "tensor_peak_tflops": layer_tc_peak,
                           "frac_tensor": flops / (ms * 1e-3) / 1e12 / layer_tc_peak,
                           "t_hbm_ms": t_hbm * 1e3, "t_tensor_ms": t_tc * 1e3},
        "stages": stages,
        "e2e": {"value": ws * wl.T / (e2e_ms * 1e-3), "unit": "tokens/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "stage_times": f"per-kernel ms from {n_prof} further steps of the profiled call (events between kernels)",
        "gpu_launches": layer.launches() * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": wall,
        "cpu_baseline": cpu,
    }
    del layer, wl, flush
    torch.cuda.empty_cache()
    return rec


def run_ours(args):
    import torch
    import torch.distributed as dist
    from block_scaled_fp4_permute_gb300 import build

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")
    build.build()
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    sampler_dev = vis.split(",")[local].strip() if vis else local

    # tensor-core peaks of the MMA kinds, measured on this GPU now
    tc, tc_clocks = None, None
    if not args.no_tc_peaks:
        sampler = ClockSampler(sampler_dev)
        sampler.start()
        tc = measure_tc_peaks(dev)
        tc_clocks = sampler.stop()
        tc["_source"] = "this run"
    else:
        tc = load_tc_peaks()
        if tc:
            tc["_source"] = "profiles/tc_peaks.json"
    if args.peaks_only:
        if rank == 0:
            print(json.dumps({"kinds": {k: v for k, v in tc.items() if not k.startswith("_")},
                              "clocks": tc_clocks, "gpu": torch.cuda.get_device_name(dev),
                              "how": "situ_tc_peak: one CTA per SM, back-to-back M=128 N=256 MMAs into one TMEM "
                                     "accumulator, operands in shared memory; best (and median) of 8 launches of "
                                     "about 20 ms, CUDA events"}), flush=True)
        if ws > 1:
            dist.destroy_process_group()
        return 0

    main = measure_workload(args.workload, args, dev, rank, ws, tc, sampler_dev, args.cpu_budget)
    line = {"metric": METRIC, "value": main["value"], "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": main["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "data": "synthetic (seeded; weights N(0,0.02) packed to "
            "the block-scaled format)"}
    line.update({k: v for k, v in main.items() if k not in ("value", "unit", "ms_per_step")})
    if tc:
        line["tc_peaks"] = {k: v for k, v in tc.items() if not k.startswith("_")}
        line["tc_peaks_clocks"] = tc_clocks
    # the second half of the metric (T=8192 prefill) rides on the same line
    if args.workload == "decode" and not args.no_prefill and args.tokens is None:
        rec = measure_workload("prefill_w4a8", args, dev, rank, ws, tc, sampler_dev, args.cpu_budget)
        rec["steps"], rec["warmup"] = args.steps, args.warmup
        line["prefill_w4a8_8192"] = rec
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=tuple(WORKLOAD_NAMES), default="decode")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the workload's token count T (smaller profiling captures); "
                         "the JSON line's config then carries that T")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="leave out the T=8192 w4a8 prefill record of the decode line")
    ap.add_argument("--no-tc-peaks", action="store_true",
                    help="take the tensor-core peaks from profiles/tc_peaks.json instead of measuring them")
    ap.add_argument("--peaks-only", action="store_true",
                    help="measure the tensor-core peaks of the MMA kinds and print them as JSON")
    ap.add_argument("--graph", action="store_true",
                    help="time replays of a CUDA graph of the layer call instead of eager C-ABI calls")
    ap.add_argument("--h1-nvfp4", action="store_true",
                    help="NVFP4 workload: requantise H1 per token to NVFP4 and run FC2 as NVFP4 x NVFP4")
    ap.add_argument("--fuse-combine", action="store_true",
                    help="FC2 adds weight * Y into an fp32 accumulator (block-scaled prefill tiles); "
                         "not bitwise reproducible run to run")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
