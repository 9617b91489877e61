#!/usr/bin/env python
"""Throughput of the GB300 MoE FFN layer forward pass (tokens/s).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload decode|prefill|...]
    python bench.py --impl reference ...     # the CPU oracle, timed on the host cores

One step = one pass of the whole layer (route -> permute -> expert FFN +
shared expert -> combine) over one batch of T synthetic tokens whose inputs
and weights are already resident in HBM.  The timed region is exactly K steps
between a barrier + device synchronisation on each side; every stage is
bracketed by CUDA events on the launching stream, which gives the per-stage
times the roofline uses.  The end-to-end figure repeats the measurement
through the public call with host buffers (pinned x in, y out, copies inside
the timed region).

Multi-GPU (torchrun, one process per GPU): the layer is per-token
independent, so ranks are independent replicas of the same workload (weak
scaling, no collective on the data path); value = tokens of all ranks / the
slowest rank's time.  Rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s at T=8192 and T=64; % of FP8-TC / HBM roofline"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

WORKLOAD_TEXT = {
    "decode": "decode step: T=64 tokens, d_model=4096, 128 experts, top-6 softmax routing, SwiGLU f=1024, "
              "1 shared expert f=1024, FP8 E4M3 weights with per-channel fp32 scales, bf16 x",
    "prefill": "chunked prefill: T=8192 tokens (32 x 256), d_model=4096, 128 experts, top-6, SwiGLU f=1024, "
               "1 shared expert f=1024, FP8 E4M3 weights, bf16 x",
    "skew": "skewed routing: T=4096, Zipf(1.2)-biased router (hottest expert ~8x mean, 4+ empty), FP8 weights",
    "100b_decode": "100B-style decode: T=64, d_model=4096, 128 experts, top-8, SwiGLU f=2048, NVFP4 weights",
    "100b_prefill": "100B-style prefill: T=8192, d_model=4096, 128 experts, top-8, SwiGLU f=2048, NVFP4 weights",
    "tiny": "tiny: T=32, d_model=128, 128 experts, top-6, f=64, all fp32",
    "qk_norm_rope": "fused QK-norm + RoPE alone (the attention block's step): T=8192, 32 query / 4 key heads of 128",
}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


# ------------------------------------------------------------------ algorithmic work

def weight_bytes_per_expert(cfg):
    d, f = cfg.d, cfg.f
    n = 3 * d * f
    if cfg.w_dtype == "e4m3":
        return n + 4 * (2 * f + d)
    if cfg.w_dtype == "nvfp4":
        return n // 2 + n // 16 + 8
    return 4 * n


def shared_weight_bytes(cfg):
    d, fs = cfg.d, cfg.fs
    n = 3 * d * fs
    if cfg.w_dtype == "e4m3":
        return n + 4 * (2 * fs + d)
    if cfg.w_dtype == "nvfp4":
        return n // 2 + n // 16 + 8
    return 4 * n


def algorithmic(cfg, counts):
    """Bytes and FLOPs of one layer pass (activated work only).

    Layer bytes: weights of the experts that received tokens + shared-expert
    weights + router weights + x (read) + y (fp32, written).
    Expert-FFN stage bytes (the dominant stage): active expert weights +
    shared weights + x + its outputs out_perm [T*k, d] and shared_out [T, d]
    (fp32).  FLOPs: 6*d*f per routed pair + 6*d*f_s per token (+ router).
    """
    active = int((counts > 0).sum())
    xb = cfg.T * cfg.d * (2 if cfg.x_dtype == "bf16" else 4)
    wexp = active * weight_bytes_per_expert(cfg) + shared_weight_bytes(cfg)
    P = cfg.T * cfg.k
    ffn_bytes = wexp + xb + 4 * (P + cfg.T) * cfg.d
    layer_bytes = wexp + 4 * cfg.E * cfg.d + xb + 4 * cfg.T * cfg.d
    ffn_flops = 6.0 * cfg.d * cfg.f * P + 6.0 * cfg.d * cfg.fs * cfg.T
    layer_flops = ffn_flops + 2.0 * cfg.T * cfg.d * cfg.E
    return dict(active=active, ffn_bytes=ffn_bytes, layer_bytes=layer_bytes, ffn_flops=ffn_flops,
                layer_flops=layer_flops)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu_index = gpu_index

    def __enter__(self):
        if self.gpu_index is None:
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.1)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def keep_busy(step, seconds, torch, dev):
    """Untimed passes for about `seconds` (in groups of 8, synchronised), so
    that the clock samples around a short timed region see the GPU under the
    same load and nvidia-smi's start-up falls outside the timed region."""
    t_end = time.perf_counter() + seconds
    while time.perf_counter() < t_end:
        for _ in range(8):
            step()
        torch.cuda.synchronize(dev)


# ------------------------------------------------------------------ CPU oracle timing

def time_oracle(inp, budget_s, chunk=2):
    """Oracle tokens/s on a bounded sample: consecutive tokens in chunks
    (wrapping around the batch) until the budget is spent, at least one chunk."""
    import oracle
    T = inp.cfg.T
    done, pos, t0 = 0, 0, time.perf_counter()
    while True:
        n = min(chunk, T - pos)
        oracle.layer_forward_tokens(inp, range(pos, pos + n))
        done += n
        pos = (pos + n) % T
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    return done / el, done, el


def oracle_one_thread(name, budget_s):
    """The oracle on one host thread (BLAS and OpenMP pools limited to one
    thread in a child process, set before numpy loads): tokens/s of `name`."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", VECLIB_MAXIMUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-sample", name, "--cpu-budget", str(budget_s),
           "--warmup", "3"]
    try:
        r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=300)
        line = [ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1]
        return json.loads(line)
    except (subprocess.SubprocessError, IndexError, ValueError) as e:
        return {"unavailable": f"{type(e).__name__}"}


def oracle_sample_main(name, budget_s):
    import moe_synth
    inp = moe_synth.make_inputs(name)
    v, n, el = time_oracle(inp, budget_s)
    print(json.dumps({"value": v, "unit": "tokens/s", "threads": 1, "tokens": n, "seconds": el}), flush=True)


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ traffic record

def source_hash(files=None):
    """Hash of the kernel sources a record was measured on: the listed files
    of csrc/ (every file when None)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "top_routed_expert_gb300", "csrc")
    for fn in sorted(files if files is not None else os.listdir(csrc)):
        with open(os.path.join(csrc, fn), "rb") as fh:
            h.update(fn.encode() + fh.read())
    return h.hexdigest()[:16]


# flags that change which kernels (or how many bytes) the expert stage runs
TRAFFIC_VARIANT_FLAGS = ("MOE_FLAG_SIMT_FFN", "MOE_FLAG_BF16_EXPERT_OUT", "MOE_FLAG_ACT_E4M3", "MOE_FLAG_ACT_NVFP4",
                         "MOE_FLAG_NVFP4_F16")


def traffic_key(workload, flags):
    """Key of a workload's DRAM-traffic record: the workload name, plus every
    kernel-changing flag that is set (records exist for the default flags)."""
    from top_routed_expert_gb300 import abi
    on = [n for n in TRAFFIC_VARIANT_FLAGS if flags & getattr(abi, n)]
    return "+".join([workload] + on)


def recorded_traffic(workload, kernel):
    """dram bytes per launch from a committed ncu summary, if it was taken on
    the current sources of the kernels it covers (a record lists them under
    "sources"; without the list, every kernel source counts), else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        rec = json.load(fh)
    r = rec.get(workload, {})
    if r.get("kernel") != kernel:
        return None
    try:
        current = source_hash(r.get("sources"))
    except OSError:                      # a listed source no longer exists
        return None
    if r.get("source_hash") != current:
        return None
    return r.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ multi-rank aggregation

def max_over_ranks(ms, world, dev):
    """The slowest rank's time per step: the job is as slow as its slowest
    replica (all_reduce MAX over the process group; `dev` is where the
    reduction tensor lives: the rank's GPU under NCCL, "cpu" under gloo)."""
    if world <= 1:
        return float(ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world, T, ms):
    """Whole-job tokens/s: each of the `world` replicas processes T tokens per
    step of `ms` milliseconds (the slowest rank's time)."""
    return world * T / (ms / 1e3)


# ------------------------------------------------------------------ arms

def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def run_reference_qk(args):
    """The QK-norm + RoPE oracle on the host cores: 64 tokens per step."""
    import moe_synth
    from oracle import qk_rope_oracle as qr
    inp = moe_synth.make_qk_inputs()
    n = 64

    def step(i):
        sl = slice((i * n) % inp.T, (i * n) % inp.T + n)
        qf = (inp.q[sl].astype(np.uint32) << 16).view(np.float32)
        kf = (inp.k[sl].astype(np.uint32) << 16).view(np.float32)
        qr.qk_norm_rope(qf, kf, inp.gamma_q, inp.gamma_k, inp.cos_sin, inp.positions[sl])
    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    el = time.perf_counter() - t0
    v = n * args.steps / el
    print(json.dumps({
        "impl": "reference", "metric": "fused QK-norm + RoPE tokens/s (the pages' other fused kernel)", "value": v,
        "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * el / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded q, k, gammas; float32 RoPE table)",
        "config": {"workload": WORKLOAD_TEXT["qk_norm_rope"]},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores(), "kind": "oracle",
                         "sample": f"each step: the fp64 oracle on {n} of the {inp.T} tokens"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}), flush=True)


def run_reference(args, world, rank):
    """The oracle, as it stands, on the host cores (rank 0 only)."""
    if rank != 0:
        return
    import moe_synth
    if args.workload == "qk_norm_rope":
        return run_reference_qk(args)
    inp = moe_synth.make_inputs(args.workload)
    chunk = 2
    for _ in range(args.warmup):
        time_oracle(inp, 0.0, chunk)
    t0 = time.perf_counter()
    toks = 0
    for _ in range(args.steps):
        _, n, _ = time_oracle(inp, 0.0, chunk)
        toks += n
    el = time.perf_counter() - t0
    v = toks / el
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) activations, N(0,1/d) weights quantised to the stored format)",
        "config": {"workload": WORKLOAD_TEXT[args.workload], "T": inp.cfg.T},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores(), "kind": "oracle",
                         "sample": f"each step: the fp64 CPU oracle on {chunk} of the {inp.cfg.T} tokens "
                                   f"(routing + every expert they use, dequantised one at a time)"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def measure(layer, x, cfg, steps, warmup, world, dev, gpu_index, abi, torch, clocks=True):
    """Times `steps` passes of the layer (four ABI calls with CUDA events
    between the stages) and returns timings, algorithmic work and clocks."""
    T, k, E, d = cfg.T, cfg.k, cfg.E, cfg.d
    P = T * k
    c = layer.config(T)
    ws = layer.workspace(T)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    offs = torch.empty(E + 1, dtype=torch.int32, device=dev)
    sp = torch.empty(P, dtype=torch.int32, device=dev)
    row_of = torch.empty(P, dtype=torch.int32, device=dev)
    edt = torch.bfloat16 if (layer.flags & abi.MOE_FLAG_BF16_EXPERT_OUT) else torch.float32
    out_perm = torch.empty((P, d), dtype=edt, device=dev)
    shared = torch.empty((T, d), dtype=edt, device=dev)
    y = torch.empty((T, d), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        abi.moe_route(c, x, layer.w_router, layer.bias, ids, w, ws, stream)
        if ev is not None:
            ev[1].record(stream)
        abi.moe_permute(c, ids, offs, sp, row_of, ws, stream)
        if ev is not None:
            ev[2].record(stream)
        abi.moe_expert_ffn(c, x, w, offs, sp, layer.weights, out_perm, shared, ws, stream)
        if ev is not None:
            ev[3].record(stream)
        abi.moe_combine(c, out_perm, row_of, shared, y, stream)
        if ev is not None:
            ev[4].record(stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(warmup):
        step()
    st = abi.moe_get_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {abi.STATUS.get(st, st)}")
    counts = np.diff(offs.cpu().numpy())
    alg = algorithmic(cfg, counts)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    clk = ClockSampler(gpu_index if clocks else None)
    with clk:
        keep_busy(step, 0.4 if clocks else 0.0, torch, dev)
        barrier()
        launches0 = abi.moe_launch_count()
        for i in range(steps):
            step(evs[i])
        barrier()
        launches = abi.moe_launch_count() - launches0   # this library's kernels in the timed steps
        keep_busy(step, 0.3 if clocks else 0.0, torch, dev)
    st = abi.moe_get_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {abi.STATUS.get(st, st)}")
    total_ms = evs[0][0].elapsed_time(evs[-1][4])
    stage_ms = {name: sum(e[j].elapsed_time(e[j + 1]) for e in evs) / steps
                for j, name in enumerate(["route", "permute", "expert_ffn", "combine"])}
    ms_step = max_over_ranks(total_ms / steps, world, dev)
    return dict(ms_step=ms_step, stage_ms=stage_ms, alg=alg, launches=launches, clocks=clk.summary())


def time_graph(layer, x, steps, warmup, world, dev, torch, gpu_index=None):
    """K replays of the layer captured as one CUDA graph, between a barrier +
    device synchronisation on each side, with the SM clocks sampled meanwhile;
    returns (ms per step (max over ranks), clock summary)."""
    graph, _ = layer.capture(x)
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        graph.replay()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_index) as clk:
        keep_busy(graph.replay, 0.4, torch, dev)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)
        g0.record(stream)
        for _ in range(steps):
            graph.replay()
        g1.record(stream)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)
        keep_busy(graph.replay, 0.3, torch, dev)
    ms = max_over_ranks(g0.elapsed_time(g1) / steps, world, dev)
    return ms, clk.summary()


# Workloads whose metric point is the tensor roofline (the two T = 8192
# batches); the rest report the slower of the two bounds.
TENSOR_WORKLOADS = ("prefill", "100b_prefill")


def nvfp4_on_f16_path(cfg, flags):
    """Whether the library runs these NVFP4 weights on the f16-rebuild path:
    when forced, or for the exact contract at more than 16 routed rows per
    expert on average (the block-scaled path takes decode-sized batches and
    every batch with NVFP4 activations)."""
    if flags & 0x20:          # MOE_FLAG_NVFP4_F16
        return True
    if flags & 0x10:          # MOE_FLAG_ACT_NVFP4
        return False
    return cfg.T * cfg.k > 16 * cfg.E


def roofline(alg, ms_ffn, ms_step, workload, w_dtype="e4m3", simt=False, act_terms=None, nvfp4_f16=False,
             traffic_key=None):
    """Roofline of the dominant stage (moe_expert_ffn) and of the whole layer.

    HBM bound: algorithmic bytes at the measured copy bandwidth.  Tensor
    bound: the layer's expert FLOPs (6*d*f per pair + 6*d*f_s per token) at
    the dense peak of the weight format (FP8 = 2x, FP4 = 4x the measured bf16
    cuBLAS rate).  `issued` adds what the tensor pipe really executes: FP8
    weights meet two E4M3 terms per activation by default (2x the FLOPs at
    the FP8 rate) or one (MOE_FLAG_ACT_E4M3); NVFP4 weights meet four NVFP4
    activation terms by default (4x the FLOPs at the FP4 rate) or one
    (MOE_FLAG_ACT_NVFP4), or are rebuilt exactly in f16 (MOE_FLAG_NVFP4_F16:
    1x at the bf16 rate).
    """
    if act_terms is None:
        act_terms = 4 if w_dtype == "nvfp4" else 2
    peaks, peak_src = load_peaks()
    hbm = peaks["hbm_gbs"]
    bf16 = peaks["bf16_tflops"]
    lowp = 4.0 if w_dtype == "nvfp4" else 2.0
    tc_peak = lowp * bf16
    ffn_s = ms_ffn / 1e3
    t_hbm = alg["ffn_bytes"] / (hbm * 1e9)
    t_tc = alg["ffn_flops"] / (tc_peak * 1e12)
    tensor = workload in TENSOR_WORKLOADS if not simt else False
    if not tensor and t_hbm >= t_tc:
        roof = {"bound": "hbm", "achieved": alg["ffn_bytes"] / ffn_s / 1e9, "peak": hbm, "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": alg["ffn_flops"] / ffn_s / 1e12, "peak": tc_peak, "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["kernel"] = "moe_expert_ffn (grouped SwiGLU GEMMs + shared expert)"
    fmt = "FP4 dense = 4" if w_dtype == "nvfp4" else "FP8 dense = 2"
    roof["peak_source"] = (f"{peak_src}: " + ("HBM copy GB/s" if roof["bound"] == "hbm"
                                              else f"{fmt} x bf16 cuBLAS TFLOP/s"))
    if roof["bound"] == "tensor" and not simt:
        if w_dtype == "nvfp4" and nvfp4_f16:
            issued = {"tflops": alg["ffn_flops"] / ffn_s / 1e12, "peak": bf16,
                      "how": "weights rebuilt exactly in f16: kind::f16 MMAs at the bf16/f16 rate"}
        elif w_dtype == "nvfp4":
            issued = {"tflops": act_terms * alg["ffn_flops"] / ffn_s / 1e12, "peak": tc_peak,
                      "how": (f"{act_terms} NVFP4 terms per activation row: block-scaled kind::mxf4nvf4 MMAs issue "
                              f"{act_terms}x the layer's FLOPs at the FP4 rate")}
        elif act_terms == 2:
            issued = {"tflops": 2.0 * alg["ffn_flops"] / ffn_s / 1e12, "peak": 2.0 * bf16,
                      "how": "two E4M3 terms per activation: the FP8 MMAs (kind::f8f6f4, or block-scaled kind::mxf8f6f4 on CTA pairs) issue 2x the FLOPs"}
        else:
            issued = {"tflops": alg["ffn_flops"] / ffn_s / 1e12, "peak": 2.0 * bf16,
                      "how": "one E4M3 term per activation (MOE_FLAG_ACT_E4M3): the MMAs issue the layer's FLOPs"}
        issued["frac"] = issued["tflops"] / issued["peak"]
        roof["issued"] = issued
    # a variant (a flag that changes the kernels) has no record unless one was
    # captured under its own key
    roof["traffic"] = recorded_traffic(traffic_key or workload, roof["kernel"])
    t_layer_roof = max(alg["layer_bytes"] / (hbm * 1e9), alg["layer_flops"] / (tc_peak * 1e12))
    return roof, t_layer_roof / (ms_step / 1e3)


def qk_rope_point(args, world, dev, gpu_index, abi, torch):
    """moe_qk_norm_rope on the T = 8192 prefill batch (32 query / 4 key heads
    of 128).  q and k (75 MB) fit in L2, so a 512 MB buffer is read between
    launches (which leaves L2 full of clean lines: no write-back of the flush
    lands inside the timed launch) and each launch is timed alone with CUDA
    events on the launching stream; the roofline is HBM: q and k read and
    written once, plus the table rows, positions and gammas."""
    import moe_synth
    from top_routed_expert_gb300.layer import _to_dev
    inp = moe_synth.make_qk_inputs()
    q, k = _to_dev(inp.q, dev).clone(), _to_dev(inp.k, dev).clone()
    gq, gk = _to_dev(inp.gamma_q, dev), _to_dev(inp.gamma_k, dev)
    cs, pos = _to_dev(inp.cos_sin, dev), _to_dev(inp.positions, dev)
    cfg = abi.moe_qk_rope_config_t(inp.T, inp.n_q_heads, inp.n_kv_heads, inp.head_dim, inp.n_pos, 1e-6)
    flush = torch.ones(128 << 20, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    steps = max(5, args.steps)
    for _ in range(args.warmup):
        abi.moe_qk_norm_rope(cfg, q, k, gq, gk, cs, pos, stream)
    if abi.moe_get_device_status(stream) != 0:
        raise RuntimeError("moe_qk_norm_rope reported a device fault")
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with ClockSampler(gpu_index) as clk:
        torch.cuda.synchronize(dev)
        for e0, e1 in evs:
            flush.sum()
            e0.record(stream)
            abi.moe_qk_norm_rope(cfg, q, k, gq, gk, cs, pos, stream)
            e1.record(stream)
        torch.cuda.synchronize(dev)
    us = max_over_ranks(sum(e0.elapsed_time(e1) for e0, e1 in evs) / steps, world, dev) * 1e3
    rows = inp.T * (inp.n_q_heads + inp.n_kv_heads)
    n_used = len(np.unique(inp.positions))
    bytes_ = 2 * rows * inp.head_dim * 2 + n_used * inp.head_dim // 2 * 8 + 4 * inp.T + 2 * 4 * inp.head_dim
    peaks, src = load_peaks()
    achieved = bytes_ / (us * 1e-6) / 1e9
    return {"workload": f"fused QK-norm + RoPE, in place: T={inp.T}, {inp.n_q_heads} query / {inp.n_kv_heads} key heads "
                        f"of {inp.head_dim}, bf16, rotate-half RoPE from a {inp.n_pos}-row float32 table",
            "value": job_value(world, inp.T, us / 1e3), "unit": "tokens/s", "us_per_launch": us, "steps": steps,
            "l2": "512 MB read between launches (q and k, 75 MB, would otherwise stay in L2); each launch timed alone",
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"],
                         "traffic": recorded_traffic("qk_norm_rope", "qk_norm_rope_kernel"),
                         "kernel": "qk_norm_rope_kernel", "peak_source": f"{src}: HBM copy GB/s",
                         "algorithmic_bytes": bytes_},
            "pages_context": "Sarvam blog Table 1: 414 -> 54 us per layer on H100 (their batch size not given)",
            "clocks": clk.summary()}


def run_qk_only(args, world, rank, local):
    """--workload qk_norm_rope: the fused QK-norm + RoPE step alone, one JSON line."""
    import torch
    import top_routed_expert_gb300 as moe
    from top_routed_expert_gb300 import abi
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    moe.build()
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0]
    gpu_index = int(vis) if vis.isdigit() else local
    p = qk_rope_point(args, world, dev, gpu_index, abi, torch)
    if rank != 0:
        return
    line = {"metric": "fused QK-norm + RoPE tokens/s (the pages' other fused kernel)", "value": p["value"],
            "unit": "tokens/s", "n_gpus": world, "steps": p["steps"], "warmup": args.warmup,
            "ms_per_step": p["us_per_launch"] / 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16 in / out, fp32 arithmetic", "data": "synthetic (seeded q, k, gammas; float32 RoPE table)",
            "config": {"workload": WORKLOAD_TEXT["qk_norm_rope"], "l2": p["l2"]}, "roofline": p["roofline"],
            "clocks": p["clocks"], "gpu_launches": p["steps"], "cpu_baseline": None}
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    if args.workload == "qk_norm_rope":
        return run_qk_only(args, world, rank, local)
    import torch
    import moe_synth
    import top_routed_expert_gb300 as moe
    from top_routed_expert_gb300 import abi
    from top_routed_expert_gb300.layer import MoELayer, _to_dev

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    moe.build()
    inp = moe_synth.make_inputs(args.workload)
    cfg = inp.cfg
    flags = ((abi.MOE_FLAG_SIMT_FFN if args.simt else 0) | (abi.MOE_FLAG_BF16_EXPERT_OUT if args.bf16_expert_out else 0) |
             (abi.MOE_FLAG_ACT_E4M3 if args.act_e4m3 else 0))
    layer = MoELayer(inp, device=dev, flags=flags)
    x = _to_dev(inp.x, dev)
    T, d = cfg.T, cfg.d
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0]
    gpu_index = int(vis) if vis.isdigit() else local

    m = measure(layer, x, cfg, args.steps, args.warmup, world, dev, gpu_index, abi, torch)

    # end to end through the public call, host buffers
    stream = torch.cuda.current_stream(dev)
    x_host = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    x_host.copy_(x)
    y_host = torch.empty((T, d), dtype=torch.float32, pin_memory=True)
    x_stage = torch.empty_like(x)
    y_stage = torch.empty((T, d), dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        layer.forward_host(x_host, y_host, x_stage, y_stage, stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        layer.forward_host(x_host, y_host, x_stage, y_stage, stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)

    # the same layer pass replayed as one CUDA graph (no host launch gaps)
    graph_ms, graph_clk = time_graph(layer, x, args.steps, args.warmup, world, dev, torch, gpu_index)
    # and with the shared expert in the routed launches instead of beside the
    # routing on a second stream (MOE_FLAG_NO_OVERLAP), for comparison
    one_stream_ms = None
    if not args.simt:
        import copy
        l1 = copy.copy(layer)
        l1.flags = layer.flags | abi.MOE_FLAG_NO_OVERLAP
        one_stream_ms, _ = time_graph(l1, x, args.steps, args.warmup, world, dev, torch, None)
        del l1
    st = abi.moe_get_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {abi.STATUS.get(st, st)}")

    # further points of the metric, each with its own roofline: the T = 8192
    # prefill (the metric's second point) and the skewed batch on the same
    # resident FP8 weights (the generator draws identical expert weights for
    # every FP8 workload), then the 100B-style NVFP4 layer at T = 64 and 8192
    points = {}
    if args.workload == "decode" and not args.no_prefill:
        def point(lay, name, steps, act_terms=None, flag_note=None, nvfp4_f16=False):
            src = moe_synth.make_inputs(name, router_only=True)
            if src.bias is not None:
                import copy
                lay = copy.copy(lay)
                lay.bias = _to_dev(src.bias, dev)
            xp = _to_dev(src.x, dev)
            mp = measure(lay, xp, src.cfg, steps, args.warmup, world, dev, gpu_index, abi, torch)
            gp, gp_clk = time_graph(lay, xp, steps, args.warmup, world, dev, torch, gpu_index)
            g1 = None
            if not args.simt:
                import copy
                l1 = copy.copy(lay)
                l1.flags = lay.flags | abi.MOE_FLAG_NO_OVERLAP
                g1, _ = time_graph(l1, xp, steps, args.warmup, world, dev, torch, None)
            f16 = nvfp4_f16 or (src.cfg.w_dtype == "nvfp4" and nvfp4_on_f16_path(src.cfg, lay.flags))
            rp, lfp = roofline(mp["alg"], mp["stage_ms"]["expert_ffn"], gp, name, src.cfg.w_dtype, args.simt,
                               act_terms, f16, traffic_key(name, lay.flags))
            out = {"workload": WORKLOAD_TEXT[name], "value": job_value(world, src.cfg.T, gp), "unit": "tokens/s",
                   "ms_per_step": gp, "steps": steps, "roofline": rp, "layer_roofline_frac": lfp,
                   "active_experts": mp["alg"]["active"],
                   "stream_launch": {"ms_per_step": mp["ms_step"], "stages_ms": mp["stage_ms"],
                                     "value": job_value(world, src.cfg.T, mp["ms_step"])},
                   "gpu_launches": int(mp["launches"]), "clocks": gp_clk,
                   "one_stream_ms_per_step": g1}
            if flag_note:
                out.update(flag_note)
            return out

        psteps = max(3, args.steps // 2)
        points["prefill"] = point(layer, "prefill", psteps)
        # the same point with the opt-in 8-bit activations (a different
        # numerical contract: see the flag's description in the header)
        if not args.simt and not args.act_e4m3 and cfg.w_dtype == "e4m3":
            import copy
            la = copy.copy(layer)
            la.flags = layer.flags | abi.MOE_FLAG_ACT_E4M3
            la._ws = None
            points["prefill"]["act_e4m3"] = point(la, "prefill", psteps, 1, {
                "flag": "MOE_FLAG_ACT_E4M3",
                "numerics": "one E4M3 term per activation row: parity against the oracle's restatement of that "
                            "rounding; about 5e-2 relative L2 from exact bf16 activations"})
            del la
        points["skew"] = point(layer, "skew", psteps)
        if not args.no_100b:
            layer = None                      # the FP8 weights are no longer needed
            torch.cuda.empty_cache()
            inp100 = moe_synth.make_inputs("100b_decode")
            l100 = MoELayer(inp100, device=dev, flags=flags & ~abi.MOE_FLAG_ACT_E4M3)
            points["100b_decode"] = point(l100, "100b_decode", args.steps)
            points["100b_prefill"] = point(l100, "100b_prefill", psteps)
            if not args.simt:
                import copy
                # the same points on the f16-rebuild path (exact, slower), and
                # the prefill with one NVFP4 term per activation (W4A4, lossy)
                lf = copy.copy(l100)
                lf.flags = l100.flags | abi.MOE_FLAG_NVFP4_F16
                lf._ws = None
                points["100b_decode"]["nvfp4_f16"] = point(lf, "100b_decode", args.steps, None, {
                    "flag": "MOE_FLAG_NVFP4_F16",
                    "numerics": "weights rebuilt exactly in f16, row-scaled f16 activations"}, True)
                lw = copy.copy(l100)
                lw.flags = l100.flags | abi.MOE_FLAG_ACT_NVFP4
                lw._ws = None
                points["100b_prefill"]["act_nvfp4"] = point(lw, "100b_prefill", psteps, 1, {
                    "flag": "MOE_FLAG_ACT_NVFP4",
                    "numerics": "one NVFP4 term per activation row (W4A4): parity against the oracle's restatement "
                                "of that rounding; about 0.1 relative L2 from exact bf16 activations"})
                del lf, lw
            del l100, inp100
            torch.cuda.empty_cache()

    # the fused QK-norm + RoPE step of the same model's attention block
    if args.workload == "decode" and not args.no_prefill:
        points["qk_norm_rope"] = qk_rope_point(args, world, dev, gpu_index, abi, torch)

    if rank != 0:
        return
    value = job_value(world, T, graph_ms)
    roof, layer_frac = roofline(m["alg"], m["stage_ms"]["expert_ffn"], graph_ms, args.workload, cfg.w_dtype,
                                args.simt, 1 if args.act_e4m3 else None,
                                cfg.w_dtype == "nvfp4" and nvfp4_on_f16_path(cfg, flags),
                                traffic_key(args.workload, flags))
    cpu = None
    if not args.no_cpu_baseline and world == 1:   # the oracle baseline: rank 0 of a single-GPU run only
        v, n, el = time_oracle(inp, args.cpu_budget)
        cpu = {"value": v, "unit": "tokens/s", "cores": cores(), "kind": "oracle",
               "sample": f"{n} of the {T} tokens of this workload through the fp64 CPU oracle ({el:.1f} s)",
               "single_thread": {name: oracle_one_thread(name, args.cpu_budget / 3) for name in ("tiny", "decode")}}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": graph_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32" if args.simt else (
            ("f16 MMA with fp32 accumulate (NVFP4 weights rebuilt exactly in f16, row-scaled f16 activations, bf16 H)"
             if nvfp4_on_f16_path(cfg, flags) else
             "e2m1 block-scaled MMA with fp32 accumulate (NVFP4 weights; four NVFP4 terms per activation row, bf16 H)")
            if cfg.w_dtype == "nvfp4" else
            "e4m3 MMA with fp32 accumulate (one-term E4M3 activations: MOE_FLAG_ACT_E4M3, lossy)" if args.act_e4m3 else
            "e4m3 MMA with fp32 accumulate (two-term E4M3 activations, bf16 H)"),
        "data": "synthetic (seeded N(0,1) bf16 activations, N(0,1/d) weights quantised to the stored format)",
        "config": {"workload": WORKLOAD_TEXT[args.workload], "T": T, "d_model": d, "n_experts": cfg.E,
                   "top_k": cfg.k, "d_ff": cfg.f, "d_ff_shared": cfg.fs, "weights": cfg.w_dtype,
                   "ffn_path": "simt" if args.simt else "default",
                   "activations": ("one E4M3 term per row (lossy)" if args.act_e4m3 else
                                   "exact (bf16, or two E4M3 terms per row on the FP8 tensor cores)"),
                   "expert_out": "bf16" if args.bf16_expert_out else "fp32",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (no flush needed): the expert stage moves %.2f GB per pass, "
                         "the expert weights alone over 1.5 GB" % (m["alg"]["ffn_bytes"] / 1e9)},
        "timing": "each step replays the layer (moe_layer_forward: the shared expert on a second stream beside "
                  "the routing) captured as one CUDA graph; one_stream_ms_per_step replays it with "
                  "MOE_FLAG_NO_OVERLAP (everything on one stream); stream_launch times the same step as the four "
                  "ABI calls launched one by one, with CUDA events between the stages; clocks are sampled while "
                  "the layer runs (the timed steps plus ~0.7 s of untimed passes around them)",
        "stream_launch": {"ms_per_step": m["ms_step"], "value": job_value(world, T, m["ms_step"]),
                          "stages_ms": m["stage_ms"], "clocks": m["clocks"]},
        "roofline": roof,
        "layer_roofline_frac": layer_frac,
        "one_stream_ms_per_step": one_stream_ms,
        "active_experts": m["alg"]["active"],
        "clocks": graph_clk,
        "e2e": {"value": job_value(world, T, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": x.numel() * x.element_size(), "d2h_bytes_per_step": T * d * 4},
        "gpu_launches": int(m["launches"]),
        "cpu_baseline": cpu,
        **points,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOAD_TEXT), default="decode")
    ap.add_argument("--simt", action="store_true", help="force the CUDA-core expert kernels")
    ap.add_argument("--bf16-expert-out", action="store_true",
                    help="store the expert outputs in bf16 (MOE_FLAG_BF16_EXPERT_OUT)")
    ap.add_argument("--act-e4m3", action="store_true",
                    help="8-bit activations (MOE_FLAG_ACT_E4M3: one E4M3 term per row, lossy; FP8 weights only)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the further points of the decode run (prefill, skew, 100B decode / prefill)")
    ap.add_argument("--no-100b", action="store_true", help="skip the 100B-style NVFP4 points of the decode run")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--oracle-sample", choices=sorted(WORKLOAD_TEXT), help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.oracle_sample:   # child process of oracle_one_thread
        oracle_sample_main(args.oracle_sample, args.cpu_budget)
        return
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
