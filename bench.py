#!/usr/bin/env python
"""Benchmark of the routed-expert MoE layer forward on GB300 (libmoe.so, C ABI).

One step = one moe_forward over one batch of synthetic tokens: routing,
dispatch quantisation, L1 GEMM (+SwiGLU, requant), L2 GEMM, [shared expert],
combine [+RMSNorm]. Inputs are resident in HBM when the timed region starts;
the L2 cache is flushed before every timed step (a 256 MB write, then a 256 MB read
so that no dirty line of the flush is written back inside the step), outside the
step's own events. Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Multi-GPU (torchrun): every rank runs its own batch of the workload (tokens
are independent), no collective on the data path; value = all ranks' tokens /
the slowest rank's time ("weak" scaling).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthetic as S  # noqa: E402

METRIC = "MoE layer tokens/s"
# The metric is quoted on the largest single-GPU workload: T=8192 H=7168 I=2048 E=256 k=8,
# MXFP8 with Zipf-skewed routing (the prefill shape); --workload selects the others.
DEFAULT_WORKLOAD = "mxfp8_prefill_zipf"
FLUSH_BYTES = 256 << 20
PEAK_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# dense tensor throughput relative to bf16 (nominal 2.25 / 4.5 / 13.5 PFLOP/s)
TENSOR_RATIO = {"bf16": 1.0, "mxfp8": 2.0, "nvfp4": 6.0, "mxfp4": 6.0}
# nominal dense tensor peaks of one GB300 (TFLOP/s), for context beside the measured-peak fraction
NOMINAL_TENSOR_TFLOPS = {"bf16": 2250.0, "mxfp8": 4500.0, "nvfp4": 13500.0, "mxfp4": 13500.0}
ELEM_BYTES = {"bf16": 2.0, "mxfp8": 1.0, "nvfp4": 0.5, "mxfp4": 0.5}
SF_PER_ELEM = {"bf16": 0.0, "mxfp8": 1.0 / 32, "nvfp4": 1.0 / 16, "mxfp4": 1.0 / 32}
# DRAM bytes per launch of the dominant kernel, from ncu captures, keyed by workload and
# kernel; each entry records a hash of the kernel's sources at capture time and is dropped
# when the built sources differ (the capture no longer describes the kernel).
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = {
    "mlp": ["csrc/gemm_fused.cu", "csrc/gemm_epilogue.cuh", "csrc/common.cuh", "csrc/kernels.h"],
}
# tokens of one reference-arm step, and of the first (sizing) call of cpu_baseline
CPU_SAMPLE_TOKENS = {"bf16_toy": 64, "mxfp8_small": 24, "nvfp4_decode": 3, "mxfp8_prefill_zipf": 12,
                     "nvfp4_shared_norm": 6, "mxfp4_small": 24}


def kernel_source_hash(kernel: str) -> str | None:
    """sha256 (first 16 hex digits) over the sources that make up a kernel, in a fixed order."""
    import hashlib
    files = KERNEL_SOURCES.get(kernel)
    if not files:
        return None
    h = hashlib.sha256()
    pkg_dir = os.path.join(ROOT, "serving_topk_permute_gb300")
    for rel in files:
        with open(os.path.join(pkg_dir, rel), "rb") as f:
            h.update(rel.encode() + b"\0" + f.read() + b"\0")
    return h.hexdigest()[:16]


def measured_traffic(workload: str, kernel: str):
    """(DRAM bytes per launch, description) of the kernel on this workload from the traffic
    file, or (None, reason) when there is no capture of the current sources."""
    if not os.path.exists(TRAFFIC_FILE):
        return None, "no capture"
    with open(TRAFFIC_FILE) as f:
        entries = json.load(f).get("entries", [])
    want = kernel_source_hash(kernel)
    for e in entries:
        if e.get("workload") == workload and e.get("kernel") == kernel:
            if e.get("source_sha") != want:
                return None, f"capture of other sources ({e.get('source_sha')} != {want}): dropped"
            return float(e["dram_bytes_per_launch"]), f"profiles/traffic.json: {e.get('how', '')}".strip()
    return None, "no capture of this workload"


# ----------------------------------------------------------------------------- distributed plumbing

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def reduce_max(value: float) -> float:
    """Max over ranks (identity when torch.distributed is not initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def rank_seed(rank: int) -> int:
    """Each rank draws its own tokens (weak scaling: independent batches)."""
    return rank


# ----------------------------------------------------------------------------- work accounting

def algorithmic_work(shape: S.MoeShape, ids: np.ndarray) -> dict:
    """Bytes and FLOPs the method itself needs per step and per kernel: weights of the
    touched experts read once (codes + block scales), the token rows read once and the
    layer output written once. BLOCK_M padding rows, the k permuted copies of the
    dispatched rows, the L2-input round trip and the per-row L2 output are staging
    traffic of this implementation: counted apart, in `staging_bytes`."""
    eb, sf = ELEM_BYTES[shape.fmt], SF_PER_ELEM[shape.fmt]
    H, I, T, k = shape.H, shape.I, shape.T, shape.k
    routed = ids[ids >= 0]
    R = routed.size
    touched = len(np.unique(routed))
    w13 = touched * 2 * I * H * (eb + sf)
    w2 = touched * H * I * (eb + sf)
    gs = 8 * touched if shape.fmt == "nvfp4" else 0
    x_once = T * H * (eb + sf)          # the quantised token rows, once per token
    out_once = T * H * 2                # the layer output (bf16), once per token
    staging = {
        "dispatched_rows": R * H * (eb + sf),    # written by dispatch, read by L1 (k copies per token)
        "l2_input": 2 * R * I * (eb + sf),        # written by L1, read by L2
        "per_row_output": 2 * R * H * 2,          # written by L2, read by combine (bf16)
    }
    per_kernel = {
        "l1": {"bytes": w13 + x_once, "flops": 2.0 * R * 2 * I * H, "fmt": shape.fmt},
        "l2": {"bytes": w2 + gs + out_once, "flops": 2.0 * R * H * I, "fmt": shape.fmt},
        "dispatch": {"bytes": T * H * 2 + x_once, "flops": 0.0, "fmt": shape.fmt},
        "combine": {"bytes": 2 * out_once, "flops": 0.0, "fmt": shape.fmt},
        "route": {"bytes": R * 4 * 3, "flops": 0.0, "fmt": shape.fmt},
    }
    flops = 2.0 * R * 3 * I * H
    nbytes = w13 + w2 + gs + T * H * 2 + out_once
    if shape.shared_I:
        Is, se, ss = shape.shared_I, ELEM_BYTES[shape.shared_fmt], SF_PER_ELEM[shape.shared_fmt]
        sw = 3 * Is * H * (se + ss)
        flops += 2.0 * T * 3 * Is * H
        nbytes += sw
        per_kernel["shared_l1"] = {"bytes": 2 * Is * H * (se + ss) + T * H * (se + ss),
                                   "flops": 2.0 * T * 2 * Is * H, "fmt": shape.shared_fmt}
        per_kernel["shared_l2"] = {"bytes": Is * H * (se + ss) + out_once,
                                   "flops": 2.0 * T * Is * H, "fmt": shape.shared_fmt}
        staging["shared_l2_input"] = 2 * T * Is * (se + ss)
        staging["shared_output"] = 2 * T * H * 2
    return {"flops": flops, "bytes": nbytes, "touched_experts": touched, "per_kernel": per_kernel,
            "staging_bytes": staging}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAK_FALLBACK), "fallback"


def roofline(kernel: str, work: dict, avg_ms: float, peaks: dict, source: str, sustained: bool) -> dict:
    w = work["per_kernel"][kernel]
    hbm = float(peaks.get("hbm_gbs", PEAK_FALLBACK["hbm_gbs"]))
    bf16 = float(peaks.get("bf16_tflops_sustained" if sustained else "bf16_tflops",
                           peaks.get("bf16_tflops", PEAK_FALLBACK["bf16_tflops"])))
    tensor = bf16 * TENSOR_RATIO[w["fmt"]]
    t_mem = w["bytes"] / (hbm * 1e9)
    t_tc = w["flops"] / (tensor * 1e12) if w["flops"] else 0.0
    sec = avg_ms / 1e3
    if t_mem >= t_tc:
        achieved = w["bytes"] / sec / 1e9
        return {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "traffic": None, "kernel": kernel,
                "peak_source": f"{source} hbm_gbs", "algorithmic_bytes": int(w["bytes"]),
                "kernel_ms_avg": round(avg_ms, 5)}
    achieved = w["flops"] / sec / 1e12
    nominal = NOMINAL_TENSOR_TFLOPS[w["fmt"]]
    return {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(tensor, 1), "unit": "TFLOP/s",
            "frac": round(achieved / tensor, 4), "traffic": None, "kernel": kernel,
            "peak_source": f"{source} {'bf16_tflops_sustained' if sustained else 'bf16_tflops'} x "
                           f"{TENSOR_RATIO[w['fmt']]:g} ({w['fmt']} nominal ratio)",
            "algorithmic_flops": w["flops"], "algorithmic_bytes": int(w["bytes"]),
            "kernel_ms_avg": round(avg_ms, 5),
            "frac_of_nominal_dense": round(achieved / nominal, 4), "nominal_dense_tflops": nominal}


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- CPU oracle (baseline / reference arm)

class OracleSample:
    """The CPU oracle on the first n tokens of a workload, with recipe-B weights of the experts those
    tokens touch (generated once per sample size, outside the timed call)."""

    def __init__(self, shape: S.MoeShape, seed: int = 0):
        self.shape, self.seed = shape, seed
        self.x = S.hidden_states(shape, seed)
        self.ids, self.w = S.router(shape, seed)
        self.layer, self.n_built = None, 0

    def _build(self, n: int):
        from oracle import moe as OM
        shape, seed = self.shape, self.seed
        touched = sorted(set(int(e) for e in self.ids[:n].reshape(-1)))
        ck = S.routed_code_checkpoint(shape, seed, experts=touched)
        layer = OM.Layer(shape.E, shape.k, OM.ExpertWeights(ck.fmt, ck.w13, ck.w2, ck.w13_sf, ck.w2_sf,
                                                             ck.w13_gs, ck.w2_gs))
        if shape.fmt == "nvfp4":
            layer.a2 = OM.l2_activation_scale(ck.w2_input_scale)
        if shape.shared_I:
            sc = S.shared_code_checkpoint(shape, seed)
            layer.shared = OM.ExpertWeights(sc.fmt, sc.w13, sc.w2, sc.w13_sf, sc.w2_sf)
        if shape.post_norm:
            layer.norm_gamma = S.norm_gamma(shape, seed)
            layer.norm_eps = shape.norm_eps
        self.layer, self.n_built = layer, n

    def time(self, n: int) -> float:
        """Seconds of one oracle forward over tokens [0, n)."""
        from oracle import moe as OM
        n = max(1, min(n, self.shape.T))
        if n > self.n_built:
            self._build(n)
        t0 = time.perf_counter()
        OM.forward(self.layer, self.x, self.ids, self.w, tokens=list(range(n)))
        return time.perf_counter() - t0


def oracle_baseline(shape: S.MoeShape, target_s: float = 12.0):
    """cpu_baseline: a first timed call on CPU_SAMPLE_TOKENS tokens sizes a second one to about target_s
    seconds of host work. When even the whole batch takes less, the whole batch is run repeatedly until
    target_s has passed. Returns (seconds, tokens, cores, description)."""
    smp = OracleSample(shape)
    n = min(CPU_SAMPLE_TOKENS[shape.name.split("+")[0]], shape.T)
    dt = smp.time(n)
    while dt < 0.8 * target_s and n < shape.T:   # the oracle's time grows slower than its token count
        n = min(shape.T, max(n + 1, int(n * target_s / max(dt, 1e-3))))
        dt = smp.time(n)
    if dt >= target_s or n < shape.T:
        return dt, n, blas_threads(), f"first {n} tokens of {shape.name}"
    total, reps = dt, 1
    while total < target_s:
        total += smp.time(shape.T)
        reps += 1
    return total, reps * shape.T, blas_threads(), f"the whole batch of {shape.name} ({shape.T} tokens) x {reps}"


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count() or 1


REFERENCE_BUDGET_S = 150.0   # host seconds the reference arm's timed steps may take in all


def run_reference(args, shape: S.MoeShape):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    n_tok = min(CPU_SAMPLE_TOKENS[shape.name.split("+")[0]], shape.T)
    smp = OracleSample(shape)
    for _ in range(args.warmup):
        smp.time(1)
    # A step's sample: the first n_tok tokens, halved (down to one token) until the K timed steps
    # fit the budget, so that the run ends within a few minutes whatever K is.
    while n_tok > 1 and smp.time(n_tok) * args.steps > REFERENCE_BUDGET_S:
        n_tok //= 2
    total_s, total_tok, cores = 0.0, 0, blas_threads()
    for i in range(args.steps):
        total_s += smp.time(n_tok)
        total_tok += n_tok
    value = total_tok / total_s
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total_s / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(shape, world),
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {n_tok} tokens of {shape.name} per step (NumPy fp64 oracle)"},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def workload_config(shape: S.MoeShape, world: int) -> dict:
    return {"workload": shape.name, "T": shape.T, "H": shape.H, "I": shape.I, "E": shape.E, "top_k": shape.k,
            "format": shape.fmt, "shared_I": shape.shared_I, "shared_format": shape.shared_fmt if shape.shared_I
            else None, "post_norm": shape.post_norm, "global_batch": shape.T * world,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": "flushed before every timed step (256 MB write, then 256 MB read)"}


# ----------------------------------------------------------------------------- GPU arm

def run_ours(args, shape: S.MoeShape):
    import torch
    import torch.distributed as dist

    import serving_topk_permute_gb300 as pkg

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    seed = rank_seed(rank)

    # inputs (host, seeded) and weights (device, seeded)
    x = S.hidden_states(shape, seed)
    ids, w = S.router(shape, seed)
    T = shape.T
    plan = pkg.Plan(pkg.LayerConfig(shape.E, shape.H, shape.I, shape.k, T, shape.fmt, shared_inter=shape.shared_I,
                                    shared_fmt=shape.shared_fmt, post_norm=shape.post_norm,
                                    norm_eps=shape.norm_eps, tile=args.tile, cta=args.cta, serial=args.serial,
                                    split_gemm=args.split_gemm))
    ck = S.torch_code_checkpoint(shape, seed, dev)
    kw = plan.transform_weights({k: v for k, v in ck.items() if k != "w2_input_scale"})
    ks = plan.transform_shared_weights(S.torch_code_checkpoint(shape, seed, dev, shared=True)) \
        if shape.shared_I else None
    # NVFP4: one L2 input scale for all experts, the max of the per-expert input scales
    a2 = ck["w2_input_scale"].max().reshape(1).to(torch.float32) if shape.fmt == "nvfp4" else None
    del ck
    gamma = torch.from_numpy(S.norm_gamma(shape, seed)).to(dev) if shape.post_norm else None
    hidden = torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
    tid = torch.from_numpy(ids).to(dev)
    tw = torch.from_numpy(w).to(dev)
    out = torch.empty_like(hidden)
    ws = plan.alloc_workspace(T, dev)
    flush_w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush(i: int):
        """Evict the L2: overwrite 256 MB, then read another 256 MB so that the written lines are
        cleaned (written back) here rather than inside the next step."""
        flush_w.fill_(i & 0xFF)
        if not args.flush_write_only:
            torch.amax(flush_r)
    torch.cuda.synchronize()

    def step():
        plan.forward(hidden, tid, tw, kw, l2_act_scale=a2, shared=ks, norm_gamma=gamma, out=out, workspace=ws)

    host_inputs = [x, ids, w]
    if args.batched:
        # the same routed rows on the batched (masked) layout: expert e's slots, in slot order, in its
        # own slab of M rows (M = the largest count rounded up to 128); no combine
        if shape.shared_I or shape.post_norm:
            raise SystemExit("--batched: the batched layout has no shared expert and no norm")
        flat = ids.reshape(-1)
        counts = np.bincount(flat[flat >= 0], minlength=shape.E).astype(np.int32)
        M = max(128, -(-int(counts.max()) // 128) * 128)
        xb = np.zeros((shape.E, M, shape.H), np.uint16)
        fill = np.zeros(shape.E, np.int64)
        for slot in range(flat.size):
            e = int(flat[slot])
            if e >= 0:
                xb[e, fill[e]] = x[slot // shape.k]
                fill[e] += 1
        hidden = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
        cnt_d = torch.from_numpy(counts).to(dev)
        out = torch.zeros_like(hidden)
        ws = torch.zeros(plan.batched_workspace_size(M), dtype=torch.uint8, device=dev)
        host_inputs = [xb, counts]

        def step():
            plan.forward_batched(hidden, cnt_d, kw, l2_act_scale=a2, out=out, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = plan.last_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {status}: {pkg.error_string(status)}")

    # ---- device-resident timed region: K replays of a CUDA graph of one forward
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    t_busy = time.perf_counter()
    while time.perf_counter() - t_busy < 1.0:          # keep the GPU loaded while the sampler starts
        for _ in range(20):
            graph.replay()
        torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush(i)
        evs[i][0].record()
        graph.replay()
        evs[i][1].record()
    torch.cuda.synchronize()
    barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    total_ms = reduce_max(sum(step_ms))
    value = world * T * args.steps / (total_ms / 1e3)

    # ---- per-kernel times: the library's events around each launch (same stream), L2 flushed before each
    # step as above. A spin kernel ahead of each forward lets the host queue the whole forward before the
    # GPU reaches it, so no host launch gap falls between an event and its kernel.
    plan.enable_timing(True)
    ktimes = {}
    kernel_timing = "library events around plain launches queued behind a spin kernel"
    for i in range(min(args.steps, 200)):
        flush(i)
        torch.cuda._sleep(1_000_000)
        step()
        for k_, v in plan.kernel_times().items():
            ktimes.setdefault(k_, []).append(v)
    plan.enable_timing(False)

    # ---- end to end: pinned host inputs -> device -> forward -> host output, every step. The step's
    # inputs (hidden, ids, weights; or the batched slabs and counts) sit in one pinned staging buffer and
    # go over in one copy into one device buffer, whose 256-byte-aligned slices the forward reads.
    offs, o = [], 0
    for arr in host_inputs:
        offs.append(o)
        o += -(-arr.nbytes // 256) * 256
    h_stage = torch.empty(o, dtype=torch.uint8).pin_memory()
    for arr, off in zip(host_inputs, offs):
        h_stage[off:off + arr.nbytes].copy_(torch.from_numpy(np.ascontiguousarray(arr).view(np.uint8).reshape(-1)))
    d_stage = torch.empty_like(h_stage, device=dev)
    torch_dt = {np.dtype(np.uint16): torch.bfloat16, np.dtype(np.int32): torch.int32, np.dtype(np.float32): torch.float32}
    e_in = [d_stage[off:off + arr.nbytes].view(torch_dt[arr.dtype]).view(arr.shape) for arr, off in zip(host_inputs, offs)]
    e_out = torch.zeros_like(out)
    h_out = torch.empty(out.shape, dtype=torch.int16).pin_memory()
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush(i)
        e2e_ev[i][0].record()
        d_stage.copy_(h_stage, non_blocking=True)
        if args.batched:
            plan.forward_batched(e_in[0], e_in[1], kw, l2_act_scale=a2, out=e_out, workspace=ws)
        else:
            plan.forward(e_in[0], e_in[1], e_in[2], kw, l2_act_scale=a2, shared=ks, norm_gamma=gamma, out=e_out,
                         workspace=ws)
        h_out.copy_(e_out.view(torch.int16), non_blocking=True)
        e2e_ev[i][1].record()
    torch.cuda.synchronize()
    barrier()
    assert torch.equal(e_out.view(torch.int16), out.view(torch.int16)), "end-to-end output differs from the graph's"
    copy_ms = reduce_max(sum(a.elapsed_time(b) for a, b in e2e_ev))
    copy_value = world * T * args.steps / (copy_ms / 1e3)
    e2e_value, transfer = copy_value, "one pinned-host-to-device copy of the inputs, one device-to-pinned-host copy of the output"
    zc_value = None
    if not args.batched:
        # the same step with no copy engine: the forward reads its inputs from, and writes its output to,
        # the pinned host buffers themselves (routing, dispatch and combine access them over the host link)
        h_in = [h_stage[off:off + arr.nbytes].view(torch_dt[arr.dtype]).view(arr.shape)
                for arr, off in zip(host_inputs, offs)]
        z_out = torch.zeros(out.shape, dtype=out.dtype).pin_memory()
        zc_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        barrier()
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush(i)
            zc_ev[i][0].record()
            plan.forward(h_in[0], h_in[1], h_in[2], kw, l2_act_scale=a2, shared=ks, norm_gamma=gamma, out=z_out,
                         workspace=ws)
            zc_ev[i][1].record()
        torch.cuda.synchronize()
        barrier()
        assert torch.equal(z_out.view(torch.int16), out.view(torch.int16).cpu()), "zero-copy output differs from the graph's"
        zc_ms = reduce_max(sum(a.elapsed_time(b) for a, b in zc_ev))
        zc_value = world * T * args.steps / (zc_ms / 1e3)
        if zc_value > e2e_value:
            e2e_value = zc_value
            transfer = ("no copy engine: the kernels read the inputs from, and write the output to, pinned host "
                        "memory over the host link")
    ov_value = None
    if not args.batched:
        # the serving pattern: step i's inputs go over while step i-1 computes and step i-2's output
        # comes back. Two device input buffers and two output buffers; a copy-in stream, the compute
        # stream and a copy-out stream, chained by events. One timed region from the first input copy to
        # the last output copy, so every step's copies lie inside it. No L2 flush between steps: the
        # weights a step streams are larger than L2 (the workloads' touched weights are 0.16 to 8.6 GB).
        s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        d_in2 = [d_stage, torch.empty_like(d_stage)]
        x_in2 = [[d[off:off + arr.nbytes].view(torch_dt[arr.dtype]).view(arr.shape) for arr, off in zip(host_inputs, offs)]
                 for d in d_in2]
        y_dev2 = [torch.zeros_like(out), torch.zeros_like(out)]
        y_host2 = [torch.empty(out.shape, dtype=torch.int16).pin_memory() for _ in range(2)]
        ev_in = [torch.cuda.Event() for _ in range(args.steps)]
        ev_comp = [torch.cuda.Event() for _ in range(args.steps)]
        ev_out = [torch.cuda.Event() for _ in range(args.steps)]
        ov_start, ov_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        ov_start.record(s_in)
        for i in range(args.steps):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_comp[i - 2])      # forward i-2 has read this input buffer
                d_in2[b].copy_(h_stage, non_blocking=True)
                ev_in[i].record(s_in)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(ev_in[i])
                if i >= 2:
                    s_comp.wait_event(ev_out[i - 2])     # output i-2 has left this output buffer
                plan.forward(x_in2[b][0], x_in2[b][1], x_in2[b][2], kw, l2_act_scale=a2, shared=ks, norm_gamma=gamma,
                             out=y_dev2[b], workspace=ws, stream=s_comp)
                ev_comp[i].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[i])
                y_host2[b].copy_(y_dev2[b].view(torch.int16), non_blocking=True)
                ev_out[i].record(s_out)
        ov_end.record(s_out)
        torch.cuda.synchronize()
        barrier()
        assert torch.equal(y_host2[(args.steps - 1) % 2], out.view(torch.int16).cpu()), \
            "overlapped end-to-end output differs from the graph's"
        ov_ms = reduce_max(ov_start.elapsed_time(ov_end))
        ov_value = world * T * args.steps / (ov_ms / 1e3)
        if ov_value > e2e_value:
            e2e_value = ov_value
            transfer = ("copy engine, overlapped: each step's input copy and the previous step's output copy run "
                        "beside the compute of the step between them (two buffers each, three streams); one timed "
                        "region over all steps, no L2 flush (the weights streamed per step exceed L2)")
    h2d = sum(arr.nbytes for arr in host_inputs)
    d2h = h_out.numel() * 2
    if plan.last_status(ws) != 0:
        raise RuntimeError("device status after timing")

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    work = algorithmic_work(shape, ids)
    avg_k = {k_: statistics.mean(v) for k_, v in ktimes.items() if v and max(v) > 0}
    # one kernel ran both GEMMs of an MLP (the library reports it under the L1 id): it is
    # charged with the work of both
    for a_, b_, m_ in (("l1", "l2", "mlp"), ("shared_l1", "shared_l2", "shared_mlp")):
        if a_ in avg_k and b_ not in avg_k and a_ in work["per_kernel"]:
            avg_k[m_] = avg_k.pop(a_)
            pa, pb = work["per_kernel"][a_], work["per_kernel"][b_]
            work["per_kernel"][m_] = {"bytes": pa["bytes"] + pb["bytes"], "flops": pa["flops"] + pb["flops"],
                                      "fmt": pa["fmt"]}
    dominant = max(avg_k, key=avg_k.get)
    peaks, source = load_peaks()
    # the sustained (power-capped) tensor peak when the power cap acted during the timed steps, else the burst one
    rl = roofline(dominant, work, avg_k[dominant], peaks, source,
                  sustained="sw_power_cap" in (clk.get("reasons") or []))
    rl["traffic"], rl["traffic_source"] = measured_traffic(shape.name + ("+batched" if args.batched else ""), dominant)
    rl["staging_bytes"] = {k_: int(v) for k_, v in work["staging_bytes"].items()}
    rl["kernel_ms"] = {k_: round(v, 4) for k_, v in avg_k.items()}
    sec = sum(step_ms) / 1e3 / args.steps

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        dt, nt, cores, what = oracle_baseline(shape)
        cpu = {"value": round(nt / dt, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{what} (NumPy fp64 oracle, {dt:.1f} s)"}

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(sum(step_ms) / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": shape.fmt if shape.fmt != "bf16" else "bf16",
        "data": "synthetic (seeded activations and routing; checkpoint bytes drawn on the device)",
        "config": {**workload_config(shape, world), "launch": "serial" if args.serial else "programmatic dependent launch",
                   "tile": args.tile or "library", "cta": args.cta, "gemm": "split" if args.split_gemm else "library",
                   **({"layout": f"batched [E, M, H], M = {out.shape[1]} (tokens/s counts the workload's T tokens, "
                                 f"whose k routed rows the slabs hold; no combine)"} if args.batched else {}),
                   **({"l2": "flushed before every timed step (256 MB write only)"} if args.flush_write_only else {})},
        "roofline": rl,
        "layer": {"tflops": round(work["flops"] / sec / 1e12, 2), "hbm_gbs": round(work["bytes"] / sec / 1e9, 1),
                  "algorithmic_flops": work["flops"], "algorithmic_bytes": int(work["bytes"]),
                  "touched_experts": work["touched_experts"]},
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "transfer": transfer,
                "copy_engine_value": round(copy_value, 1),
                "zero_copy_value": round(zc_value, 1) if zc_value is not None else None,
                "overlapped_value": round(ov_value, 1) if ov_value is not None else None},
        "gpu_launches": len(avg_k) * args.steps,   # this library's kernels per forward (those the per-kernel timing saw run)
        "timing": "value: CUDA-graph replays of one moe_forward, events per step; e2e: C-ABI calls with host "
                  "I/O (copy engine and zero copy: events per step; overlapped: one region over all steps); "
                  "per-kernel: " + kernel_timing,
        "clocks": clk,
        "wall_s": round(wall, 3),
    }
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 500; 10 for --impl reference, whose steps take seconds)")
    ap.add_argument("--warmup", type=int, default=None, help="warm-up steps (default 10; 3 for --impl reference)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=S.WORKLOAD_ORDER, default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tile", type=int, choices=[0, 128, 256], default=0,
                    help="GEMM tile width (0: the library's choice by rows per expert)")
    ap.add_argument("--cta", choices=["auto", "pair", "single"], default="auto",
                    help="GEMMs on CTA pairs: the library's choice, always or never")
    ap.add_argument("--split-gemm", action="store_true", help="L1 and L2 as two kernels instead of one")
    ap.add_argument("--batched", action="store_true",
                    help="the workload's routed rows on the batched [E, M, H] layout (moe_forward_batched)")
    ap.add_argument("--flush-write-only", action="store_true",
                    help="flush the L2 with the 256 MB write alone (its dirty lines are written back inside the step)")
    ap.add_argument("--serial", action="store_true",
                    help="launch each kernel after the previous one finishes (no programmatic dependent launch)")
    ap.add_argument("--tokens", type=int, help="profiling only: override the workload's T")
    ap.add_argument("--experts", type=int, help="profiling only: override the workload's E")
    args = ap.parse_args(argv)
    ref = args.impl == "reference"
    if args.steps is None:
        args.steps = 10 if ref else 500
    if args.warmup is None:
        args.warmup = 3 if ref else 10
    shape = S.WORKLOADS[args.workload]
    over = {k: v for k, v in (("T", args.tokens), ("E", args.experts)) if v}
    if over:
        shape = S.shrink(shape, name=shape.name + "+" + ",".join(f"{k}={v}" for k, v in over.items()), **over)
    if args.impl == "reference":
        return run_reference(args, shape)
    return run_ours(args, shape)


if __name__ == "__main__":
    sys.exit(main())
