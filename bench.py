#!/usr/bin/env python3
"""Throughput of the GLM MoE feed-forward sublayer forward pass on B300.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload glm5_prefill] [--no-decode] [--no-dense] [--no-pack] [--no-qlatent]
                  [--only-dense]
                  [--no-cpu-baseline]

One step is one forward pass of the whole sublayer (RMSNorm, sigmoid router
and top-k, permutation, routed SwiGLU experts, shared expert, combine and
residual) over one batch of synthetic tokens already resident in HBM,
launched as the replay of a CUDA graph that captured one moe_forward call.
Per-stage times come from a second, directly launched pass of the same steps.  With
N > 1 (launched by torch.distributed.run) every rank holds a full replica of
the weights and runs its own batch: no collective is on the data path, so
scaling is weak and the value is the tokens of all ranks per second.

On the GLM-5 prefill workload the line also carries the GLM-5-shaped decode
step (``decode``), the dense feed-forward block of the first decoder
layers (``dense``: moe_dense_forward at T = 8192 and T = 64), the query
compression of the sparse latent attention (``q_latent``: moe_q_latent at
T = 8192 and T = 64) and the packing of the experts' HF weights into the
grouped layout (``pack``).

Rank 0 prints one JSON line.  ``--impl reference`` times the CPU oracle (the
plain definition of the sublayer, run on the host cores) on a bounded sample
of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mixture_experts_transformer_sigmoid_b300 import workloads as wl  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
METRIC = "MoE sublayer tokens/s"
SWEEP_T = (1, 8, 16, 32, 128)   # decode token range (GLM-5 decode weights and bias)

# DRAM bytes (read + write) per launch of the grouped GEMMs from an ncu
# capture (dram__bytes_read.sum + dram__bytes_write.sum), per workload and
# stage, with the hash of the GEMM kernel sources it was taken on.  The bench
# reports the figure only while the sources still hash to that value: any
# change to the kernels makes it null until it is captured again.
TRAFFIC_PER_LAUNCH = {
    # glm5_slice (32 experts, 1024 tokens: the GLM-5 prefill's tokens per expert), one launch each
    "glm5_slice": {"gate_up_swiglu": {"bytes": 1.9038e9 + 0.0363e9, "source_hash": "d375e9479c2fa770"},
                   "down_weighted": {"bytes": 0.8784e9 + 0.0972e9, "source_hash": "d375e9479c2fa770"}},
    # the same capture scaled by 8 to the GLM-5 prefill (routed experts and tokens grow 8x; the
    # shared expert's weights do not, so this overstates by at most 7 x its 50 / 25 MB)
    "glm5_prefill": {"gate_up_swiglu": {"bytes": 8 * (1.9038e9 + 0.0363e9), "source_hash": "d375e9479c2fa770"},
                     "down_weighted": {"bytes": 8 * (0.8784e9 + 0.0972e9), "source_hash": "d375e9479c2fa770"}},
}
TRAFFIC_SOURCES = ("k_gemm_pair.cuh", "k_gemm_tc.cuh", "ptx.cuh")


def gemm_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for name in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, "mixture_experts_transformer_sigmoid_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str, stage: str):
    """DRAM bytes per launch from an ncu capture taken on the current kernel
    sources, else None."""
    rec = TRAFFIC_PER_LAUNCH.get(workload, {}).get(stage)
    if rec is None or rec["source_hash"] != gemm_source_hash():
        return None
    return rec["bytes"]


GEMM_KERNEL = "tc_gemm_pair_kernel"


# Every line after the headline prefill is timed after this much idle: the
# power cap lowers the SM clock under the lines that run before it, so without
# it a line's number would depend on which line ran before (a decode loop,
# for one, never runs in the clock state a long prefill leaves behind).
SETTLE_S = 0.5


def settle():
    torch.cuda.synchronize()
    time.sleep(SETTLE_S)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return json.load(open(p)), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------ arithmetic
def gate_up_flops(w, T):
    """The gate|up launch: routed experts and the shared expert (stage gate_up_swiglu)."""
    return 4.0 * T * w.k * w.d * w.I + 4.0 * T * w.d * w.Is


def down_flops(w, T):
    """The down launch: routed experts and the shared expert (stage down_weighted)."""
    return 2.0 * T * w.k * w.I * w.d + 2.0 * T * w.Is * w.d


def total_flops(w, T):
    return 2.0 * T * w.d * w.E + gate_up_flops(w, T) + down_flops(w, T)


def gate_up_algorithmic_bytes(w, T):
    """Bytes the gate|up launch must move at prefill sizes (every expert active):
    the routed and shared weights, xn once, h and hs written (the permuted
    copy xp is the implementation's, not the step's)."""
    return 2 * (w.E * w.d * 2 * w.I + 2 * w.Is * w.d + T * w.d + T * w.k * w.I + T * w.Is)


def down_algorithmic_bytes(w, T):
    """The down launch: routed and shared weights, h and hs read, the fp16
    weighted rows and the fp32 shared output written."""
    return 2 * (w.E * w.I * w.d + w.d * w.Is + T * w.k * w.I + T * w.Is + T * w.k * w.d) + 4 * T * w.d


def weight_bytes(w):
    es = 4 if w.dtype == "fp32" else 2
    return es * (w.E * w.d * 3 * w.I + 3 * w.d * w.Is + w.E * w.d + w.d) + 4 * w.E


def decode_bytes(w, T, n_active):
    """Bytes a decode forward must move: the weights of every expert that
    received a token, the shared expert, the router, x in and out."""
    return (n_active + 1) * 3 * w.d * w.I * 2 + w.E * w.d * 2 + w.E * 4 + 2 * T * w.d * 2


def gate_up_decode_bytes(w, n_active):
    return n_active * w.d * 2 * w.I * 2 + 2 * w.d * w.Is * 2


# ------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.samples = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", gpu_index, "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                self.samples.append({"sm": float(f[1]), "max": float(f[2]), "power": float(f[3]),
                                     "hw": f[5], "hw_thermal": f[6], "sw_thermal": f[7],
                                     "sw_power": f[8]})
            except ValueError:
                continue

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        pw = [s["power"] for s in self.samples]
        thr = min(pw) + 0.5 * (max(pw) - min(pw)) if max(pw) - min(pw) > 50 else -1.0
        load = [s for s in self.samples if s["power"] >= thr] or self.samples
        reasons = set()
        for s in load:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if s[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s["sm"] for s in load),
                "sm_max_mhz": max(s["max"] for s in load), "reasons": sorted(reasons),
                "samples": len(load), "power_w_median": statistics.median(s["power"] for s in load)}


# ------------------------------------------------------------ helpers
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world: int, tokens_per_rank: int, ms_local: float):
    """Whole-job tokens/s of `world` replicas that each process
    tokens_per_rank tokens per step: the slowest rank's step time bounds the
    job.  Returns (that time in ms, tokens/s)."""
    ms_max = max_over_ranks(ms_local, world)
    return ms_max, world * tokens_per_rank / (ms_max / 1e3)


def replica_inputs(w, rank: int, device: str):
    """Rank 0's inputs; other ranks keep the same weights and draw their own batch."""
    inp = wl.make_inputs(w, seed=0, device=device)
    if rank > 0:
        inp["x"] = wl.make_inputs(w, seed=rank, device=device, weights_from=inp)["x"]
    return inp


def gpu_index(local):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local < len(ids):
            return ids[local]
    return str(local)


def oracle_sample(w, host, n_tokens, seed=1):
    """Runs the CPU oracle on n_tokens seeded tokens; returns (seconds, tokens)."""
    from oracle import oracle as orc
    c = orc.cfg_from_workload(w)
    rows = np.sort(np.random.default_rng(seed).choice(w.T, size=min(n_tokens, w.T), replace=False))
    t0 = time.perf_counter()
    orc.forward(c, host, rows=rows)
    return time.perf_counter() - t0, len(rows)


def cpu_baseline(w, host, target_s=15.0):
    """The oracle timed on the host cores on a bounded sample (at least
    target_s seconds of CPU work after a warm-up call), as tokens/s."""
    from oracle import oracle as orc
    oracle_sample(w, host, 4, seed=2)                   # warm-up: thread pool, page-in
    total_t, total_n, chunk, i = 0.0, 0, 32, 0
    while total_t < target_s:
        t, n = oracle_sample(w, host, chunk, seed=3 + i)
        total_t += t
        total_n += n
        i += 1
        if t < 2.0:
            chunk = min(w.T, chunk * 2)
    return {"value": round(total_n / total_t, 3), "unit": "tokens/s", "cores": orc.num_threads(),
            "kind": "oracle",
            "sample": f"{total_n} seeded tokens of the {w.name} workload in {i} batches "
                      f"({total_t:.1f} s, fp64 oracle)"}


# ------------------------------------------------------------ our arm
def run_ours(args, world, rank, local):
    from mixture_experts_transformer_sigmoid_b300 import binding as B
    peaks, peak_src = load_peaks()
    w = wl.WORKLOADS[args.workload]
    inp = replica_inputs(w, rank, "cuda")   # each replica its own batch, the same weights
    torch.cuda.synchronize()
    T = w.T
    layer = B.MoeSublayer(max_tokens=T, hidden=w.d, n_experts=w.E, inter=w.I, shared_inter=w.Is,
                          max_top_k=w.k, dtype=w.dtype, eps=w.eps, device=local)
    out = torch.empty_like(inp["x"])
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(gpu_index(local))
    time.sleep(0.3)

    for _ in range(args.warmup):
        layer.forward(inp["x"], inp, w.k, w.routed_scale, out=out)
    assert layer.sync_status() == B.MOE_OK
    # The step is one moe_forward captured in a CUDA graph and replayed, as a
    # serving loop would launch it (the forward allocates nothing and never
    # synchronises).
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.forward(inp["x"], inp, w.k, w.routed_scale, out=out)
    graph.replay()
    torch.cuda.synchronize()

    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = e0.elapsed_time(e1) / args.steps
    ms_max, value = replica_throughput(world, T, ms)
    assert layer.sync_status() == B.MOE_OK
    del graph
    # Per-stage times (CUDA events on the launching stream) and the kernel count
    # per forward, from the same number of steps launched directly.
    layer.set_profiling(True)
    layer.read_stats()
    for _ in range(args.steps):
        layer.forward(inp["x"], inp, w.k, w.routed_scale, out=out)
    st = layer.read_stats()
    layer.set_profiling(False)
    assert layer.sync_status() == B.MOE_OK

    stage_ms = {k: v / args.steps for k, v in st["stage_ms"].items()}
    gu_ms, dn_ms = stage_ms["gate_up_swiglu"], stage_ms["down_weighted"]
    dominant = "gate_up_swiglu" if gu_ms >= dn_ms else "down_weighted"
    dom_ms = gu_ms if dominant == "gate_up_swiglu" else dn_ms
    dom_flops = gate_up_flops(w, T) if dominant == "gate_up_swiglu" else down_flops(w, T)
    dom_tf = dom_flops / (dom_ms / 1e3) / 1e12
    peak_tf = peaks["bf16_tflops"]
    roofline = {"kernel": f"{GEMM_KERNEL} ({dominant})", "bound": "tensor",
                "achieved": round(dom_tf, 1), "peak": peak_tf, "unit": "TFLOP/s",
                "frac": round(dom_tf / peak_tf, 4),
                "frac_of_sustained": round(dom_tf / peaks["bf16_tflops_sustained"], 4),
                "peak_source": f"{peak_src} bf16 dense (burst)",
                "flops_per_launch": dom_flops, "avg_launch_ms": round(dom_ms, 4),
                "traffic": measured_traffic(w.name, dominant),
                "algorithmic_bytes": (gate_up_algorithmic_bytes if dominant == "gate_up_swiglu"
                                      else down_algorithmic_bytes)(w, T),
                "kernel_source_hash": gemm_source_hash()}
    if roofline["traffic"] is not None:
        roofline["traffic_over_algorithmic"] = round(roofline["traffic"] / roofline["algorithmic_bytes"], 3)
    whole_tf = total_flops(w, T) / (ms / 1e3) / 1e12
    l2 = (f"inputs larger than L2 ({weight_bytes(w) / 1e9:.1f} GB of weights read every step)"
          if weight_bytes(w) > 126e6 else "inputs smaller than L2")
    res = {
        "metric": f"{METRIC} ({w.name})", "value": round(value, 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_max, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, random-init weights)",
        "config": {"workload": w.name, "tokens_per_gpu": T, "global_tokens": world * T,
                   "hidden": w.d, "experts": w.E, "inter": w.I, "shared_inter": w.Is,
                   "top_k": w.k, "routed_scale": w.routed_scale,
                   "parallelism": f"replicas x{world} (no collective)", "l2": l2},
        "tflops_whole_step": round(whole_tf, 1),
        "tensor_frac_whole_step": round(whole_tf / peak_tf, 4),
        "roofline": roofline,
        "stage_ms": {k: round(v, 4) for k, v in stage_ms.items()},
        "gpu_launches": st["launches"],   # kernels of the timed steps (graph replays launch the same)
        "launch": "CUDA graph replay of one moe_forward per step",
    }

    # ---- decode: GLM-5 shapes, T = 64, skewed routing, L2 flushed per step
    if args.decode and w.name == "glm5_prefill":
        res["decode"] = run_decode(args, inp, local, peaks, peak_src, world)

    # ---- the dense feed-forward block of the first decoder layers (moe_dense_forward)
    if args.dense and w.name == "glm5_prefill":
        res["dense"] = run_dense(args, local, peaks, peak_src, world)

    # ---- the MLA query compression on the GLM-5 shapes (moe_q_latent)
    if args.qlatent and w.name == "glm5_prefill":
        res["q_latent"] = run_qlatent(args, local, peaks, peak_src, world)

    # ---- HF -> grouped layout packing of the GLM-5 expert weights (moe_pack_experts)
    if args.pack and w.name == "glm5_prefill":
        res["pack"] = run_pack(args, inp, peaks, peak_src)

    # ---- end to end: host buffers through the public host-I/O calls.  Every
    # step copies its batch in from pinned host memory and its result back.
    # moe_forward_host_async pipelines the copies against the neighbouring
    # steps' forwards (a stream of batches); moe_forward_host is the blocking
    # call (copy in, forward, copy out, wait), reported beside it.
    x_h = [inp["x"].cpu().pin_memory() for _ in range(2)]
    out_h = [torch.empty_like(x_h[0]).pin_memory() for _ in range(2)]
    ke = max(3, min(args.steps, 20))
    for i in range(2):
        layer.forward_host_async(x_h[i], inp, w.k, w.routed_scale, out_h[i])
    layer.forward_host_wait()
    barrier(world)
    t0 = time.perf_counter()
    for i in range(ke):
        layer.forward_host_async(x_h[i % 2], inp, w.k, w.routed_scale, out_h[i % 2])
    layer.forward_host_wait()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / ke, world)
    for _ in range(2):
        layer.forward_host(x_h[0], inp, w.k, w.routed_scale, out_h[0])
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(ke):
        layer.forward_host(x_h[0], inp, w.k, w.routed_scale, out_h[0])
    e2e_sync_s = max_over_ranks((time.perf_counter() - t0) / ke, world)
    res["e2e"] = {"value": round(world * T / e2e_s, 1), "unit": "tokens/s",
                  "h2d_bytes_per_step": x_h[0].numel() * x_h[0].element_size(),
                  "d2h_bytes_per_step": out_h[0].numel() * out_h[0].element_size(),
                  "ms_per_step": round(e2e_s * 1e3, 3), "steps": ke,
                  "call": "moe_forward_host_async (copies overlap neighbouring steps), then "
                          "moe_forward_host_wait"}
    res["e2e_sync"] = {"value": round(world * T / e2e_sync_s, 1), "unit": "tokens/s",
                       "ms_per_step": round(e2e_sync_s * 1e3, 3), "call": "moe_forward_host"}
    sampler.stop()
    res["clocks"] = sampler.summary()

    # ---- CPU baseline: the oracle on the host cores, rank 0 at N = 1 only
    if args.cpu_baseline and world == 1 and rank == 0:
        host = wl.host_arrays(inp)
        res["cpu_baseline"] = cpu_baseline(w, host)
    layer.close()
    return res


def run_decode_only(args, T, local, peaks, peak_src, world):
    """One decode batch of T tokens on the GLM-5 shapes (skewed routing), the
    forward replayed from a CUDA graph with L2 flushed before every step: the
    case for a launch list of a decode step."""
    from mixture_experts_transformer_sigmoid_b300 import binding as B
    w = wl.WORKLOADS["glm5_decode"]
    inp = wl.make_inputs(w, seed=0, device="cuda", T=T)
    layer = B.MoeSublayer(max_tokens=T, hidden=w.d, n_experts=w.E, inter=w.I, shared_inter=w.Is,
                          max_top_k=w.k, dtype=w.dtype, eps=w.eps, device=local)
    out = torch.empty_like(inp["x"])
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        layer.forward(inp["x"], inp, w.k, w.routed_scale, out=out)
    assert layer.sync_status() == B.MOE_OK
    _, _, counts = layer.routing()
    n_active = int((counts > 0).sum().item())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.forward(inp["x"], inp, w.k, w.routed_scale, out=out)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        graph.replay()
        b.record(stream)
    torch.cuda.synchronize()
    assert layer.sync_status() == B.MOE_OK
    ms = statistics.median([a.elapsed_time(b) for a, b in evs])
    nbytes = decode_bytes(w, T, n_active)
    gbs = nbytes / (ms / 1e3) / 1e9
    del graph
    layer.close()
    return {"metric": f"decode step ms (glm5_decode, {T} tokens)", "value": round(ms, 4), "unit": "ms",
            "higher_is_better": False, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "n_active_experts": n_active, "bytes_per_step": nbytes, "hbm_gbs": round(gbs, 1),
            "hbm_frac": round(gbs / peaks["hbm_gbs"], 4), "dtype": "bf16",
            "data": "synthetic (seeded, random-init weights)",
            "l2": "256 MB buffer written between steps (outside the timed events)",
            "launch": "CUDA graph replay of one moe_forward"}


def run_decode(args, inp3, local, peaks, peak_src, world):
    from mixture_experts_transformer_sigmoid_b300 import binding as B
    w = wl.WORKLOADS["glm5_decode"]
    dinp = wl.make_inputs(w, seed=0, device="cuda", weights_from=inp3)
    layer = B.MoeSublayer(max_tokens=max(SWEEP_T), hidden=w.d, n_experts=w.E, inter=w.I,
                          shared_inter=w.Is, max_top_k=w.k, dtype=w.dtype, eps=w.eps, device=local)
    out = torch.empty_like(dinp["x"])
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(5):
        layer.forward(dinp["x"], dinp, w.k, w.routed_scale, out=out)
    assert layer.sync_status() == B.MOE_OK
    _, _, counts = layer.routing()
    n_active = int((counts > 0).sum().item())
    n_iter = max(50, args.steps * 4)
    # Step time: the forward captured once in a CUDA graph and replayed (a decode
    # step's kernels are short enough that host launch latency would otherwise
    # show up between them); L2 flushed before every step, outside the events.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.forward(dinp["x"], dinp, w.k, w.routed_scale, out=out)
    settle()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n_iter)]
    for a, b in evs:
        flush.zero_()                       # evict the previous step's weights from L2
        a.record(stream)
        graph.replay()
        b.record(stream)
    torch.cuda.synchronize()
    times = [a.elapsed_time(b) for a, b in evs]
    assert layer.sync_status() == B.MOE_OK
    # Stage times (for the kernel roofline): the same steps launched directly with
    # per-stage CUDA events.
    layer.set_profiling(True)
    layer.read_stats()
    for _ in range(n_iter):
        flush.zero_()
        layer.forward(dinp["x"], dinp, w.k, w.routed_scale, out=out)
    torch.cuda.synchronize()
    st = layer.read_stats()
    layer.set_profiling(False)
    del graph
    # The decode token range: the same weights and skewed bias, T from 1 to 128
    sweep = []
    for T in SWEEP_T:
        x = wl.make_inputs(w, seed=T, device="cuda", T=T, weights_from=inp3)["x"]
        o = torch.empty_like(x)
        for _ in range(3):
            layer.forward(x, dinp, w.k, w.routed_scale, out=o)
        _, _, cnt = layer.routing()
        na = int((cnt > 0).sum().item())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            layer.forward(x, dinp, w.k, w.routed_scale, out=o)
        torch.cuda.synchronize()
        ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n_iter)]
        for a, b in ev2:
            flush.zero_()
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        t_ms = statistics.median([a.elapsed_time(b) for a, b in ev2])
        nb = decode_bytes(w, T, na)
        sweep.append({"tokens": T, "n_active_experts": na, "ms_per_step_median": round(t_ms, 4),
                      "hbm_gbs": round(nb / (t_ms / 1e3) / 1e9, 1),
                      "hbm_frac": round(nb / (t_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4)})
        del g
    assert layer.sync_status() == B.MOE_OK
    layer.close()
    ms = statistics.median(times)
    nbytes = decode_bytes(w, w.T, n_active)
    gbs = nbytes / (ms / 1e3) / 1e9
    stage_ms = {k: v / n_iter for k, v in st["stage_ms"].items()}
    gu_ms = stage_ms["gate_up_swiglu"]
    gu_bytes = gate_up_decode_bytes(w, n_active)
    gu_gbs = gu_bytes / (gu_ms / 1e3) / 1e9
    hbm = peaks["hbm_gbs"]
    return {"workload": w.name, "tokens": w.T, "n_active_experts": n_active,
            "ms_per_step_median": round(ms, 4), "ms_per_step_mean": round(statistics.mean(times), 4),
            "tokens_per_s": round(world * w.T / (ms / 1e3), 1),
            "bytes_per_step": nbytes, "hbm_gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm, 4),
            "l2": "256 MB buffer written between steps (outside the timed events)",
            "idle_before_s": SETTLE_S,
            "launch": "CUDA graph replay of one moe_forward",
            "roofline": {"kernel": "tc_gemm_kernel (gate_up_swiglu)", "bound": "hbm",
                         "achieved": round(gu_gbs, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(gu_gbs / hbm, 4), "peak_source": f"{peak_src} HBM copy",
                         "bytes_per_launch": gu_bytes, "avg_launch_ms": round(gu_ms, 4),
                         "traffic": None},
            "stage_ms": {k: round(v, 4) for k, v in stage_ms.items()},
            "token_sweep": sweep}


def run_dense(args, local, peaks, peak_src, world):
    """moe_dense_forward on the GLM-5-sized dense block: prefill (T = 8192,
    against the bf16 peak) and decode (T = 64, L2 flushed, against HBM)."""
    from mixture_experts_transformer_sigmoid_b300 import binding as B
    wp = wl.DENSE_WORKLOADS["glm5_dense_prefill"]
    wd = wl.DENSE_WORKLOADS["glm5_dense_decode"]
    inp = wl.make_dense_inputs(wp, device="cuda")
    dinp = wl.make_dense_inputs(wd, device="cuda", weights_from=inp)
    layer = B.MoeSublayer(max_tokens=wp.T, hidden=wp.d, n_experts=0, inter=0, shared_inter=0,
                          max_top_k=0, dtype=wp.dtype, eps=wp.eps, device=local, dense_inter=wp.I)
    stream = torch.cuda.current_stream()
    res = {}
    # the decode-sized batch first, after the idle of settle(); then the prefill
    for w, x in ((wd, dinp["x"]), (wp, inp["x"])):
        out = torch.empty_like(x)
        for _ in range(args.warmup):
            layer.dense_forward(x, inp, out=out)
        assert layer.sync_status() == B.MOE_OK
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            layer.dense_forward(x, inp, out=out)
        torch.cuda.synchronize()
        wbytes = 3 * w.d * w.I * 2
        if w.T >= 1024:
            # weights (453 MB) and activations exceed L2: no flush between steps
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            settle()
            e0.record(stream)
            for _ in range(args.steps):
                graph.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / args.steps
            flops = 6 * w.T * w.d * w.I
            tf = flops / (ms / 1e3) / 1e12
            res["prefill"] = {
                "workload": w.name, "tokens": w.T, "ms_per_step": round(ms, 4),
                "tokens_per_s": round(world * w.T / (ms / 1e3), 1), "flops_per_step": flops,
                "tflops": round(tf, 1), "tensor_frac": round(tf / peaks["bf16_tflops"], 4),
                "tensor_frac_of_sustained": round(tf / peaks["bf16_tflops_sustained"], 4),
                "peak_source": f"{peak_src} bf16 dense (burst)", "idle_before_s": SETTLE_S,
                "launch": "CUDA graph replay of one moe_dense_forward (3 kernels)"}
        else:
            flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
            n_iter = max(50, args.steps * 4)
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(n_iter)]
            settle()
            for a, b in evs:
                flush.zero_()
                a.record(stream)
                graph.replay()
                b.record(stream)
            torch.cuda.synchronize()
            ms = statistics.median([a.elapsed_time(b) for a, b in evs])
            nbytes = wbytes + 2 * w.T * w.d * 2 + w.d * 2
            gbs = nbytes / (ms / 1e3) / 1e9
            res["decode"] = {
                "workload": w.name, "tokens": w.T, "ms_per_step_median": round(ms, 4),
                "tokens_per_s": round(world * w.T / (ms / 1e3), 1), "bytes_per_step": nbytes,
                "hbm_gbs": round(gbs, 1), "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
                "peak_source": f"{peak_src} HBM copy",
                "l2": "256 MB buffer written between steps (outside the timed events)",
                "idle_before_s": SETTLE_S,
                "launch": "CUDA graph replay of one moe_dense_forward (5 kernels: RMSNorm, both "
                          "projections split over k-ranges, each followed by the fixed-order sum of its "
                          "partials)"}
        assert layer.sync_status() == B.MOE_OK
        del graph
    layer.close()
    return res


def run_qlatent(args, local, peaks, peak_src, world):
    """moe_q_latent (the query compression of the sparse latent attention) on
    the GLM-5 shapes (d 6144, q_lora_rank 2048): prefill (T = 8192, against the
    bf16 peak) and decode (T = 64, L2 flushed, against HBM)."""
    from mixture_experts_transformer_sigmoid_b300 import binding as B
    wp, wd = wl.QLATENT_WORKLOADS["glm5_q_prefill"], wl.QLATENT_WORKLOADS["glm5_q_decode"]
    inp = wl.make_q_inputs(wp, device="cuda")
    dinp = wl.make_q_inputs(wd, device="cuda", weights_from=inp)
    layer = B.MoeSublayer(max_tokens=wp.T, hidden=wp.d, n_experts=0, inter=0, shared_inter=0,
                          max_top_k=0, dtype=wp.dtype, eps=wp.eps, device=local, dense_inter=64)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    res = {}
    for w, x in ((wp, inp["hidden"]), (wd, dinp["hidden"])):
        c = torch.empty((w.T, w.rank), dtype=x.dtype, device="cuda")
        q = torch.empty_like(c)
        for _ in range(args.warmup):
            layer.q_latent(x, inp["w_qa"], inp["q_norm_w"], c_out=c, q_out=q)
        assert layer.sync_status() == B.MOE_OK
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            layer.q_latent(x, inp["w_qa"], inp["q_norm_w"], c_out=c, q_out=q)
        torch.cuda.synchronize()
        n_iter = max(50, args.steps * 4)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n_iter)]
        settle()
        for a, b in evs:
            flush.zero_()                  # the weights (25 MB) would otherwise stay in L2
            a.record(stream)
            graph.replay()
            b.record(stream)
        torch.cuda.synchronize()
        ms = statistics.median([a.elapsed_time(b) for a, b in evs])
        assert layer.sync_status() == B.MOE_OK
        del graph
        flops = 2.0 * w.T * w.d * w.rank
        nbytes = 2 * (w.rank * w.d + w.T * w.d + 2 * w.T * w.rank + w.rank)
        line = {"workload": w.name, "tokens": w.T, "ms_median": round(ms, 4),
                "tokens_per_s": round(world * w.T / (ms / 1e3), 1), "flops": flops, "bytes": nbytes,
                "tflops": round(flops / (ms / 1e3) / 1e12, 1),
                "tensor_frac": round(flops / (ms / 1e3) / 1e12 / peaks["bf16_tflops"], 4),
                "hbm_gbs": round(nbytes / (ms / 1e3) / 1e9, 1),
                "hbm_frac": round(nbytes / (ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
                "peak_source": f"{peak_src} (bf16 burst, HBM copy)",
                "l2": "256 MB buffer written between steps (outside the timed events)",
                "launch": "CUDA graph replay of one moe_q_latent", "idle_before_s": SETTLE_S}
        res["prefill" if w.T >= 1024 else "decode"] = line
    layer.close()
    return res


def run_pack(args, inp, peaks, peak_src):
    """moe_pack_experts on the GLM-5 expert weights: the HF per-expert stacks
    (made from the workload's grouped weights by torch transposes, outside
    the timed region) packed back into the grouped layout; the result must
    equal the workload's weights bit for bit."""
    from mixture_experts_transformer_sigmoid_b300 import binding as B
    gate_up, down = inp["gate_up"], inp["down"]
    E, d, I2 = gate_up.shape
    I = I2 // 2
    G = gate_up[:, :, :I].transpose(1, 2).contiguous()
    U = gate_up[:, :, I:].transpose(1, 2).contiguous()
    Dn = down.transpose(1, 2).contiguous()
    gu = torch.empty_like(gate_up)
    dp = torch.empty_like(down)
    stream = torch.cuda.current_stream()
    for _ in range(2):
        B.pack_experts(G, U, Dn, gate_up=gu, down_projs=dp)
    torch.cuda.synchronize()
    exact = bool(torch.equal(gu, gate_up) and torch.equal(dp, down))
    n = max(3, min(args.steps, 10))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    settle()
    e0.record(stream)
    for _ in range(n):
        B.pack_experts(G, U, Dn, gate_up=gu, down_projs=dp)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    nbytes = 2 * 3 * E * d * I * gate_up.element_size()   # every element read once, written once
    gbs = nbytes / (ms / 1e3) / 1e9
    del G, U, Dn, gu, dp
    torch.cuda.empty_cache()
    return {"experts": E, "hidden": d, "inter": I, "ms": round(ms, 4), "bytes": nbytes,
            "hbm_gbs": round(gbs, 1), "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
            "peak_source": f"{peak_src} HBM copy", "exact": exact, "launches": 3, "idle_before_s": SETTLE_S,
            "call": "moe_pack_experts (HF per-expert stacks -> gate_and_up_projs, down_projs)"}


# ------------------------------------------------------------ reference arm
def run_reference(args, world):
    """The CPU oracle on the host cores, on bounded samples of the workload."""
    from oracle import oracle as orc
    w = wl.WORKLOADS[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = wl.make_inputs(w, seed=0, device=dev)
    host = wl.host_arrays(inp)
    del inp
    t_cal, n_cal = oracle_sample(w, host, 4, seed=10)
    per_tok = t_cal / n_cal
    n_step = int(max(1, min(w.T, args.ref_budget_s / (args.steps + args.warmup) / per_tok)))
    for i in range(args.warmup):
        oracle_sample(w, host, n_step, seed=100 + i)
    times = [oracle_sample(w, host, n_step, seed=1000 + i)[0] for i in range(args.steps)]
    total_t = sum(times)
    value = args.steps * n_step / total_t
    sample = (f"{n_step} seeded tokens of the {w.name} workload per step "
              f"(T={w.T} in the full workload), fp64 oracle")
    return {"impl": "reference", "metric": f"{METRIC} ({w.name})", "value": round(value, 3),
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * total_t / args.steps, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, random-init weights)",
            "config": {"workload": w.name, "tokens_per_step": n_step, "hidden": w.d,
                       "experts": w.E, "inter": w.I, "shared_inter": w.Is, "top_k": w.k,
                       "routed_scale": w.routed_scale},
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s",
                             "cores": orc.num_threads(), "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="glm5_prefill", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--no-decode", dest="decode", action="store_false")
    ap.add_argument("--no-dense", dest="dense", action="store_false")
    ap.add_argument("--no-pack", dest="pack", action="store_false")
    ap.add_argument("--no-qlatent", dest="qlatent", action="store_false")
    ap.add_argument("--only-dense", action="store_true",
                    help="time only the dense feed-forward block (about 1 GB on the device; "
                         "the case for profiling its kernels)")
    ap.add_argument("--only-decode", type=int, default=0, metavar="T",
                    help="time only a decode step of T tokens on the GLM-5 shapes (graph replay, "
                         "L2 flushed; the case for a decode launch list)")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--ref-budget-s", type=float, default=150.0,
                    help="reference arm: seconds of oracle work for the whole run")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, world)), flush=True)
        return
    world, rank, local = dist_setup()
    if args.only_decode > 0:
        peaks, peak_src = load_peaks()
        torch.cuda.set_device(local)
        res = run_decode_only(args, args.only_decode, local, peaks, peak_src, world)
        if rank == 0:
            print(json.dumps(res), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    if args.only_dense:
        peaks, peak_src = load_peaks()
        torch.cuda.set_device(local)
        dense = run_dense(args, local, peaks, peak_src, world)
        if rank == 0:
            pf = dense["prefill"]
            print(json.dumps({"metric": "dense feed-forward block tokens/s (glm5_dense_prefill)",
                              "value": pf["tokens_per_s"], "unit": "tokens/s", "n_gpus": world,
                              "steps": args.steps, "warmup": args.warmup,
                              "ms_per_step": pf["ms_per_step"], "higher_is_better": True,
                              "dtype": "bf16", "data": "synthetic (seeded, random-init weights)",
                              "dense": dense}), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    res = run_ours(args, world, rank, local)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
