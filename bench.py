#!/usr/bin/env python
"""Benchmark of the sparse-MoE block forward on B300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

A step is one whole forward (router, dispatch, expert MLPs, combine, aux) of
one synthetic batch of the named layer configuration, inputs resident in HBM.
The default is the skewed-routing layer (T=16384 H=4096 E=128 K=8 I=1536,
expert loads following Zipf(1.2)), the largest configuration of the workload
set that fits one GPU; the same line carries the large-expert prefill layer
(T=8192) and the decode sweep (T = 1, 4, 16, 64 on the same layer, timed as
CUDA-graph replays, the way a decode server runs) under "extra_configs", each
measured the same way.  The K timed steps are enqueued back to back (no host
wait inside the timed region) and each is timed on the device with CUDA events
on the launch stream; L2 is flushed (256 MB write) between steps, outside the
events.  A second pass of K steps has the library record stage-boundary events
on the same stream, giving the live per-kernel times of the roofline object and
the stage split (those events serialise the boundaries they sit on, so they
stay out of the first pass).  With N > 1 (torchrun) every rank runs an
independent replica on its own batch (weak scaling, no collective on the data
path); value = all ranks' tokens / max-over-ranks time.

Roofline: algorithmic work only -- routed FLOPs, the touched experts' weights,
the router weights and the block's own inputs and outputs (x read once, out,
logits, top-k); the intermediates x_perm, h and Y are implementation overhead
and count for nothing.  Fractions are against the measured burst bf16 peak and
the measured copy bandwidth (MEASURED_PEAKS.json); the fraction against the
sustained bf16 figure (cuBLAS looped for seconds under the power limit) is
reported beside it.

--impl reference times the CPU oracle (the plain fp64 C implementation) on
bounded token samples of the same workload, on the host cores.
"""
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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import moe_inputs as mi  # noqa: E402

METRIC = "MoE-layer tokens/s on 1 B300 and % of roofline (tensor peak or HBM GB/s)"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
# The sources a stage's kernel is built from, per expert path: a recorded DRAM
# traffic figure is reported only while these files are unchanged.
_COMMON = ["moe_common.cuh", "sm100_ptx.cuh"]
STAGE_SOURCES = {
    "router": ["router_tc.cu", "router.cu", "routing.cuh"] + _COMMON,
    "dispatch": ["dispatch.cu", "routing.cuh"] + _COMMON,
    "combine": ["combine.cu"] + _COMMON,
}
PATH_SOURCES = {
    "tcgen05": ["experts_tc.cu"], "tcgen05_pair": ["experts_pair.cu"],
    "tcgen05_wt": ["experts_wt.cu"],
    "tcgen05_decode": ["experts_decode.cu", "experts_wt.cu", "routing.cuh"],
    "streaming": ["experts_stream.cu"], "warp_mma_q4": ["experts_q4_mma.cu", "quant.cu"],
    "tcgen05_q4": ["experts_q4.cu", "quant.cu"],
}


def stage_sources(stage, path):
    if stage in ("gate_up", "down"):
        return PATH_SOURCES.get(path, []) + _COMMON
    return STAGE_SOURCES[stage]


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="skew", choices=sorted(mi.CONFIGS))
    ap.add_argument("--no-extras", action="store_true",
                    help="time the main configuration only (no extra_configs)")
    ap.add_argument("--shape", default=None,
                    help="T,H,E,K,I: a custom layer (norm_topk_prob on, seed 0) instead of --config, "
                         "for small profiling cases")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--quiet-clocks", action="store_true", help="skip nvidia-smi sampling")
    ap.add_argument("--ref-step-seconds", type=float, default=None,
                    help="reference arm: oracle seconds per step (default: ~150 s in total)")
    ap.add_argument("--warmup-seconds", type=float, default=1.0,
                    help="warm-up lasts at least W steps and this long (0 for profiling runs)")
    ap.add_argument("--graph", action="store_true",
                    help="time replays of the forward captured as a CUDA graph (decode serving)")
    ap.add_argument("--weights", default="packed", choices=["packed", "row-major", "q4"],
                    help="expert weights packed once into the tile-major layout before timing "
                         "(moe_pack_experts, a model-load step), read row-major, or quantised "
                         "once to 4 bits in groups of 128 (moe_quantize_experts_q4)")
    ap.add_argument("--expert-path", default="auto",
                    choices=["auto", "streaming", "tcgen05", "tcgen05_wt", "tcgen05_pair",
                             "tcgen05_decode", "warp_mma"],
                    help="expert MLP kernels (auto picks by rows per expert)")
    return ap.parse_args(argv)


def workload(args):
    if args.shape:
        T, H, E, K, I = (int(v) for v in args.shape.split(","))
        return mi.MoEConfig(f"shape_T{T}_H{H}_E{E}_K{K}_I{I}", T, H, E, K, I, True)
    return mi.CONFIGS[args.config]


# ---- distributed ------------------------------------------------------------------

def dist_setup(args):
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


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate_value(tokens_per_rank, world, max_ms):
    """Whole-job tokens/s: every rank processes its own batch of tokens_per_rank
    tokens per step (weak scaling); the slowest rank's step time bounds the job."""
    return tokens_per_rank * world / (max_ms * 1e-3)


def replica_seed(cfg, rank):
    """Each replica draws its own synthetic batch (and weights) from the
    workload's seed offset by its rank."""
    return cfg.seed + rank


def max_over_ranks(v, world, device):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---- measured peaks ---------------------------------------------------------------

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", 0) or 0),
                    source="measured")
    return dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0,
                source="fallback")


# ---- algorithmic work per stage: bytes and flops a launch must move or compute -----

# bytes per expert weight: bf16, or 4-bit codes plus a bf16 scale and bias per 128
WEIGHT_BYTES = {"bf16": 2.0, "q4": 0.5 + 4.0 / 128}


def stage_work(cfg, counts, fused=False, wb=2.0):
    """Algorithmic work of each stage's kernel per launch: FLOPs of the
    contractions it computes and the bytes of the block's own tensors it must
    touch (expert and router weights, x read once, out, logits, top-k).  The
    intermediates x_perm, h and Y are implementation overhead and count for
    nothing, so the stages that only move them (dispatch's gather, combine's
    reads) carry only the block outputs they write.
    fused: the decode kernel runs gate/up, down and the combine in one launch,
    timed as the gate_up stage, so that stage carries all three stages' work.
    wb: bytes per expert weight."""
    T, H, E, K, I = cfg.T, cfg.H, cfg.E, cfg.K, cfg.I
    P = T * K
    touched = int((np.asarray(counts) > 0).sum())
    w = {
        "router": dict(flops=2.0 * T * H * E, bytes=T * H * 2 + E * H * 2 + T * E * 4 + T * K * 8),
        "dispatch": dict(flops=0.0, bytes=T * K * 8 + 4),
        "gate_up": dict(flops=4.0 * P * H * I, bytes=touched * 2 * I * H * wb + T * H * 2),
        "down": dict(flops=2.0 * P * I * H, bytes=touched * H * I * wb),
        "combine": dict(flops=0.0, bytes=T * H * 2),
    }
    if fused:
        w["gate_up"] = {k: w["gate_up"][k] + w["down"][k] + w["combine"][k] for k in ("flops", "bytes")}
    return w, touched


def block_work(cfg, counts, wb=2.0):
    """Whole-block roofline: routed FLOPs and the bytes of the touched experts'
    weights (wb bytes each) plus the block's inputs and outputs (intermediates
    excluded)."""
    T, H, E, K, I = cfg.T, cfg.H, cfg.E, cfg.K, cfg.I
    touched = int((np.asarray(counts) > 0).sum())
    flops = 6.0 * T * K * H * I + 2.0 * T * H * E
    byts = touched * 3 * H * I * wb + E * H * 2 + T * H * 2 * 2 + T * E * 4 + T * K * 8 + 4
    return flops, byts


def roofline_of(work, stage_mean, path_name, pk, cfg, weights="packed"):
    """The roofline object of the dominant stage's kernel: algorithmic work per
    launch over its live mean duration, against the burst tensor peak or the
    copy bandwidth, whichever bound is slower."""
    dom = max(stage_mean, key=stage_mean.get)
    wk = work[dom]
    t_s = stage_mean[dom] * 1e-3
    t_flop = wk["flops"] / (pk["bf16_tflops"] * 1e12)
    t_byte = wk["bytes"] / (pk["hbm_gbs"] * 1e9)
    if t_flop >= t_byte:
        roof = {"bound": "tensor", "achieved": wk["flops"] / t_s / 1e12, "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s"}
        if pk["bf16_tflops_sustained"]:
            roof["frac_sustained"] = roof["achieved"] / pk["bf16_tflops_sustained"]
    else:
        roof = {"bound": "hbm", "achieved": wk["bytes"] / t_s / 1e9, "peak": pk["hbm_gbs"],
                "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = traffic_for(dom, cfg.name, path_name, weights)
    roof["kernel"] = "experts_fused" if (dom == "gate_up" and path_name == "tcgen05_decode") else dom
    roof["kernel_ms"] = stage_mean[dom]
    roof["algorithmic"] = {"flops": wk["flops"], "bytes": wk["bytes"]}
    roof["peak_source"] = pk["source"] + (
        " burst bf16 (frac); sustained bf16 beside it (frac_sustained)" if roof["bound"] == "tensor"
        else " copy bandwidth")
    return roof


def block_roofline_of(cfg, counts, wb, mean_ms, pk):
    bf, bb = block_work(cfg, counts, wb=wb)
    t = mean_ms * 1e-3
    t_tc = bf / (pk["bf16_tflops"] * 1e12)
    t_hbm = bb / (pk["hbm_gbs"] * 1e9)
    t_roof = max(t_tc, t_hbm)
    out = {"flops": bf, "bytes": bb, "t_roof_us": t_roof * 1e6, "t_us": mean_ms * 1e3,
           "bound": "tensor" if t_tc >= t_hbm else "hbm",
           "frac": t_roof / t,
           "tensor_frac": bf / t / (pk["bf16_tflops"] * 1e12),
           "hbm_frac": bb / t / (pk["hbm_gbs"] * 1e9),
           "touched_experts": int((np.asarray(counts) > 0).sum()),
           "peaks": "burst bf16 and copy bandwidth (frac); sustained bf16 (frac_sustained)"}
    if pk["bf16_tflops_sustained"]:
        t_roof_s = max(bf / (pk["bf16_tflops_sustained"] * 1e12), t_hbm)
        out["frac_sustained"] = t_roof_s / t
    return out


def kernel_source_sha(stage, path):
    h = hashlib.sha256()
    for n in stage_sources(stage, path):
        with open(os.path.join(ROOT, "mixture_experts_layer_98_b300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(stage, config, path, weights="packed"):
    """DRAM bytes per launch of the stage's kernel from the committed ncu summary,
    or None when there is none or the kernel's sources changed since."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    d = json.load(open(TRAFFIC_FILE))
    e = d.get("entries", {}).get(f"{config}:{weights}:{path}:{stage}")
    if e is None or e.get("source_sha") != kernel_source_sha(stage, path):
        return None
    return float(e["dram_bytes_per_launch"])


# ---- clocks -------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 10:
                rows.append(parts)
        os.unlink(self.path)
        return rows

    @staticmethod
    def summarize(rows, t0, t1):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        import datetime

        def ts(r):
            try:
                return datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                return 0.0
        inside = [r for r in rows if t0 - 0.1 <= ts(r) <= t1 + 0.1] or rows[-3:]
        sm = [float(r[2]) for r in inside if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in inside if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4)
                          if r[6 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside)}


# ---- CPU oracle baseline ---------------------------------------------------------------

def oracle_sample_rate(cfg, bits, target_s, max_tokens=None):
    """Time the oracle's full forward on the first n tokens of the batch
    (n sized for about target_s seconds).  Returns (tokens/s, n, seconds, threads)."""
    import oracle
    T = bits["x"].shape[0]
    per_tok = None
    for n in (min(4, T), min(32, T)):  # the first call also pays one-time page-in costs
        t = time.perf_counter()
        oracle.moe_forward(bits["x"][:n], bits["W_router"], bits["W_gate"], bits["W_up"],
                           bits["W_down"], cfg.K, cfg.norm)
        per_tok = max((time.perf_counter() - t) / n, 1e-6)
    n = int(max(4, min(T, target_s / per_tok)))
    if max_tokens:
        n = min(n, max_tokens)
    t = time.perf_counter()
    oracle.moe_forward(bits["x"][:n], bits["W_router"], bits["W_gate"], bits["W_up"],
                       bits["W_down"], cfg.K, cfg.norm)
    dt = time.perf_counter() - t
    return n / dt, n, dt, oracle.threads()


# ---- the reference arm: the CPU oracle -------------------------------------------------

def run_reference(args, world, rank):
    if rank != 0:
        return
    cfg = workload(args)
    inp = mi.make_inputs(cfg, "cpu")
    bits = {k: mi.bits(v) for k, v in inp.items()}
    import oracle
    # size one step's token sample so that warmup + steps take about 2-3 minutes
    per_step_s = (args.ref_step_seconds if args.ref_step_seconds
                  else max(0.5, 150.0 / max(1, args.steps + args.warmup)))
    _, n, _, threads = oracle_sample_rate(cfg, bits, per_step_s)
    for _ in range(args.warmup):
        oracle.moe_forward(bits["x"][:n], bits["W_router"], bits["W_gate"], bits["W_up"],
                           bits["W_down"], cfg.K, cfg.norm)
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle.moe_forward(bits["x"][:n], bits["W_router"], bits["W_gate"], bits["W_up"],
                           bits["W_down"], cfg.K, cfg.norm)
        times.append(time.perf_counter() - t)
    mean = sum(times) / len(times)
    value = n / mean
    sample = (f"first {n} of {cfg.T} tokens of {cfg.name} per step (full routing, dispatch, "
              f"experts and combine for those tokens), fp64 C oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_block(cfg, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_block(cfg, world):
    return {"workload": f"{cfg.name}: T={cfg.T} H={cfg.H} E={cfg.E} K={cfg.K} I={cfg.I} "
                        f"norm_topk_prob={str(cfg.norm).lower()}"
                        + (f" zipf={cfg.zipf}" if cfg.zipf else ""),
            "T": cfg.T, "H": cfg.H, "E": cfg.E, "K": cfg.K, "I": cfg.I, "norm_topk_prob": cfg.norm,
            "seed": cfg.seed, "global_batch_tokens": cfg.T * world,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": "flushed between steps (256 MB write, outside the timed events); "
                  "expert weights alone exceed L2"}


# ---- our arm ------------------------------------------------------------------------

# The same line's extra configurations: (name, timed as CUDA-graph replays)
# (config, CUDA-graph replay, expert weights: None = the run's --weights); an
# entry with its own weights is keyed "config:weights"
EXTRA_CONFIGS = [("prefill_h4096", False, None), ("prefill_h2048", False, None),
                 ("mixtral_prefill", False, None),
                 ("decode_t1", True, None), ("decode_t4", True, None), ("decode_t16", True, None),
                 ("decode_t64", True, None), ("mixtral_decode_t1", True, None),
                 ("decode_t1", True, "q4"), ("decode_t4", True, "q4"), ("decode_t16", True, "q4"),
                 ("decode_t64", True, "q4"), ("mixtral_decode_t1", True, "q4")]


def measure(moe, cfg, args, world, rank, local, dev, graph, want_e2e, want_clocks,
            weights=None):
    """Times K forwards of cfg (after warm-up) and a second pass with stage
    events; returns the fields of one result (main line or extra entry).
    weights: the expert weight format (default: --weights)."""
    weights = weights or args.weights
    inp = mi.make_inputs(cfg, dev, seed=replica_seed(cfg, rank))
    T, H, E, K, I = cfg.T, cfg.H, cfg.E, cfg.K, cfg.I
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    logits = torch.empty((T, E), dtype=torch.float32, device=dev)
    idx = torch.empty((T, K), dtype=torch.int32, device=dev)
    w = torch.empty((T, K), dtype=torch.float32, device=dev)
    aux = torch.empty((1,), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    packed = None
    q4 = None
    if weights == "packed" and moe.moe_packed_experts_bytes(H, E, I):
        # one-time weight layout transform (model load), outside every timed region
        packed = moe.moe_pack_experts(inp["W_gate"], inp["W_up"], inp["W_down"])
        torch.cuda.synchronize()
    if weights == "q4":
        q4 = moe.moe_quantize_experts_q4(inp["W_gate"], inp["W_up"], inp["W_down"])
        torch.cuda.synchronize()

    def forward(workspace=None):
        if q4 is not None:
            moe.moe_forward_q4(inp["x"], inp["W_router"], q4, K, cfg.norm, out=out,
                               router_logits=logits, topk_idx=idx, topk_w=w, aux=aux,
                               workspace=workspace)
        elif packed is not None:
            moe.moe_forward_packed(inp["x"], inp["W_router"], packed, K, cfg.norm, out=out,
                                   router_logits=logits, topk_idx=idx, topk_w=w, aux=aux,
                                   workspace=workspace)
        else:
            moe.moe_forward(inp["x"], inp["W_router"], inp["W_gate"], inp["W_up"], inp["W_down"],
                            K, cfg.norm, out=out, router_logits=logits, topk_idx=idx, topk_w=w,
                            aux=aux, workspace=workspace)

    def eager():
        forward()

    eager()
    torch.cuda.synchronize()
    counts = moe.moe_last_expert_counts(E).numpy()
    n0 = moe.moe_kernel_launch_count()
    eager()
    launches_per_step = moe.moe_kernel_launch_count() - n0
    step = eager
    if graph:
        # A serving loop replays the captured forward: the caller owns the
        # workspace, and the host enqueues one graph launch per step.
        ws = torch.empty(moe.moe_workspace_bytes(T, H, E, K, I), dtype=torch.uint8, device=dev)

        def fwd_ws():
            forward(ws)

        fwd_ws()
        torch.cuda.synchronize()
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg):
            fwd_ws()
        step = cg.replay

    # warm-up: at least W steps and at least ~1 s of work so clocks settle
    t_end = time.time() + args.warmup_seconds
    n = 0
    while n < max(3, args.warmup) or time.time() < t_end:
        step()
        n += 1
        if n % 50 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()

    # Timed region: K steps enqueued back to back (no host wait inside), each
    # bracketed by CUDA events on the launch stream, L2 flushed between steps
    # outside the events.  No stage events here: an event recorded between two
    # kernels serialises that boundary and would hide the programmatic overlap.
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    if want_clocks:
        sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    launches0 = moe.moe_kernel_launch_count()
    t0 = time.time()
    for k in range(args.steps):
        flush.zero_()
        ev0[k].record(stream)
        step()
        ev1[k].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    launches = moe.moe_kernel_launch_count() - launches0
    if graph:  # graph replays bypass the library's launch counter
        launches = launches_per_step * args.steps
    rows = sampler.stop() if want_clocks else None
    clocks = ClockSampler.summarize(rows, t0, t1) if rows is not None else {"reasons": ["unsampled"]}

    # Second timed pass, same workload: per-step stage-boundary events recorded
    # by the library on the launch stream give each kernel's live duration (the
    # roofline's kernel time and the stage split).
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(moe.STAGE_NAMES) + 1)]
           for _ in range(args.steps)]
    for row in evs:
        for e in row:
            e.record(stream)  # creates the CUDA events
    torch.cuda.synchronize()
    for k in range(args.steps):
        flush.zero_()
        moe.moe_set_next_stage_events(evs[k])
        eager()
    torch.cuda.synchronize()
    stage_ms = {name: [evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(args.steps)]
                for i, name in enumerate(moe.STAGE_NAMES)}
    step_ms = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    mean_ms = sum(step_ms) / len(step_ms)
    mean_ms_all = max_over_ranks(mean_ms, world, dev)
    value = aggregate_value(T, world, mean_ms_all)
    assert moe.moe_device_status() == 0, "device-side timeout during the benchmark"

    pk = peaks()
    path_name = (q4_path_name(args.expert_path, cfg) if q4 is not None
                 else expert_path_name(args.expert_path, cfg))
    wb = WEIGHT_BYTES["q4" if q4 is not None else "bf16"]
    work, touched = stage_work(cfg, counts, fused=path_name == "tcgen05_decode", wb=wb)
    stage_mean = {k: sum(v) / len(v) for k, v in stage_ms.items()}
    roof = roofline_of(work, stage_mean, path_name, pk, cfg,
                       "q4" if q4 is not None else weights)
    block = block_roofline_of(cfg, counts, wb, mean_ms, pk)

    e2e = None
    if want_e2e:
        e2e = e2e_measure(moe, inp, cfg, args, stream, flush, world, dev, packed, q4)
    res = {
        "value": value, "unit": UNIT, "ms_per_step": mean_ms_all,
        "launch": "CUDA graph replay" if graph else "eager launches",
        "expert_weights": (
            "quantised once to 4 bits, groups of 128 with a bf16 scale and bias "
            "(moe_quantize_experts_q4, a model-load step)" if q4 is not None
            else "packed once into the tile-major layout before timing "
                 "(moe_pack_experts, a model-load step)" if packed is not None
            else "row-major"),
        "roofline": roof, "block_roofline": block, "e2e": e2e, "gpu_launches": launches,
        "clocks": {"sm_mhz": clocks.get("sm_mhz"), "sm_max_mhz": clocks.get("sm_max_mhz"),
                   "reasons": clocks.get("reasons"), "samples": clocks.get("samples")},
        "stage_ms": {k: round(v, 5) for k, v in stage_mean.items()},
        "expert_path": path_name,
    }
    bits = {k: mi.bits(v) for k, v in inp.items()} if (rank == 0 and world == 1) else None
    del inp, out, logits, idx, w, aux, flush, packed, q4
    torch.cuda.empty_cache()
    return res, bits


def run_ours(args, world, rank, local):
    import mixture_experts_layer_98_b300 as moe
    from mixture_experts_layer_98_b300 import build
    if rank == 0:
        build.build()
    barrier(world)
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    moe.moe_set_expert_path({"auto": 0, "streaming": 1, "tcgen05": 2, "tcgen05_wt": 3,
                             "tcgen05_pair": 4, "tcgen05_decode": 5,
                             "warp_mma": 6}[args.expert_path])
    cfg = workload(args)
    main, bits = measure(moe, cfg, args, world, rank, local, dev, graph=args.graph,
                         want_e2e=not args.no_e2e, want_clocks=not args.quiet_clocks)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, n, dt, threads = oracle_sample_rate(cfg, bits, args.cpu_seconds)
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"first {n} of {cfg.T} tokens of {cfg.name} (full forward for those "
                         f"tokens), {dt:.1f} s, fp64 C oracle"}
    del bits

    extras = {}
    if not args.no_extras and not args.shape:
        for name, graph, ew in EXTRA_CONFIGS:
            if name == cfg.name and ew in (None, args.weights):
                continue
            ecfg = mi.CONFIGS[name]
            r, _ = measure(moe, ecfg, args, world, rank, local, dev, graph=graph, want_e2e=False,
                           want_clocks=not args.quiet_clocks, weights=ew)
            r.pop("e2e")
            r["config"] = config_block(ecfg, world)["workload"]
            extras[name if ew is None else f"{name}:{ew}"] = r

    if rank == 0:
        line = {
            "metric": METRIC, "value": main["value"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": main["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": dict(config_block(cfg, world), launch=main["launch"],
                           expert_weights=main["expert_weights"]),
            "roofline": main["roofline"], "block_roofline": main["block_roofline"],
            "cpu_baseline": cpu, "e2e": main["e2e"], "gpu_launches": main["gpu_launches"],
            "clocks": main["clocks"], "stage_ms": main["stage_ms"],
            "expert_path": main["expert_path"],
            "extra_configs": extras,
        }
        print(json.dumps(line), flush=True)


def q4_path_name(flag, cfg):
    """Which 4-bit expert kernels the library runs for this flag and shape."""
    if flag == "warp_mma" or (flag != "tcgen05" and cfg.T <= 64):
        return "warp_mma_q4"
    return "tcgen05_q4"


def expert_path_name(flag, cfg):
    """Which expert kernels the library runs for this flag and shape."""
    wt_ok = cfg.I % 128 == 0 and cfg.H % 256 == 0  # also the CTA-pair kernels' condition
    if flag == "warp_mma":  # 4-bit experts only; bf16 weights run AUTO's choice
        flag = "auto"
    if flag == "auto":
        if cfg.T * cfg.K >= 32 * cfg.E:
            pair = wt_ok and cfg.E <= 32 and cfg.T * cfg.K >= 1024 * cfg.E
            return "tcgen05_pair" if pair else "tcgen05"
        if wt_ok and 1 <= cfg.T <= 16:
            return "tcgen05_decode"
        return "tcgen05_wt" if wt_ok else "streaming"
    if flag in ("tcgen05_wt", "tcgen05_decode") and not wt_ok:
        return "streaming"
    if flag == "tcgen05_decode" and not 1 <= cfg.T <= 64:
        return "tcgen05_wt"
    if flag == "tcgen05_pair" and not wt_ok:
        return "tcgen05"
    return flag


def e2e_measure(moe, inp, cfg, args, stream, flush, world, dev, packed, q4=None):
    T, H, E, K = cfg.T, cfg.H, cfg.E, cfg.K
    x_h = inp["x"].cpu().pin_memory()
    out_h = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    lg_h = torch.empty((T, E), dtype=torch.float32).pin_memory()
    aux_h = torch.empty(1, dtype=torch.float32).pin_memory()

    def call():
        if q4 is not None:
            moe.moe_forward_host_q4(x_h, inp["W_router"], q4, K, cfg.norm, out_h,
                                    router_logits_host=lg_h, aux_host=aux_h)
        elif packed is not None:
            moe.moe_forward_host_packed(x_h, inp["W_router"], packed, K, cfg.norm, out_h,
                                        router_logits_host=lg_h, aux_host=aux_h)
        else:
            moe.moe_forward_host(x_h, inp["W_router"], inp["W_gate"], inp["W_up"], inp["W_down"],
                                 K, cfg.norm, out_h, router_logits_host=lg_h, aux_host=aux_h)

    for _ in range(max(3, args.warmup)):
        call()
    times = []
    barrier(world)
    for _ in range(args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        t = time.perf_counter()
        call()  # returns with the results in host memory
        times.append(time.perf_counter() - t)
    mean = sum(times) / len(times)
    mean = max_over_ranks(mean, world, dev)
    # the link alone: the same bytes as plain pinned copies, one way at a time
    x_d = torch.empty_like(inp["x"])
    out_d = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    lg_d = torch.empty((T, E), dtype=torch.float32, device=dev)

    def timed(fn, n=5):
        fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(n):
            t = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            ts.append(time.perf_counter() - t)
        return min(ts)

    t_h2d = timed(lambda: x_d.copy_(x_h, non_blocking=True))
    t_d2h = timed(lambda: (out_h.copy_(out_d, non_blocking=True),
                           lg_h.copy_(lg_d, non_blocking=True)))
    h2d_b, d2h_b = T * H * 2, T * H * 2 + T * E * 4 + 4
    return {"value": T * world / mean, "unit": UNIT, "h2d_bytes_per_step": h2d_b,
            "d2h_bytes_per_step": d2h_b, "ms_per_step": mean * 1e3,
            "link": {"h2d_gbs": h2d_b / t_h2d / 1e9, "d2h_gbs": (d2h_b - 4) / t_d2h / 1e9,
                     "copy_ms": (t_h2d + t_d2h) * 1e3,
                     "note": "plain pinned copies of the same bytes, best of 5; the routing "
                             "outputs are copied back while the experts run, so e2e can "
                             "undercut device time + copy_ms by their share"},
            "api": ("moe_forward_host_q4" if q4 is not None
                    else "moe_forward_host_packed" if packed is not None else "moe_forward_host")
                   + " (pinned host x in; out, router_logits, aux out)"}


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
