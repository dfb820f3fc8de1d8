"""Benchmark of the MoE FFN layer forward on GB300.

Default workload (the benchmark line): the Qwen3-235B-shaped layer (H=4096,
128 experts, top-8 softmax renormalised, expert intermediate 1536, SwiGLU,
no shared expert, bf16 weights and activations), T = 8192 tokens, seeded
synthetic inputs (x ~ N(0,1), router bias from Zipf(1.1) ranks, weights
~ N(0, 0.02)).  --config / --T / --zipf / --w-fmt select any other
workload of synth/ (the NVFP4 layers, the DeepSeek-V3 sweep).

One step = one moe_forward over the whole batch: route, (NVFP4 activation
quantisation), permute, grouped GEMM gate/up + SwiGLU, grouped GEMM down,
combine.  Inputs are resident in HBM; L2 is flushed (a 256 MB write) before
every timed step, outside the step's events.  Each step records CUDA events
at the stage boundaries (moe_forward_profiled), which gives the
grouped-GEMM kernel time live.

Prints one JSON line.  --impl reference times the fp64 CPU oracle on the
same workload (bounded token samples per step) instead.

Multi-GPU: the layer forward runs whole on each GPU (one GPU per process);
under torchrun each rank runs an independent replica on its own GPU and the
job value is the sum of tokens over the max per-rank time.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

CFG = synth.QWEN3_235B
T_MAIN = 8192
T_DECODE = 256
UNIT = "tokens/s"
# nominal dense FP4 / bf16 and FP8 / bf16 tensor throughput ratios of GB300
# (13.5 / 2.25 and 4.5 / 2.25 PFLOP/s)
FP4_OVER_BF16 = 6.0
FP8_OVER_BF16 = 2.0

# Profiling case for ncu captures: same H, k, I and rows per expert as the
# main workload (T*k/E = 512), 32 experts and T=2048 (1.2 GB of weights).
SMALL_CFG = synth.small_variant(CFG, H=4096, E=32, k=8, I=1536, name="qwen3-235b-e32")
T_SMALL = 2048


def metric_name(cfg, T):
    return f"MoE-layer tokens/s ({cfg.name} layer, {cfg.w_fmt} weights, {cfg.act_fmt} activations, T={T})"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)  # let the sampler start before the timed region
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
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


# The bf16 grouped-GEMM kernel's translation unit and every header it
# includes: the kernel is "the same" only while all of them are.
PAIR_KERNEL_SOURCES = ("mixture_experts_layer_fwd_gb300/csrc/gemm_pair.cu",
                       "mixture_experts_layer_fwd_gb300/csrc/gemm_common.cuh",
                       "mixture_experts_layer_fwd_gb300/csrc/nvfp4.cuh",
                       "mixture_experts_layer_fwd_gb300/csrc/common.cuh",
                       "mixture_experts_layer_fwd_gb300/csrc/internal.h",
                       "include/moe_gb300.h")


def pair_kernel_sources_hash():
    """sha256 over the bf16 grouped-GEMM kernel's sources, in the order of
    PAIR_KERNEL_SOURCES (None if one is missing)."""
    import hashlib
    h = hashlib.sha256()
    try:
        for rel in PAIR_KERNEL_SOURCES:
            with open(os.path.join(ROOT, rel), "rb") as f:
                h.update(f.read())
    except OSError:
        return None
    return h.hexdigest()


def gemm_traffic_per_launch():
    """DRAM bytes per grouped-GEMM launch at the bench workload, from the
    committed ncu summary -- only while the kernel's sources (the .cu and the
    headers it includes) hash to the "sources sha256 prefix" the summary
    states; otherwise None."""
    import re
    prof = os.path.join(ROOT, "profiles", "grouped_gemm_pair_qwen3-235b-e32_T2048.md")
    try:
        text = open(prof).read()
    except OSError:
        return None
    h = pair_kernel_sources_hash()
    m_h = re.search(r"sources sha256 prefix ([0-9a-f]{8,})", text)
    m_t = re.search(r"scales to ([0-9.]+) GB per launch", text)
    if h is None or not (m_h and m_t) or not h.startswith(m_h.group(1)):
        return None
    return float(m_t.group(1)) * 1e9


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def dist_teardown(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


def max_over_ranks(v: float, world: int, device) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, local_s: float, world: int, device) -> tuple[float, float]:
    """Whole-job throughput of N independent replicas: the units all ranks
    processed over the slowest rank's time.  Returns (rate, max seconds)."""
    slowest = max_over_ranks(local_s, world, device)
    return world * units_per_rank / slowest, slowest


def workload(args):
    if args.workload == "small":
        return SMALL_CFG, T_SMALL
    if args.config is None:
        return CFG, (CFG.E // CFG.k if args.forced else (args.T or T_MAIN))
    if args.config == "deepseek-v3-sweep":
        cfg = synth.sweep_config(args.w_fmt or "nvfp4", args.zipf if args.zipf is not None else 1.1)
    else:
        cfg = synth.CONFIGS[args.config]
        if args.zipf is not None:
            cfg = dataclasses.replace(cfg, zipf=args.zipf)
    T = args.T or max(cfg.Ts)
    if args.forced:
        if cfg.E % cfg.k:
            raise SystemExit(f"--forced needs E % k == 0 ({cfg.name}: E={cfg.E}, k={cfg.k})")
        T = cfg.E // cfg.k  # every expert receives exactly one token
    if args.experts:
        # profiling variant: fewer experts, same tokens per expert (T*k/E)
        T = max(1, T * args.experts // cfg.E)
        cfg = dataclasses.replace(cfg, E=args.experts, name=f"{cfg.name}-e{args.experts}")
    return cfg, T


# ------------------------------------------------------------------ model
def bytes_per_elem(fmt: str) -> float:
    # NVFP4: 4-bit code + one E4M3 byte per 16; MXFP8: one byte + one E8M0 byte
    # per 32; MXFP4: 4-bit code + one E8M0 byte per 32
    return {"bf16": 2.0, "nvfp4": 0.5625, "mxfp8": 1.03125, "mxfp4": 0.53125}[fmt]


def gemm_work(cfg, T, active_experts):
    """Algorithmic flops and DRAM bytes of the two grouped-GEMM launches of
    one step: weights of the experts that received tokens (+ shared expert),
    A read once, C written once."""
    flops = cfg.flops_per_token() * T
    wb = bytes_per_elem(cfg.w_fmt)
    ab = bytes_per_elem(cfg.act_fmt)
    Tk = T * cfg.k
    weights = (active_experts * 3 * cfg.H * cfg.I + 3 * cfg.H * cfg.I_s) * wb
    acts = (Tk * cfg.H + T * cfg.H * (1 if cfg.I_s else 0)) * ab      # GEMM1 A
    acts += 2 * (Tk * cfg.I + T * cfg.I_s) * ab                       # h written, read back
    acts += (Tk + (T if cfg.I_s else 0)) * cfg.H * 2                  # GEMM2 output (bf16)
    return flops, weights + acts, weights


def gemm_kernel_name(cfg, T=None):
    """The grouped-GEMM kernels a layer's formats and shapes dispatch to (the
    NVFP4 kernels with 256-element k stages need every reduction length, H
    and I, to be a multiple of 256; with 512-element multiples and at least
    64 routed rows per expert on average, the down projection takes the
    CTA-pair kernel)."""
    if cfg.w_fmt == "bf16" and cfg.act_fmt == "bf16":
        return "grouped_gemm_pair_kernel"
    if cfg.w_fmt == "mxfp8":
        return "grouped_gemm_mxf8p_kernel"
    if cfg.w_fmt == "mxfp4":
        return "grouped_gemm_mxf4_kernel"
    k256 = cfg.H % 256 == 0 and cfg.I % 256 == 0 and cfg.I_s % 256 == 0
    if cfg.w_fmt == "nvfp4" and cfg.act_fmt == "nvfp4":
        k512 = cfg.H % 512 == 0 and cfg.I % 512 == 0 and cfg.I_s % 512 == 0
        if k512 and T is not None and T * cfg.k >= 64 * cfg.E:
            return "grouped_gemm_nvf4w_kernel (gate/up) + grouped_gemm_nvf4p_kernel (down)"
        return "grouped_gemm_nvf4w_kernel" if k256 else "grouped_gemm_nvf4_kernel"
    return "grouped_gemm_w4a16_kernel" if k256 else "grouped_gemm_kernel"


def tensor_peak(cfg, p):
    """Dense tensor peak of the MMA the path runs: bf16 (bf16 layers and the
    NVFP4-weight / bf16-activation layer, whose MMA is bf16), or NVFP4 (both
    operands NVFP4: block-scaled FP4 MMA) = measured bf16 x the nominal ratio."""
    if (cfg.w_fmt, cfg.act_fmt) in (("nvfp4", "nvfp4"), ("mxfp4", "mxfp4")):
        return p["bf16_tflops"] * FP4_OVER_BF16, cfg.w_fmt, f"bf16_tflops x {FP4_OVER_BF16:g} (nominal fp4/bf16)"
    if cfg.w_fmt == "mxfp8":
        return p["bf16_tflops"] * FP8_OVER_BF16, "mxfp8", f"bf16_tflops x {FP8_OVER_BF16:g} (nominal fp8/bf16)"
    return p["bf16_tflops"], "bf16", "bf16_tflops (burst)"


def roofline(cfg, T, gemm_ms, active, traffic, src):
    p, _ = peaks()
    flops, nbytes, wbytes = gemm_work(cfg, T, active)
    tpk, mma, how = tensor_peak(cfg, p)
    t_tensor = flops / (tpk * 1e12)
    t_hbm = nbytes / (p["hbm_gbs"] * 1e9)
    sec = gemm_ms / 1e3
    if t_tensor >= t_hbm:
        ach = flops / sec / 1e12
        r = {"bound": "tensor", "achieved": round(ach, 1), "peak": round(tpk, 1), "unit": "TFLOP/s",
             "frac": round(ach / tpk, 4), "peak_source": f"{how} of {src} peaks",
             "algorithmic": f"{flops / 2 / 1e9:.1f} GFLOP per launch ({cfg.flops_per_token() / 1e6:.1f} "
                            f"MFLOP/token x {T} tokens / 2 launches)"}
    else:
        ach = nbytes / sec / 1e9
        r = {"bound": "hbm", "achieved": round(ach, 1), "peak": p["hbm_gbs"], "unit": "GB/s",
             "frac": round(ach / p["hbm_gbs"], 4), "peak_source": f"hbm_gbs of {src} peaks",
             "algorithmic": f"{nbytes / 2 / 1e9:.3f} GB per launch ({wbytes / 1e9:.3f} GB of weights of "
                            f"{active} active experts per step)"}
    r.update({"traffic": traffic, "kernel": f"{gemm_kernel_name(cfg, T)} (2 launches/step)", "mma": mma,
              "t_roof_ms": round(max(t_tensor, t_hbm) * 1e3, 4)})
    return r


# ------------------------------------------------------------------ oracle
# One method for both CPU legs (the GPU arm's cpu_baseline and --impl
# reference): the oracle's expert weights are widened to fp64 once, before
# any timing (as the GPU path's weights are prepared once), and each timed
# step runs oracle.forward on a fresh seeded sample of ORACLE_SAMPLE tokens
# of the T = 8192 batch.  Every output row depends only on its own token, so
# a sample is exact work of the workload; tokens/s = sampled tokens / time.
ORACLE_SAMPLE = 512


def oracle_experts(w_host):
    """fp64 ExpertWeights of every expert, from the bf16 masters on the host."""
    import oracle
    w13, w2 = w_host
    return [oracle.ExpertWeights(w13[e].double().numpy(), w2[e].double().numpy()) for e in range(w13.shape[0])]


def oracle_step_s(cfg, acts, experts, tokens):
    """Seconds of one oracle.forward (as it stands) over `tokens`."""
    import oracle
    x = acts.x.double().numpy()
    logits = acts.logits.numpy()
    t0 = time.perf_counter()
    oracle.forward(x, logits, cfg.k, cfg.E, lambda e: experts[e], None, tokens=tokens)
    return time.perf_counter() - t0


def oracle_run(cfg, T, acts, experts, steps, seed0):
    """`steps` oracle steps on fresh samples; returns (tokens/s, seconds per step)."""
    times = [oracle_step_s(cfg, acts, experts, synth.sample_tokens(T, ORACLE_SAMPLE, seed=seed0 + i))
             for i in range(steps)]
    return ORACLE_SAMPLE * steps / sum(times), times


def cpu_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_sample_note(T, steps):
    return (f"{steps} steps of {ORACLE_SAMPLE} seeded tokens of the T={T} batch (fresh sample per step; "
            f"rows are token-independent), expert weights widened to fp64 once before timing")


def run_reference(args):
    """--impl reference: the CPU oracle on the bench workload, W + K steps
    of the oracle method above."""
    # rank 0 alone runs the oracle; the other ranks exit without work and
    # without joining a process group
    if int(os.environ.get("RANK", "0")) != 0:
        return
    cfg, T = CFG, T_MAIN
    acts = synth.make_activations(cfg, T, seed=0)
    w = synth.make_weights(cfg, seed=0, device="cuda" if torch.cuda.is_available() else "cpu")
    experts = oracle_experts((w.w13.cpu(), w.w2.cpu()))
    del w
    oracle_run(cfg, T, acts, experts, args.warmup, seed0=100)
    value, times = oracle_run(cfg, T, acts, experts, args.steps, seed0=100 + args.warmup)
    line = {
        "impl": "reference", "metric": metric_name(cfg, T), "value": round(value, 3), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * sum(times) / args.steps, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{cfg.name} moe layer bf16 weights, T={T} (oracle on {ORACLE_SAMPLE}-token "
                               f"samples)",
                   "H": cfg.H, "E": cfg.E, "k": cfg.k, "I": cfg.I, "T": T, "zipf": cfg.zipf},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                         "sample": oracle_sample_note(T, args.steps)},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
# The NVFP4 and MX workloads measured on the default run besides the
# benchmark line's own (each carries its own roofline): the Qwen3.5-397B-
# shaped layer (NVFP4 weights, bf16 activations) at decode and prefill sizes,
# the DeepSeek-V3-shaped layer (NVFP4 weights and activations), and the
# Qwen3-235B-shaped layer in MXFP8 (the format the pages serve it in).
EXTRA_POINTS = (("qwen35-397b", (64, 512, 4096)), ("deepseek-v3", (256, 16384)), ("qwen3-235b-mxfp8", (256, 8192)))
EXTRA_STEPS = 20
STAGES = ["quant", "dispatch", "gemm_gate_up", "gemm_down", "combine"]
N_EVENTS = len(STAGES) + 1


def new_events():
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(N_EVENTS)]
    for ev in evs:
        ev.record()  # creates the underlying CUDA events
    return evs


def timed_steps(api, layer, x, logits, out, ws, flush, steps, warmup, evsets=None):
    """warmup + steps forwards (moe_forward_profiled), L2 flushed before each
    (outside the events).  Returns the per-step event sets of the timed ones."""
    warm = new_events()
    for _ in range(warmup):
        flush.zero_()
        api.moe_forward_profiled(layer.c, x, logits, out, ws, warm)
    evsets = evsets or [new_events() for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        flush.zero_()
        api.moe_forward_profiled(layer.c, x, logits, out, ws, evsets[i])
    torch.cuda.synchronize()
    return evsets


def stage_table(evsets):
    return np.array([[evs[i].elapsed_time(evs[i + 1]) for i in range(len(STAGES))] for evs in evsets])


def active_experts(api, logits, cfg):
    idx, _ = api.moe_route(logits, cfg.k)
    return int((torch.bincount(idx.reshape(-1).long(), minlength=cfg.E) > 0).sum())


def measure_point(api, moe_sync_status, layer, cfg, T, dev, flush, steps, warmup, src):
    """One workload point: mean step time, stage times and the grouped-GEMM
    roofline over `steps` timed forwards."""
    acts = synth.make_activations(cfg, T, seed=0)
    x, logits = acts.x.to(dev), acts.logits.to(dev)
    out = torch.empty(T, cfg.H, dtype=torch.bfloat16, device=dev)
    ws = layer.workspace(T)
    evsets = timed_steps(api, layer, x, logits, out, ws, flush, steps, warmup)
    if moe_sync_status() != 0:
        raise RuntimeError(f"device status not clean at {cfg.name} T={T}")
    st = stage_table(evsets)
    ms = float(np.mean([evs[0].elapsed_time(evs[-1]) for evs in evsets]))
    gemm_ms = float(np.mean(st[:, 2] + st[:, 3]))
    active = active_experts(api, logits, cfg)
    return {"ms": round(ms, 4), "tokens_per_s": round(T / (ms / 1e3), 1), "active_experts": active,
            "roofline": roofline(cfg, T, gemm_ms, active, None, src),
            "stage_ms": {n: round(float(np.mean(st[:, i])), 4) for i, n in enumerate(STAGES)}}


def run_gpu(args):
    from mixture_experts_layer_fwd_gb300 import MoELayer, api, moe_sync_status
    from mixture_experts_layer_fwd_gb300 import build as _build

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _build.build()
    cfg, T = workload(args)
    is_main = args.workload == "main" and args.config is None and T == T_MAIN and not args.forced
    acts = synth.make_activations(cfg, T, seed=0)
    if args.forced:
        # the decode microbenchmark shape: all experts active, one token each
        _, forced_logits = synth.forced_one_token_per_expert_logits(cfg)
        acts = dataclasses.replace(acts, logits=forced_logits)
    w = synth.make_weights(cfg, seed=0, device=str(dev))
    layer = MoELayer.from_config(cfg, w)
    keep_master = rank == 0 and world == 1 and is_main and not args.no_cpu_baseline
    w_host = (w.w13.cpu(), w.w2.cpu()) if keep_master else None
    del w  # the layer holds its own copy or encoding of the weights
    torch.cuda.empty_cache()
    x = acts.x.to(dev)
    logits = acts.logits.to(dev)
    out = torch.empty(T, cfg.H, dtype=torch.bfloat16, device=dev)
    ws = layer.workspace(T)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    evsets = [new_events() for _ in range(args.steps)]
    warm = new_events()
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        flush.zero_()
        api.moe_forward_profiled(layer.c, x, logits, out, ws, warm)
    torch.cuda.synchronize()
    if moe_sync_status() != 0:
        raise RuntimeError("device status not clean after warm-up")

    graph = api.ForwardGraph(layer.c, x, logits, out, ws) if args.graph else None
    if graph is not None:
        for _ in range(3):
            graph.launch()
        torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        if graph is None:
            api.moe_forward_profiled(layer.c, x, logits, out, ws, evsets[i])
        else:
            # one graph launch per step: the step's first and last events
            # bracket it (stage times come from the profiled warm-up below)
            evsets[i][0].record()
            graph.launch()
            evsets[i][-1].record()
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    if moe_sync_status() != 0:
        raise RuntimeError("device status not clean after the timed steps")

    step_ms = [evs[0].elapsed_time(evs[-1]) for evs in evsets]
    if graph is not None:
        # per-stage times of the same forward, launched stage by stage
        timed_steps(api, layer, x, logits, out, ws, flush, args.steps, 0, evsets)
    stage_ms = stage_table(evsets)
    value, total_s = job_rate(T * args.steps, float(sum(step_ms)) / 1e3, world, dev)
    total_ms = total_s * 1e3

    active = active_experts(api, logits, cfg)
    gemm_ms = float(np.mean(stage_ms[:, 2] + stage_ms[:, 3]))
    _, src = peaks()
    roof = roofline(cfg, T, gemm_ms, active, gemm_traffic_per_launch() if is_main else None, src)

    # e2e through the C ABI with host buffers (pinned), copies inside the timing
    xh = acts.x.pin_memory()
    lh = acts.logits.pin_memory()
    oh = torch.empty(T, cfg.H, dtype=torch.bfloat16).pin_memory()
    xd = torch.empty_like(x)
    ld = torch.empty_like(logits)
    for _ in range(2):
        api.moe_forward_host(layer.c, xh, lh, oh, xd, ld, out, ws)
    e2e_t = []
    for _ in range(max(3, min(args.steps, 10))):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        api.moe_forward_host(layer.c, xh, lh, oh, xd, ld, out, ws)
        e2e_t.append(time.perf_counter() - t0)
    e2e_call_value, _ = job_rate(T, float(np.mean(e2e_t)), world, dev)
    # the serving loop: n batches through one moe_forward_host_pipelined call
    # (batch i+1's inputs copied in and batch i-1's output copied out while
    # batch i runs), two host buffer sets used alternately; every batch's
    # copies are inside the timed region
    n_pipe = max(3, min(args.steps, 10))
    xh2, lh2 = xh.clone().pin_memory(), lh.clone().pin_memory()
    oh2 = torch.empty_like(oh).pin_memory()
    xd2 = torch.empty((2,) + tuple(x.shape), dtype=x.dtype, device=dev)
    ld2 = torch.empty((2,) + tuple(logits.shape), dtype=logits.dtype, device=dev)
    od2 = torch.empty((2,) + tuple(out.shape), dtype=out.dtype, device=dev)
    compute_stream, copy_stream = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    pick = lambda a, b, m: [a if i % 2 == 0 else b for i in range(m)]
    api.moe_forward_host_pipelined(layer.c, pick(xh, xh2, 2), pick(lh, lh2, 2), pick(oh, oh2, 2), xd2, ld2, od2,
                                   ws, stream=compute_stream, copy_stream=copy_stream)
    flush.zero_()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    api.moe_forward_host_pipelined(layer.c, pick(xh, xh2, n_pipe), pick(lh, lh2, n_pipe), pick(oh, oh2, n_pipe),
                                   xd2, ld2, od2, ws, stream=compute_stream, copy_stream=copy_stream)
    pipe_s = time.perf_counter() - t0
    e2e_value, _ = job_rate(T, pipe_s / n_pipe, world, dev)
    del xd2, ld2, od2

    a4 = cfg.act_fmt == "nvfp4"
    # fused route + permutation (its barrier-counter memset is not a kernel),
    # 2 grouped GEMMs, combine (+ amax and quantise on NVFP4 activations)
    launches = 4 + (2 if a4 else 0)
    line = {
        "metric": metric_name(cfg, T), "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "nvfp4" if a4 else "bf16", "data": "synthetic",
        "config": {"workload": f"{cfg.name} moe layer, {cfg.w_fmt} weights, {cfg.act_fmt} activations, T={T}"
                               + (", routing forced to one token per expert" if args.forced else ""),
                   "H": cfg.H, "E": cfg.E, "k": cfg.k, "I": cfg.I, "I_s": cfg.I_s, "T": T, "zipf": cfg.zipf,
                   "seed": 0, "active_experts": active,
                   "l2": "flushed before every step (256 MB write, outside the events)",
                   "parallelism": f"replicas x{world}", "cuda_graph": bool(args.graph)},
        "roofline": roof,
        "stage_ms": {n: round(float(np.mean(stage_ms[:, i])), 4) for i, n in enumerate(STAGES)},
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT,
                "h2d_bytes_per_step": T * cfg.H * 2 + T * cfg.E * 4, "d2h_bytes_per_step": T * cfg.H * 2,
                "mode": f"moe_forward_host_pipelined over {n_pipe} batches (pinned host buffers; a batch's "
                        "copies overlap its neighbours' compute; per-step working set > L2)",
                "per_call_value": round(e2e_call_value, 1),
                "per_call_mode": "moe_forward_host, one synchronous call per step, L2 flushed before each"},
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
    }

    if is_main:
        # decode-size point on the same weights (weight-streaming bound)
        line["decode_T256"] = measure_point(api, moe_sync_status, layer, cfg, T_DECODE, dev, flush, 10,
                                            args.warmup, src)
    del layer, ws, out
    torch.cuda.empty_cache()
    if is_main and world == 1 and not args.no_extra:
        # the NVFP4 workloads, each point with its own roofline
        for name, Ts in EXTRA_POINTS:
            c = synth.CONFIGS[name]
            wc = synth.make_weights(c, seed=0, device=str(dev))
            lc = MoELayer.from_config(c, wc)
            del wc
            torch.cuda.empty_cache()
            for Tc in Ts:
                line[f"{name}_T{Tc}"] = measure_point(api, moe_sync_status, lc, c, Tc, dev, flush, EXTRA_STEPS,
                                                      args.warmup, src)
            del lc
            torch.cuda.empty_cache()
    if keep_master:
        experts = oracle_experts(w_host)
        del w_host
        steps = 0
        r, times = oracle_run(cfg, T, acts, experts, 1, seed0=1)
        # about 10-30 s of CPU work: as many sample steps as fit in ~15 s
        steps = max(1, min(30, int(15.0 / max(times[0], 1e-3))))
        r, times = oracle_run(cfg, T, acts, experts, steps, seed0=2)
        line["cpu_baseline"] = {"value": round(r, 3), "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                                "sample": oracle_sample_note(T, steps) + f" ({sum(times):.1f} s)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    dist_teardown(world)


def run_sweep(args):
    """--sweep: the size and load-imbalance sweep on DeepSeek-V3 shapes
    (T = 1..65536 in powers of 2, router-bias Zipf exponent 0 / 1.1 / 2.0,
    bf16 weights with bf16 activations and NVFP4 weights with NVFP4
    activations).  One JSON line per point.  The weights of a format are built
    once; each point runs on the first T tokens of one seeded 65536-token batch
    per Zipf exponent (rows are token-independent, so the prefix is a T-token
    batch of the same distribution).  Not the benchmark line."""
    from mixture_experts_layer_fwd_gb300 import MoELayer, api, moe_sync_status
    from mixture_experts_layer_fwd_gb300 import build as _build

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    _build.build()
    _, src = peaks()
    Ts = [int(t) for t in args.sweep_ts.split(",")] if args.sweep_ts else list(synth.SWEEP_TS)
    fmts = [args.w_fmt] if args.w_fmt else ["bf16", "nvfp4"]
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    Tmax = max(Ts)
    for fmt in fmts:
        cfg0 = synth.sweep_config(fmt, 1.1)
        w = synth.make_weights(cfg0, seed=0, device=str(dev))
        layer = MoELayer.from_config(cfg0, w)
        del w
        torch.cuda.empty_cache()
        ws = layer.workspace(Tmax)
        out_full = torch.empty(Tmax, cfg0.H, dtype=torch.bfloat16, device=dev)
        for z in synth.SWEEP_ZIPF:
            cfg = synth.sweep_config(fmt, z)
            acts = synth.make_activations(cfg, Tmax, seed=0)
            x_full, lg_full = acts.x.to(dev), acts.logits.to(dev)
            for T in Ts:
                x, lg, out = x_full[:T].contiguous(), lg_full[:T].contiguous(), out_full[:T]
                evs = [torch.cuda.Event(enable_timing=True) for _ in range(N_EVENTS)]
                for ev in evs:
                    ev.record()
                steps = args.sweep_steps
                res = []
                for i in range(args.warmup + steps):
                    flush.zero_()
                    api.moe_forward_profiled(layer.c, x, lg, out, ws, evs)
                    torch.cuda.synchronize()
                    if i >= args.warmup:
                        res.append((evs[0].elapsed_time(evs[-1]), evs[2].elapsed_time(evs[4])))
                if moe_sync_status() != 0:
                    raise RuntimeError(f"device status not clean at {fmt} z={z} T={T}")
                idx, _ = api.moe_route(lg, cfg.k)
                active = int((torch.bincount(idx.reshape(-1).long(), minlength=cfg.E) > 0).sum())
                ms = float(np.median([r[0] for r in res]))
                gms = float(np.median([r[1] for r in res]))
                roof = roofline(cfg, T, gms, active, None, src)
                print(json.dumps({"sweep": "deepseek-v3 shapes", "w_fmt": fmt, "act_fmt": cfg.act_fmt, "zipf": z,
                                  "T": T, "active_experts": active, "ms_per_step": round(ms, 4),
                                  "tokens_per_s": round(T / (ms / 1e3), 1), "gemm_ms": round(gms, 4),
                                  "roofline": {k: roof[k] for k in ("bound", "achieved", "unit", "frac")}}),
                      flush=True)
            del x_full, lg_full
        del layer, ws, out_full
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the NVFP4 workload points of the default run")
    ap.add_argument("--workload", default="main", choices=["main", "small"],
                    help="main: the benchmark workload; small: the ncu profiling case")
    ap.add_argument("--config", default=None, choices=list(synth.CONFIGS) + ["deepseek-v3-sweep"],
                    help="measure another workload of synth/ instead of the benchmark one")
    ap.add_argument("--T", type=int, default=None, help="tokens (default: the workload's largest)")
    ap.add_argument("--zipf", type=float, default=None, help="router-bias Zipf exponent override")
    ap.add_argument("--w-fmt", default=None, choices=["bf16", "nvfp4"], help="sweep weight format")
    ap.add_argument("--sweep", action="store_true",
                    help="run the DeepSeek-V3-shape size / imbalance sweep (one JSON line per point)")
    ap.add_argument("--sweep-ts", default=None, help="comma-separated T values of the sweep (default 1..65536)")
    ap.add_argument("--sweep-steps", type=int, default=10, help="timed steps per sweep point")
    ap.add_argument("--graph", action="store_true",
                    help="time the forward replayed as one CUDA graph (moe_forward_graph_create)")
    ap.add_argument("--forced", action="store_true",
                    help="route every expert exactly one token (T = E / k; the decode microbenchmark shape)")
    ap.add_argument("--experts", type=int, default=None,
                    help="profiling variant: this many experts, tokens scaled to keep tokens per expert")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.sweep:
        run_sweep(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
