#!/usr/bin/env python
"""Benchmark of the Stable LatentMoE layer forward on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one lmoe_forward of the whole layer (router, dispatch, latent
down-projection, routed MXFP4 experts, combine + RMSNorm, shared experts,
output GEMM) over one batch of seeded synthetic tokens; weights and tokens
resident in HBM.  Tokens rotate over 4 seeded batches so the routed expert
set changes between steps; every step streams the selected experts' weights
(~11 GB at T = 64), far more than the 129 MB L2, so no flush is needed.

Under torchrun (N > 1) every rank runs its own replica on its own tokens
(the layer is per-token: no collective on the data path); value = tokens of
all ranks / the slowest rank's time.

Prints one JSON line: metric/value (device-timed tokens/s), e2e (through
lmoe_forward_host with host buffers and the copies inside the timed
region), roofline of the dominant kernel (the grouped MXFP4 gate/up GEMM,
algorithmic bytes over its CUDA-event time), the whole-layer HBM roofline,
per-stage times, clocks sampled during the timed region, and the fp64
oracle timed on the host cores as cpu_baseline.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
from dataclasses import replace

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# Forwards of the timed region whose expert kernels carry timing events.
PROFILE_PERIOD = 8
METRIC = "LatentMoE layer tokens/s at T=1..8192; % of HBM or FP4-TC roofline"
UNIT = "tokens/s"
# DRAM bytes (read + write) per algorithmic byte of the gate/up expert
# kernel of each weight format, from one ncu capture of the kernel as it
# stands on a small case of the same instantiation (K3 shapes with 64
# experts at T = 8: 702.8 MB for 645.2 MB; K2 shapes with 32 experts at
# T = 384: 1043.2 MB for 998.1 MB), keyed by (weight format, token tile).
# An entry is removed when its kernel changes until it is captured again.
GU_DRAM_PER_ALGO_BYTE = {("mxfp4", 16): 1.089, ("fp8_block128", 96): 1.045}


def expert_tile(cfg, T: int) -> int:
    """Token tile the library picks for the grouped expert GEMMs (the rule of
    moe_tile_tokens / fp8_tile_tokens in the library's internal header)."""
    P, E = T * cfg.top_k, cfg.n_experts
    if cfg.expert_wfmt == "mxfp4":
        return 16 if P <= 4 * E else 32 if P <= 16 * E else 64 if P <= 64 * E else 96
    m = -(-P // E)
    return 16 if m <= 16 else 32 if m <= 32 else 64 if m <= 64 else 96


def _mat_bytes(cfg, N: int, K: int) -> int:
    """Stored bytes of one N x K weight matrix in the expert format: MXFP4
    (two E2M1 codes per byte + one E8M0 per 32) or FP8 E4M3 with an fp32
    scale per 128 x 128 block."""
    if cfg.expert_wfmt == "mxfp4":
        return N * K // 2 + N * K // 32
    return N * K + 4 * (-(-N // 128)) * (-(-K // 128))


def accounting(cfg) -> dict:
    """Algorithmic bytes and FLOPs of the layer (each weight byte read once,
    activations between kernels in the format the path stores them).

    expert: weight bytes of one routed expert (gate + up + down);
    dense: router (bf16 + fp32 bias), latent projections and norm (bf16),
    shared MLP (bf16 for K3, FP8 block-128 as stored for K2);
    token_io: x in + Delta out (bf16); flops_per_token: 2 x MACs of every
    contraction (router, latent, k experts, shared)."""
    d, l, E, k, F, Fs = cfg.d_model, cfg.d_latent, cfg.n_experts, cfg.top_k, cfg.d_expert_ff, cfg.d_shared_ff
    din = l or d
    gu_w = 2 * _mat_bytes(cfg, F, din)
    dn_w = _mat_bytes(cfg, din, F)
    dense = E * d * 2 + E * 4
    if l:
        dense += 2 * l * d * 2 + (l * 2 if cfg.use_latent_norm else 0)
    if Fs:
        dense += 3 * Fs * d * 2 if cfg.expert_wfmt == "mxfp4" else 2 * _mat_bytes(cfg, Fs, d) + _mat_bytes(cfg, d, Fs)
    flops = 2 * E * d + (4 * l * d if l else 0) + k * 6 * F * din + 6 * Fs * d
    # hi/lo E4M3 activation pairs with one E8M0 per 32 in, the same for h
    act_in = 2 * din + 2 * din // 32
    h_io = 2 * F + 2 * F // 32
    return dict(din=din, gu_w=gu_w, dn_w=dn_w, expert=gu_w + dn_w, dense=dense, token_io=2 * d * 2,
                flops_per_token=flops, gu_per_assign=act_in + h_io, dn_per_assign=h_io + din * 4)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"], src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_uuid: str | None):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        # one GPU per box: sample every visible GPU
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        try:
            self.p = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self, t0: float, t1: float) -> dict:
        """Samples taken between host times t0 and t1 (the timed region)."""
        import datetime
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        rows = [[c.strip() for c in r.split(",")] for r in open(self.f.name).read().strip().splitlines()
                if r.count(",") >= 9]
        os.unlink(self.f.name)

        def ts(r):
            try:
                return datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                return None
        inside = [r for r in rows if ts(r) is not None and t0 <= ts(r) <= t1]
        rows = inside if inside else rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[2]) for r in rows if num(r[2]) is not None]
        mx = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        pw = [num(r[4]) for r in rows if num(r[4]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "samples_in_timed_region": len(inside),
                "power_w_max": max(pw) if pw else None}


# ------------------------------------------------------------- cpu oracle
def oracle_for(wl, W_dev):
    import oracle as O
    dense = {k: v for k, v in W_dev.items() if not k.startswith("ex_")}
    Wn = O.numpy_inputs(dense)
    Wn["expert_fn"] = lambda name, e: (W_dev[name + "_q"][e].cpu().numpy(), W_dev[name + "_s"][e].cpu().numpy())
    return O, Wn


def cpu_baseline(wl, W_dev, x_dev, ntok=2) -> dict:
    """The fp64 oracle, as it stands, on the first `ntok` tokens of a batch
    (its routing, 16 fresh expert dequantisations per token, dense parts)."""
    import numpy as np
    import torch
    O, Wn = oracle_for(wl, W_dev)
    xb = x_dev[:ntok].cpu().view(torch.int16).numpy().view(np.uint16)
    layer = O.Layer(wl.cfg, Wn)
    for name in ("router_w", "w_down_latent", "w_up_latent", "norm_w"):
        if name in Wn:
            layer.dense(name)        # host-side fp64 copies of the dense weights: input preparation
    for name in ("sh_gate", "sh_up", "sh_down"):
        if name in Wn:
            layer.shared(name)
    t0 = time.perf_counter()
    O.forward(layer, xb)
    dt = time.perf_counter() - t0
    return {"value": ntok / dt, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{ntok} tokens of the {wl.name} batch through the fp64 oracle (routing, "
                      f"{ntok * wl.cfg.top_k} expert dequantisations, dense parts); numpy BLAS threads = default",
            "seconds": dt}


# ------------------------------------------------------------- replicas
# One process per GPU, each a full replica of the layer on its own tokens;
# the only cross-rank traffic is the barrier and the max of the timings.
def replica_seeds(wl, rank: int, n: int = 4) -> list:
    """Seeds of rank `rank`'s n rotating token batches (distinct over ranks)."""
    return [wl.seed + 7919 * (rank * 8 + i + 1) for i in range(n)]


def max_over_ranks(v: float, world: int, device="cuda") -> float:
    """The slowest rank's value (all ranks get it)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, tokens_per_rank_step: int, steps: int, seconds: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank_step * steps / seconds


# ------------------------------------------------------------------ ours
def run_ours(args):
    import torch
    import torch.distributed as dist
    from lmoe_inputs import configs as C
    from lmoe_inputs import generate as G
    from latent_mixture_experts_gb300 import LatentMoE, build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    if rank == 0:
        build.build()
    if world > 1:
        dist.barrier()
    wl = C.workload(args.workload)
    T, cfg = wl.T, wl.cfg
    W = G.gen_weights(wl, device="cuda")
    xs = [G.gen_x(replace(wl, seed=sd), device="cuda") for sd in replica_seeds(wl, rank)]
    out = torch.empty(T, cfg.d_model, dtype=torch.bfloat16, device="cuda")
    layer = LatentMoE(cfg, W, max_tokens=T)
    stream = torch.cuda.current_stream()

    # distinct experts each batch selects (units of the expert bytes)
    U = []
    for xb in xs:
        layer.lmoe_forward(xb, out=out)
        U.append(layer.lmoe_last_active_experts())
    layer.lmoe_sync_status()
    launches = layer.lmoe_last_launch_count()

    for i in range(args.warmup):
        layer.lmoe_forward(xs[i % 4], out=out)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    # Inside the timed region only the two expert kernels carry timing events,
    # and only on every PROFILE_PERIOD-th forward (an event between two
    # kernels ends their launch overlap and costs ~10 us of a one-token
    # forward); the per-stage breakdown comes from a separate pass after it.
    layer.lmoe_set_profiling(args.steps, stages=["expert_gate_up", "expert_down"])
    layer.lmoe_set_profiling_period(PROFILE_PERIOD)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        pass
    clk = ClockSampler(uuid)
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_start = time.time()
    e0.record(stream)
    for i in range(args.steps):
        layer.lmoe_forward(xs[i % 4], out=out)
    e1.record(stream)
    torch.cuda.synchronize()
    t_end = time.time()
    if world > 1:
        dist.barrier()
    clocks = clk.stop(t_start, t_end)
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    prof = layer.lmoe_profile_get()
    n_prof = min(args.steps, 100)
    layer.lmoe_set_profiling_period(1)
    layer.lmoe_set_profiling(n_prof)
    for i in range(n_prof):
        layer.lmoe_forward(xs[i % 4], out=out)
    stage_prof = layer.lmoe_profile_get()
    layer.lmoe_set_profiling(0)
    layer.lmoe_sync_status()

    steps = args.steps
    ms_step = ms / steps
    value = job_throughput(world, T, steps, ms / 1e3)
    U_mean = sum(U[i % 4] for i in range(steps)) / steps
    pk = peaks()

    # dominant kernel: the grouped gate/up expert GEMM.  Algorithmic bytes
    # per launch: the selected experts' gate+up weights (codes and scales),
    # the hi/lo E4M3 activations in (with their scales) and the hi/lo h out.
    A = accounting(cfg)
    din, F, k = A["din"], cfg.d_expert_ff, cfg.top_k
    gu_bytes = U_mean * A["gu_w"] + T * k * A["gu_per_assign"]
    gu_ms, gu_n = prof["expert_gate_up"]
    gu_avg = gu_ms / max(gu_n, 1)
    achieved = gu_bytes / (gu_avg * 1e-3) / 1e9
    # The kernel's bound: HBM below the ridge of the measured peaks, the
    # tensor pipe above it.  Its MMAs run in FP8 (E2M1 or E4M3 weights x E4M3
    # activations) with two activation terms, i.e. two FP8 MACs per MAC of the
    # layer; the FP8 peak is the measured bf16 peak x 2 (the nominal ratio).
    gu_flops = 2.0 * T * k * 2 * cfg.d_expert_ff * din            # layer FLOPs of the gate/up GEMMs
    fp8_peak = 2.0 * pk["bf16"]
    tensor_bound = gu_flops / gu_bytes > 1e3 * pk["bf16"] / pk["hbm"]
    dn_bytes = U_mean * A["dn_w"] + T * k * A["dn_per_assign"]
    dn_ms, dn_n = prof["expert_down"]
    layer_bytes = A["dense"] + U_mean * A["expert"] + T * A["token_io"]
    fp4 = cfg.expert_wfmt == "mxfp4"
    gu_traffic = GU_DRAM_PER_ALGO_BYTE.get((cfg.expert_wfmt, expert_tile(cfg, T)))
    stages = {name: round(v[0] / max(v[1], 1), 5) for name, v in stage_prof.items()}

    # end to end through the host-buffer entry point
    xh = [xb.cpu().pin_memory() for xb in xs]
    oh = torch.empty(T, cfg.d_model, dtype=torch.bfloat16).pin_memory()
    for i in range(2):
        layer.lmoe_forward_host(xh[i], oh)
    n_e2e = max(10, min(steps, 200))
    t0 = time.perf_counter()
    for i in range(n_e2e):
        layer.lmoe_forward_host(xh[i % 4], oh)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    e2e = {"value": job_throughput(world, T, n_e2e, e2e_s), "unit": UNIT, "h2d_bytes_per_step": T * cfg.d_model * 2,
           "d2h_bytes_per_step": T * cfg.d_model * 2, "steps": n_e2e}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, W, xs[0], ntok=args.cpu_tokens)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("e2m1 x e4m3(hi+lo) block-scaled; bf16 dense; fp32 accumulate" if fp4 else
                  "e4m3 x e4m3(hi+lo), fp32 block-128 scales; bf16 dense; fp32 accumulate"),
        "data": "synthetic (seeded, N(0,1/fan_in) weights quantised to "
                + ("MXFP4" if fp4 else "FP8 E4M3 block-128") + "; x ~ N(0,1) bf16)",
        "config": {"workload": wl.name, "T": T, "d_model": cfg.d_model, "d_latent": cfg.d_latent, "n_experts": cfg.n_experts,
                   "top_k": k, "d_expert_ff": F, "d_shared_ff": cfg.d_shared_ff, "expert_format": cfg.expert_wfmt,
                   "parallelism": f"replicas x{world}", "token_batches_rotated": 4,
                   "l2": "no flush: each step streams the selected experts' weights (GBs) >> 129 MB L2",
                   "active_experts_mean": round(U_mean, 1)},
        "roofline": {"kernel": ("moe_gemm_kernel<gate/up> (grouped MXFP4 x E4M3 hi/lo, tcgen05)" if fp4 else
                                "moe_fp8_kernel<gate/up> (grouped E4M3 x E4M3 hi/lo, block-128 promotion, tcgen05)"),
                     **({"bound": "tensor", "achieved": round(2 * gu_flops / (gu_avg * 1e-3) / 1e12, 1),
                         "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                         "frac": round(2 * gu_flops / (gu_avg * 1e-3) / 1e12 / fp8_peak, 4),
                         "flops_note": "executed FP8 FLOPs (2 per layer FLOP: hi and lo activation terms) over "
                                       "the FP8 peak = measured bf16 peak x 2",
                         "hbm_gbs": round(achieved, 1)} if tensor_bound else
                        {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm"], "unit": "GB/s",
                         "frac": round(achieved / pk["hbm"], 4)}),
                     "traffic": int(gu_traffic * gu_bytes) if gu_traffic else None,
                     "traffic_source": ("ncu dram__bytes_read+write of this kernel on a small case of the same "
                                        "instantiation (" + ("profiles/moe_gemm_k3_e64_t8.md" if fp4 else
                                                             "profiles/moe_fp8_k2_e32_t384.md") +
                                        "), scaled to this launch by its algorithmic bytes"),
                     "bytes_per_launch": int(gu_bytes), "ms_per_launch": round(gu_avg, 5),
                     "launches_timed": int(gu_n),
                     "timing": f"CUDA events on the launch stream around every {PROFILE_PERIOD}th timed forward's launch",
                     "peak_source": f"{pk['src']} (MEASURED_PEAKS.json "
                                    + ("bf16_tflops x 2)" if tensor_bound else "hbm_gbs)")},
        "layer_roofline": {"bound": "hbm", "bytes_per_step": int(layer_bytes),
                           "achieved": round(layer_bytes / (ms_step * 1e-3) / 1e9, 1), "peak": pk["hbm"],
                           "unit": "GB/s", "frac": round(layer_bytes / (ms_step * 1e-3) / 1e9 / pk["hbm"], 4),
                           "tflops": round(T * A["flops_per_token"] / (ms_step * 1e-3) / 1e12, 1),
                           "frac_of_bf16_peak": round(T * A["flops_per_token"] / (ms_step * 1e-3) / 1e12
                                                      / pk["bf16"], 4),
                           "frac_of_bf16_sustained": round(T * A["flops_per_token"] / (ms_step * 1e-3) / 1e12
                                                           / pk["bf16_sus"], 4)},
        "down_kernel": {"achieved": round(dn_bytes / (dn_ms / max(dn_n, 1) * 1e-3) / 1e9, 1), "unit": "GB/s",
                        "ms_per_launch": round(dn_ms / max(dn_n, 1), 5)},
        "stage_ms": stages,
        "stage_ms_source": f"separate pass of {n_prof} forwards with every stage timed (outside the timed region)",
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": launches * steps,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    layer.close()
    if world > 1:
        dist.destroy_process_group()


# ------------------------------------------------------------------ sweep
def run_sweep(args):
    """Token-count sweep on one GPU: the K3 layer of the sweep workload (seed 4,
    uniform bias) built once, one JSON line per T with tokens/s, the layer's
    HBM-roofline fraction, its FLOP rate against the bf16 tensor peak (the hi/lo
    E4M3 activations make the routed MMAs cost what bf16 would), the expert
    kernels' GB/s and the per-stage times."""
    import torch
    from lmoe_inputs import configs as C
    from lmoe_inputs import generate as G
    from latent_mixture_experts_gb300 import LatentMoE, build
    build.build()
    torch.cuda.set_device(0)
    Ts = [int(t) for t in args.sweep.split(",")]
    wl = C.workload("k3_sweep_t1")
    cfg = wl.cfg
    W = G.gen_weights(wl, device="cuda")
    layer = LatentMoE(cfg, W, max_tokens=max(Ts))
    pk = peaks()
    A = accounting(cfg)
    flops_per_token = A["flops_per_token"]
    for T in Ts:
        wlT = replace(wl, T=T, name=f"k3_sweep_t{T}")
        xs = [G.gen_x(replace(wlT, seed=wl.seed + 7919 * (i + 1)), device="cuda") for i in range(4)]
        out = torch.empty(T, cfg.d_model, dtype=torch.bfloat16, device="cuda")
        U = []
        for xb in xs:
            layer.lmoe_forward(xb, out=out)
            U.append(layer.lmoe_last_active_experts())
        for i in range(max(args.warmup, 3)):
            layer.lmoe_forward(xs[i % 4], out=out)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        layer.lmoe_forward(xs[0], out=out)
        torch.cuda.synchronize()
        est = time.perf_counter() - t0
        steps = max(10, min(args.steps, int(0.5 / max(est, 1e-5))))
        layer.lmoe_set_profiling(steps, stages=["expert_gate_up", "expert_down"])
        layer.lmoe_set_profiling_period(PROFILE_PERIOD)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(steps):
            layer.lmoe_forward(xs[i % 4], out=out)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        prof = layer.lmoe_profile_get()
        n_prof = min(steps, 50)
        layer.lmoe_set_profiling_period(1)
        layer.lmoe_set_profiling(n_prof)
        for i in range(n_prof):
            layer.lmoe_forward(xs[i % 4], out=out)
        stage_prof = layer.lmoe_profile_get()
        layer.lmoe_set_profiling(0)
        layer.lmoe_sync_status()
        U_mean = sum(U[i % 4] for i in range(steps)) / steps
        layer_bytes = A["dense"] + U_mean * A["expert"] + T * A["token_io"]
        gu_bytes = U_mean * A["gu_w"]
        dn_bytes = U_mean * A["dn_w"]
        gu = prof["expert_gate_up"][0] / max(prof["expert_gate_up"][1], 1)
        dn = prof["expert_down"][0] / max(prof["expert_down"][1], 1)
        tflops = T * flops_per_token / (ms * 1e-3) / 1e12
        print(json.dumps({
            "workload": wlT.name, "T": T, "steps": steps, "tokens_per_s": round(T / (ms * 1e-3), 1),
            "ms_per_step": round(ms, 4), "active_experts_mean": round(U_mean, 1),
            "layer_hbm": {"bytes": int(layer_bytes), "gbs": round(layer_bytes / (ms * 1e-3) / 1e9, 1),
                          "frac": round(layer_bytes / (ms * 1e-3) / 1e9 / pk["hbm"], 4)},
            "layer_tensor": {"tflops": round(tflops, 1), "frac_of_bf16_peak": round(tflops / pk["bf16"], 4),
                             "frac_of_bf16_sustained": round(tflops / pk["bf16_sus"], 4)},
            "expert_gate_up_gbs": round(gu_bytes / (gu * 1e-3) / 1e9, 1),
            "expert_down_gbs": round(dn_bytes / (dn * 1e-3) / 1e9, 1),
            "stage_ms": {n: round(v[0] / max(v[1], 1), 4) for n, v in stage_prof.items()}}), flush=True)
    layer.close()


# ------------------------------------------------------------- reference
class ReferenceArm:
    """The fp64 oracle restated one (token, slot) assignment at a time, for
    the reference arm.  step(s) handles assignment s = t*k + j: at slot 0 it
    also runs token t's latent down-projection (latent layers) and shared
    MLP, at the last slot its RMSNorm and up-projection (latent layers);
    every step dequantises and applies one routed expert afresh.  The router
    runs on all tokens up front and the needed expert codes are generated
    before timing (input preparation).  delta[t] holds each finished token's
    Delta; a CPU test checks it against oracle.forward."""

    def __init__(self, wl, n_assign: int, dev: str = "cpu", x_seed_offset: int = 7919):
        import numpy as np
        import torch
        from lmoe_inputs import generate as G
        import oracle as O
        self.O, self.np = O, np
        self.cfg = cfg = wl.cfg
        self.k = k = cfg.top_k
        ntok = (n_assign + k - 1) // k + 1
        x = G.gen_x(replace(wl, seed=wl.seed + x_seed_offset), device="cpu", T=ntok)
        self.x_bits = x.view(torch.int16).numpy().view(np.uint16)
        Wn = O.numpy_inputs({n: t.cpu() for n, t in G.gen_dense_weights(wl, device=dev).items()})
        self.layer = layer = O.Layer(cfg, Wn)
        for name in ("router_w", "w_down_latent", "w_up_latent", "norm_w"):
            if name in Wn:
                layer.dense(name)
        for name in ("sh_gate", "sh_up", "sh_down"):
            if name in Wn:
                layer.shared(name)
        self.xo = O.bf16_bits_to_f64(self.x_bits)
        self.routes = O.router(self.xo, layer.dense("router_w"), Wn["router_bias"], k, cfg.routed_scale)
        self.need = {}
        for s in range(n_assign):
            t, j = divmod(s, k)
            e = int(self.routes["idx"][t, j])
            for m in ("ex_gate", "ex_up", "ex_down"):
                if (m, e) not in self.need:
                    q, sc = G.gen_expert(wl, m, e, device=dev)
                    self.need[(m, e)] = (q.cpu().numpy(), sc.cpu().numpy())
        self.dequant = O.dequant_mxfp4 if cfg.expert_wfmt == "mxfp4" else O.dequant_fp8_block128
        self.state = {}
        self.delta = {}

    def step(self, s: int) -> None:
        cfg, layer, st, O = self.cfg, self.layer, self.state, self.O
        t, j = divmod(s, self.k)
        if j == 0:
            x = self.xo[t]
            st["xe"] = x @ layer.dense("w_down_latent").T if cfg.d_latent else x
            st["u"] = self.np.zeros(st["xe"].shape[0])
            if cfg.d_shared_ff:
                g = x @ layer.shared("sh_gate").T
                u = x @ layer.shared("sh_up").T
                st["ys"] = layer.act(g, u) @ layer.shared("sh_down").T
            else:
                st["ys"] = 0.0
        e = int(self.routes["idx"][t, j])
        Wg = self.dequant(*self.need[("ex_gate", e)])
        Wu = self.dequant(*self.need[("ex_up", e)])
        Wd = self.dequant(*self.need[("ex_down", e)])
        h = layer.act(Wg @ st["xe"], Wu @ st["xe"])
        st["u"] += self.routes["G"][t, j] * (Wd @ h)
        if j == self.k - 1:
            if cfg.d_latent:
                uh = O.rms_norm(st["u"], layer.dense("norm_w"), cfg.norm_eps) if cfg.use_latent_norm else st["u"]
                yr = uh @ layer.dense("w_up_latent").T
            else:
                yr = st["u"]
            self.delta[t] = yr + st["ys"]


def run_reference(args):
    """The fp64 oracle as the reference arm, on the host cores (ReferenceArm):
    one step = one (token, slot) assignment, k steps = one token."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch
    from lmoe_inputs import configs as C

    wl = C.workload(args.workload)
    cfg = wl.cfg
    k = cfg.top_k
    total = args.warmup + args.steps
    arm = ReferenceArm(wl, total, dev="cuda" if torch.cuda.is_available() else "cpu")
    for s in range(args.warmup):
        arm.step(s)
    t0 = time.perf_counter()
    for s in range(args.warmup, total):
        arm.step(s)
    dt = time.perf_counter() - t0
    value = (args.steps / k) / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same seeded generator)",
        "config": {"workload": wl.name, "T": wl.T, "d_model": cfg.d_model, "d_latent": cfg.d_latent,
                   "n_experts": cfg.n_experts, "top_k": k},
        "cpu_baseline": {"kind": "oracle", "cores": os.cpu_count(), "value": round(value, 4), "unit": UNIT,
                         "sample": f"{args.steps} (token, slot) assignments = {args.steps / k:.2f} tokens "
                                   f"of {wl.name}; each step dequantises and applies one routed expert, "
                                   "slot 0 / last slot add the token's dense parts"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="k3_decode_t64")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-tokens", type=int, default=2)
    ap.add_argument("--sweep", default=None,
                    help="comma-separated token counts: one JSON line per T on one GPU (not the driver's contract)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.sweep:
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
