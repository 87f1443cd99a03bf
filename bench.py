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

Prints one JSON line: metric/value (device-timed tokens/s of the headline
workload, Kimi-K3 shapes at T = 64), e2e (through lmoe_forward_host with
host buffers and the copies inside the timed region), roofline of the
dominant kernel (the grouped gate/up expert GEMM: algorithmic bytes over its
CUDA-event time against the HBM peak, or its executed MMA FLOPs against the
measured rate of the same MMA form above the ridge), the whole layer's
roofline fraction (max of the HBM time and the FP4 + bf16 tensor time over
the step time), per-stage times, the tensor-pipe peaks measured in the same
run, clocks sampled during the timed region, the fp64 oracle timed on the
host cores as cpu_baseline, and per_config: the same measurements for the
token-count sweep (T = 1 .. 2048, seed 4), the Zipf-skewed prefill batch
(T = 8192) and the Kimi-K2 block (T = 4096), each with its own clocks.
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
# Coprime with the 4 rotating token batches, so the sampled forwards cycle
# through all of them.
PROFILE_PERIOD = 7
METRIC = "LatentMoE layer tokens/s at T=1..8192; % of HBM or FP4-TC roofline"
UNIT = "tokens/s"
# DRAM bytes (read + write) per algorithmic byte of the gate/up expert
# kernel of each weight format, from one ncu capture of the kernel as it
# stands on a small case of the same instantiation (K3 shapes with 64
# experts at T = 8: 702.2 MB for 645.2 MB; at T = 1024, the prefill tile:
# 997.0 MB for 974 MB; K2 shapes with 32 experts at T = 384: 1033.2 MB for
# 998.1 MB), keyed by (weight format, token tile, K-split form).  The K-split
# form of one to a few tokens (K3 shapes with 64 experts at T = 1: 260.9 MB
# for 187.4 MB) also prefetches 64 MiB of the batch's down weights into L2
# for the down pass, which its DRAM bytes include.  An entry is removed when
# its kernel changes until it is captured again.
GU_DRAM_PER_ALGO_BYTE = {("mxfp4", 16, False): 1.088, ("mxfp4", 16, True): 1.392, ("mxfp4", 96, False): 1.024,
                         ("fp8_block128", 96, False): 1.035}
KSPLIT_MAX_P = 1024   # largest batch (assignments) the library considers for the K-split form


def expert_tile(cfg, T: int) -> int:
    """Token tile the library picks for the grouped expert GEMMs (the rule of
    moe_tile_tokens / fp8_tile_tokens in the library's internal header)."""
    P, E = T * cfg.top_k, cfg.n_experts
    if cfg.expert_wfmt == "mxfp4":
        return 16 if P <= 4 * E else 32 if P <= 16 * E else 64 if P <= 64 * E else 96
    m = -(-P // E)
    return 16 if m <= 16 else 32 if m <= 32 else 64 if m <= 64 else 96


def gate_up_ksplit(cfg, T: int, num_sms: int = 152) -> bool:
    """Whether the library runs the gate/up pass in its K-split form (the rule
    of expert_ksplit in the library: MXFP4 weights, the 16-assignment tile and
    fewer than two 256-row weight items per SM)."""
    P, E = T * cfg.top_k, cfg.n_experts
    if cfg.expert_wfmt != "mxfp4" or P > KSPLIT_MAX_P or expert_tile(cfg, T) != 16:
        return False
    tiles = min(P, P // 16 + min(E, P))
    return tiles * -(-cfg.d_expert_ff // 256) < 2 * num_sms


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
    # E4M3 activation terms (hi + lo, or one) with one E8M0 each per 32 in, the same for h
    t = getattr(cfg, "act_terms", 2)
    nb = 0.5 if getattr(cfg, "act_format", "e4m3") == "e2m1" else 1.0     # bytes per code
    act_in = int(t * din * nb) + t * din // 32
    h_io = int(t * F * nb) + t * F // 32
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


def cpu_baseline(wl, W_dev, x_dev, budget_s: float = 10.0) -> dict:
    """The fp64 oracle, as it stands, one token at a time on the first tokens
    of a batch (its routing, k fresh expert dequantisations, dense parts)
    until `budget_s` of CPU time has passed."""
    import numpy as np
    import torch
    O, Wn = oracle_for(wl, W_dev)
    layer = O.Layer(wl.cfg, Wn, cache_experts=False)
    for name in ("router_w", "w_down_latent", "w_up_latent", "norm_w"):
        if name in Wn:
            layer.dense(name)        # host-side fp64 copies of the dense weights: input preparation
    for name in ("sh_gate", "sh_up", "sh_down"):
        if name in Wn:
            layer.shared(name)
    xb = x_dev.cpu().view(torch.int16).numpy().view(np.uint16)
    t0 = time.perf_counter()
    n = 0
    while n < xb.shape[0] and (n == 0 or time.perf_counter() - t0 < budget_s):
        O.forward(layer, xb[n:n + 1])
        n += 1
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} tokens of the {wl.name} batch, one oracle forward each (routing, "
                      f"{wl.cfg.top_k} expert dequantisations per token, dense parts); numpy BLAS threads = default",
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


def sampled_forwards(steps: int, period: int = PROFILE_PERIOD) -> list:
    """Indices of the timed forwards whose expert kernels carry events."""
    return list(range(0, steps, period))


# ------------------------------------------------------------ tensor peaks
def tensor_peaks(iters: int = 150000) -> dict:
    """Measured tensor-pipe rates (TFLOP/s, best of three) of the MMA forms,
    from the library's own tcgen05 loop (include/lmoe_peak.h)."""
    from latent_mixture_experts_gb300 import binding
    return {k: round(max(binding.tc_peak(k, iters) for _ in range(3)), 1) for k in binding.TC_KINDS}


def mma_per_flop(cfg, T: int) -> int:
    """MMA FLOPs the routed expert GEMMs execute per layer FLOP: one per
    activation term on the split (large-batch) tiles and on the packed-FP4
    kernel; the interleaved (small-batch) E4M3 tiles always multiply a hi and
    a lo column."""
    if getattr(cfg, "act_format", "e4m3") == "e2m1":
        return getattr(cfg, "act_terms", 3)
    split = cfg.expert_wfmt != "mxfp4" or expert_tile(cfg, T) >= 64
    return getattr(cfg, "act_terms", 2) if split else 2


def rooflines(cfg, T: int, U: float, ms: float, pk: dict, tc: dict | None) -> dict:
    """The layer's roofline time for T tokens selecting U distinct experts:
    max(bytes / HBM, routed FLOPs / FP4 peak + dense FLOPs / bf16 peak), and
    the measured step's fraction of it; plus the fraction of the pipe the
    kernels actually issue on (the routed MMAs run E2M1 or E4M3 weights
    against two E4M3 activation terms on kind::mxf8f6f4)."""
    A = accounting(cfg)
    bytes_ = A["dense"] + U * A["expert"] + T * A["token_io"]
    din = A["din"]
    f_routed = T * cfg.top_k * 6 * cfg.d_expert_ff * din
    f_dense = T * A["flops_per_token"] - f_routed
    t_hbm = bytes_ / (pk["hbm"] * 1e9) * 1e3
    out = {"bytes": int(bytes_), "hbm_gbs": round(bytes_ / (ms * 1e-3) / 1e9, 1),
           "hbm_frac": round(t_hbm / ms, 4), "tflops": round(T * A["flops_per_token"] / (ms * 1e-3) / 1e12, 1)}
    if tc:
        fp4 = tc["mxfp4"] if cfg.expert_wfmt == "mxfp4" else tc["e4m3_e4m3"]
        issued = (tc["mxfp4"] if getattr(cfg, "act_format", "e4m3") == "e2m1" else
                  tc["e2m1_e4m3"] if cfg.expert_wfmt == "mxfp4" else tc["e4m3_e4m3"])
        t_tensor = (f_routed / (fp4 * 1e12) + f_dense / (tc["bf16"] * 1e12)) * 1e3
        t_issued = (mma_per_flop(cfg, T) * f_routed / (issued * 1e12) + f_dense / (tc["bf16"] * 1e12)) * 1e3
        out.update({"tensor_floor_ms": round(t_tensor, 4), "roofline_ms": round(max(t_hbm, t_tensor), 4),
                    "frac": round(max(t_hbm, t_tensor) / ms, 4),
                    "bound": "hbm" if t_hbm >= t_tensor else "tensor",
                    "issued_pipe_frac": round(t_issued / ms, 4),
                    "routed_peak": ("mxfp4" if cfg.expert_wfmt == "mxfp4" else "e4m3_e4m3") + " (measured)"})
    else:
        out.update({"frac": round(t_hbm / ms, 4), "bound": "hbm"})
    return out


def gate_up_roofline(cfg, T: int, U: float, gu_ms: float, pk: dict, tc: dict | None) -> dict:
    """The dominant kernel, the grouped gate/up expert GEMM: its algorithmic
    bytes (the selected experts' gate and up weights, the hi/lo activations
    in, the hi/lo h out) over its CUDA-event time against the HBM peak, or,
    above the ridge, its executed MMA FLOPs (two per layer FLOP: the hi and lo
    activation terms) against the measured peak of the form it issues."""
    A = accounting(cfg)
    fp4 = cfg.expert_wfmt == "mxfp4"
    k = cfg.top_k
    gu_bytes = U * A["gu_w"] + T * k * A["gu_per_assign"]
    gu_flops = 2.0 * T * k * 2 * cfg.d_expert_ff * A["din"]
    e2m1 = getattr(cfg, "act_format", "e4m3") == "e2m1"
    issued = (tc or {}).get("mxfp4" if e2m1 else "e2m1_e4m3" if fp4 else "e4m3_e4m3")
    peak_t = issued if issued else 2.0 * pk["bf16"]
    achieved_gbs = gu_bytes / (gu_ms * 1e-3) / 1e9
    mf = mma_per_flop(cfg, T)
    tensor = gu_flops / gu_bytes > 1e3 * peak_t / mf / pk["hbm"]
    terms = "hi/lo" if getattr(cfg, "act_terms", 2) == 2 else "one term (MXFP8)"
    name = (f"moe_fp4_kernel<gate/up> (grouped MXFP4 x {getattr(cfg, 'act_terms', 3)} MXFP4 terms, packed, "
            "tcgen05 kind::mxf4)" if e2m1 else
            f"moe_gemm_kernel<gate/up> (grouped MXFP4 x E4M3 {terms}, tcgen05)" if fp4 else
            "moe_fp8_kernel<gate/up> (grouped E4M3 x E4M3 hi/lo, block-128 promotion, tcgen05)")
    r = {"kernel": name, "bytes_per_launch": int(gu_bytes), "ms_per_launch": round(gu_ms, 5)}
    if tensor:
        ach = mf * gu_flops / (gu_ms * 1e-3) / 1e12
        r.update({"bound": "tensor", "achieved": round(ach, 1), "peak": round(peak_t, 1), "unit": "TFLOP/s",
                  "frac": round(ach / peak_t, 4), "hbm_gbs": round(achieved_gbs, 1),
                  "flops_note": f"executed MMA FLOPs ({mf} per layer FLOP: one per activation term)",
                  "peak_source": ("measured tcgen05 loop of the same MMA form" if issued else
                                  "fallback: MEASURED_PEAKS.json bf16_tflops x 2")})
    else:
        r.update({"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": pk["hbm"], "unit": "GB/s",
                  "frac": round(achieved_gbs / pk["hbm"], 4),
                  "peak_source": f"{pk['src']} (MEASURED_PEAKS.json hbm_gbs)"})
    tr = None if e2m1 else GU_DRAM_PER_ALGO_BYTE.get((cfg.expert_wfmt, expert_tile(cfg, T), gate_up_ksplit(cfg, T)))
    r["traffic"] = int(tr * gu_bytes) if tr else None
    r["traffic_source"] = ("ncu dram__bytes_read+write of this kernel on a small case of the same instantiation, "
                           "scaled to this launch by its algorithmic bytes" if tr else
                           "no ncu capture of this instantiation as it stands")
    return r


def time_forwards(layer, xs, out, steps: int, stream, world: int = 1):
    """K forwards over the rotating batches between CUDA events on the
    stream, the expert kernels of every PROFILE_PERIOD-th forward carrying
    their own events; clocks sampled meanwhile.  Returns (ms, clocks,
    profile)."""
    import torch
    import torch.distributed as dist
    layer.lmoe_set_profiling(steps, stages=["expert_gate_up", "expert_down"])
    layer.lmoe_set_profiling_period(PROFILE_PERIOD)
    clk = ClockSampler(None)
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_start = time.time()
    e0.record(stream)
    for i in range(steps):
        layer.lmoe_forward(xs[i % len(xs)], out=out)
    e1.record(stream)
    torch.cuda.synchronize()
    t_end = time.time()
    if world > 1:
        dist.barrier()
    clocks = clk.stop(t_start, t_end)
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    prof = layer.lmoe_profile_get()
    layer.lmoe_set_profiling_period(1)
    layer.lmoe_set_profiling(0)
    return ms, clocks, prof


def stage_pass(layer, xs, out, n: int) -> dict:
    """Per-stage averages from a separate pass with every stage timed."""
    layer.lmoe_set_profiling_period(1)
    layer.lmoe_set_profiling(n)
    for i in range(n):
        layer.lmoe_forward(xs[i % len(xs)], out=out)
    sp = layer.lmoe_profile_get()
    layer.lmoe_set_profiling(0)
    return {name: round(v[0] / max(v[1], 1), 5) for name, v in sp.items()}


def active_experts(layer, xs, out) -> list:
    U = []
    for xb in xs:
        layer.lmoe_forward(xb, out=out)
        U.append(layer.lmoe_last_active_experts())
    return U


def measure_config(wl, layer, xs, out, steps_min: int, warmup: int, pk: dict, tc: dict | None,
                   target_s: float = 0.3, max_steps: int = 4000) -> dict:
    """One entry of the per-configuration block: tokens/s over a timed region
    of about target_s (at least steps_min forwards), the layer's roofline
    fraction, the dominant kernel's roofline, clocks."""
    import torch
    cfg, T = wl.cfg, xs[0].shape[0]
    U = active_experts(layer, xs, out)
    for i in range(warmup):
        layer.lmoe_forward(xs[i % len(xs)], out=out)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(3):
        layer.lmoe_forward(xs[i % len(xs)], out=out)
    torch.cuda.synchronize()
    est = (time.perf_counter() - t0) / 3
    steps = int(min(max_steps, max(steps_min, target_s / max(est, 1e-6))))
    stream = torch.cuda.current_stream()
    ms, clocks, prof = time_forwards(layer, xs, out, steps, stream)
    ms_step = ms / steps
    samp = sampled_forwards(steps)
    U_s = sum(U[i % len(xs)] for i in samp) / len(samp)
    U_all = sum(U[i % len(xs)] for i in range(steps)) / steps
    gu_ms, gu_n = prof["expert_gate_up"]
    return {"workload": wl.name, "T": T, "steps": steps, "tokens_per_s": round(T / (ms_step * 1e-3), 1),
            "ms_per_step": round(ms_step, 5), "active_experts_mean": round(U_all, 1),
            "layer_roofline": rooflines(cfg, T, U_all, ms_step, pk, tc),
            "roofline": {**gate_up_roofline(cfg, T, U_s, gu_ms / max(gu_n, 1), pk, tc), "launches_timed": int(gu_n)},
            "clocks": clocks}


# ------------------------------------------------------------------ ours
# Configurations measured beside the headline one, one GPU: the token-count
# sweep (seed 4), the Zipf-skewed prefill batch (two activation terms, and
# one: MXFP8) and the Kimi-K2 block.
PER_CONFIG = (("k3_sweep", (1, 8, 32, 128, 512, 2048)), ("k3_prefill_t8192", None),
              ("k3_prefill_t8192_mxfp8", None), ("k2_t4096", None))


def expert_dtype(cfg) -> str:
    """The operand types of the routed-expert MMAs."""
    if cfg.expert_wfmt != "mxfp4":
        return "e4m3 x e4m3(hi+lo), fp32 block-128 scales" if cfg.act_terms == 2 else "e4m3 x e4m3, fp32 block-128 scales"
    if getattr(cfg, "act_format", "e4m3") == "e2m1":
        return f"e2m1 x e2m1 ({cfg.act_terms} mxfp4 terms) block-scaled"
    return "e2m1 x e4m3(hi+lo) block-scaled" if cfg.act_terms == 2 else "e2m1 x e4m3 (mxfp8) block-scaled"


def run_per_config(args, pk, tc, budget_s: float = 240.0) -> list:
    import torch
    from lmoe_inputs import configs as C
    from lmoe_inputs import generate as G
    from latent_mixture_experts_gb300 import LatentMoE
    entries = []
    t_start = time.time()
    for name, Ts in PER_CONFIG:
        if time.time() - t_start > budget_s:
            entries.append({"workload": name, "skipped": "time budget of the per-configuration block spent"})
            continue
        wl = C.workload(f"k3_sweep_t{max(Ts)}" if Ts else name)
        W = G.gen_weights(wl, device="cuda")
        layer = LatentMoE(wl.cfg, W, max_tokens=wl.T)
        try:
            for T in (Ts or (wl.T,)):
                wlT = replace(wl, T=T, name=f"k3_sweep_t{T}") if Ts else wl
                xs = [G.gen_x(replace(wlT, seed=sd), device="cuda") for sd in replica_seeds(wlT, 0)]
                out = torch.empty(T, wl.cfg.d_model, dtype=torch.bfloat16, device="cuda")
                entries.append(measure_config(wlT, layer, xs, out, args.steps, args.warmup, pk, tc))
            layer.lmoe_sync_status()
        finally:
            layer.close()
            del W
            torch.cuda.empty_cache()
    return entries


def with_activation_format(wl, args):
    """The workload with the command line's activation format / terms / token
    count, if given."""
    if getattr(args, "T", None):
        wl = replace(wl, T=args.T, name=f"{wl.name}_T{args.T}")
    over = {}
    if getattr(args, "act_format", None):
        over["act_format"] = args.act_format
    if getattr(args, "act_terms", None):
        over["act_terms"] = args.act_terms
    if not over:
        return wl
    tag = "_".join(f"{k}{v}" for k, v in over.items())
    return replace(wl, cfg=replace(wl.cfg, **over), name=f"{wl.name}_{tag}")


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
    pk = peaks()
    tc = None if args.no_tc_peaks else tensor_peaks()
    wl = with_activation_format(C.workload(args.workload), args)
    T, cfg = wl.T, wl.cfg
    W = G.gen_weights(wl, device="cuda")
    xs = [G.gen_x(replace(wl, seed=sd), device="cuda") for sd in replica_seeds(wl, rank)]
    out = torch.empty(T, cfg.d_model, dtype=torch.bfloat16, device="cuda")
    layer = LatentMoE(cfg, W, max_tokens=T)
    stream = torch.cuda.current_stream()

    # distinct experts each batch selects (units of the expert bytes)
    U = active_experts(layer, xs, out)
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
    ms, clocks, prof = time_forwards(layer, xs, out, args.steps, stream, world)
    stages = stage_pass(layer, xs, out, min(args.steps, 100))
    layer.lmoe_sync_status()

    steps = args.steps
    ms_step = ms / steps
    value = job_throughput(world, T, steps, ms / 1e3)
    U_mean = sum(U[i % 4] for i in range(steps)) / steps
    samp = sampled_forwards(steps)
    U_samp = sum(U[i % 4] for i in samp) / len(samp)      # batches whose kernel times were taken
    gu_ms, gu_n = prof["expert_gate_up"]
    dn_ms, dn_n = prof["expert_down"]
    A = accounting(cfg)
    dn_bytes = U_samp * A["dn_w"] + T * cfg.top_k * A["dn_per_assign"]
    fp4 = cfg.expert_wfmt == "mxfp4"
    roof = gate_up_roofline(cfg, T, U_samp, gu_ms / max(gu_n, 1), pk, tc)
    roof.update({"launches_timed": int(gu_n), "sampled_batches": sorted({i % 4 for i in samp}),
                 "timing": f"CUDA events on the launch stream around every {PROFILE_PERIOD}th timed forward's "
                           f"launch (forwards {samp[:6]}{'...' if len(samp) > 6 else ''}); bytes from the "
                           "distinct experts of the batches those forwards ran"})

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
        cpu = cpu_baseline(wl, W, xs[0])
    layer.close()
    del W
    torch.cuda.empty_cache()
    per_config = None
    if world == 1 and not args.no_per_config:
        per_config = run_per_config(args, pk, tc)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": expert_dtype(cfg) + "; bf16 dense; fp32 accumulate",
        "data": "synthetic (seeded, N(0,1/fan_in) weights quantised to "
                + ("MXFP4" if fp4 else "FP8 E4M3 block-128") + "; x ~ N(0,1) bf16)",
        "config": {"workload": wl.name, "T": T, "d_model": cfg.d_model, "d_latent": cfg.d_latent, "n_experts": cfg.n_experts,
                   "top_k": cfg.top_k, "d_expert_ff": cfg.d_expert_ff, "d_shared_ff": cfg.d_shared_ff,
                   "expert_format": cfg.expert_wfmt,
                   "parallelism": f"replicas x{world}", "token_batches_rotated": 4,
                   "l2": "no flush: each step streams the selected experts' weights (GBs) >> 129 MB L2",
                   "active_experts_mean": round(U_mean, 1)},
        "roofline": roof,
        "layer_roofline": rooflines(cfg, T, U_mean, ms_step, pk, tc),
        "down_kernel": {"achieved": round(dn_bytes / (dn_ms / max(dn_n, 1) * 1e-3) / 1e9, 1), "unit": "GB/s",
                        "ms_per_launch": round(dn_ms / max(dn_n, 1), 5)},
        "stage_ms": stages,
        "stage_ms_source": f"separate pass of {min(steps, 100)} forwards with every stage timed (outside the timed region)",
        "tensor_peaks_tflops": tc,
        "tensor_peaks_source": "measured in this run: tcgen05 loop, one CTA per SM, M=128 N=256, best of 3",
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": launches * steps,
        "cpu_baseline": cpu,
        "per_config": per_config,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


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
    ap.add_argument("--no-per-config", action="store_true", help="headline workload only")
    ap.add_argument("--no-tc-peaks", action="store_true", help="skip the tensor-pipe peak measurement")
    ap.add_argument("--act-format", choices=["e4m3", "e2m1"], default=None,
                    help="routed-expert activation format (default: the workload's)")
    ap.add_argument("--act-terms", type=int, default=None, help="activation terms (default: the workload's)")
    ap.add_argument("--T", type=int, default=None, help="token count (default: the workload's)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
