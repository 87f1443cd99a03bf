"""Layer shapes and seeded workloads for the Stable LatentMoE feed-forward layer.

Shapes follow the pages:
  * Kimi K3 "Latent mixture of experts" card, equations and parameter table:
    d = 7168, latent l = 3584, 896 routed experts, top-16, routed SiTU-GLU
    3584 -> 3072 -> 3584, shared SiTU-GLU 7168 -> 6144 -> 7168 (two 3072-wide
    shared experts merged into one MLP, as the code's ``KimiMLP`` does).
  * Kimi K2 "Mixture of experts" card: 384 routed experts, top-8, routed scale
    2.827, SwiGLU 7168 -> 2048 -> 7168, one shared expert.
  * Stable LatentMoE tutorial chapter: the small reproduction, 64 experts,
    top-2, 640 -> 320 latent.

This module holds shapes, seeds and distribution names only; it computes
nothing of the layer.
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class LayerConfig:
    d_model: int
    d_latent: int          # 0 = non-latent block (K2): experts run on the full width
    n_experts: int
    top_k: int
    d_expert_ff: int
    d_shared_ff: int       # 0 = no shared expert
    use_latent_norm: bool = True
    norm_eps: float = 1e-6
    routed_scale: float = 1.0
    situ_beta: float = 4.0
    situ_linear_beta: float = 25.0
    act: str = "situ"              # "situ" | "swiglu"
    expert_wfmt: str = "mxfp4"     # "mxfp4" | "fp8_block128"
    act_terms: int = 2             # activation terms per routed-expert input on the GPU (E4M3: 1 = MXFP8)
    act_format: str = "e4m3"       # "e4m3" (E4M3 terms) | "e2m1" (packed MXFP4 terms, 4-bit x 4-bit MMAs)

    @property
    def d_expert_in(self) -> int:
        """Width the routed experts work at (the latent, or d for K2)."""
        return self.d_latent if self.d_latent else self.d_model


@dataclass(frozen=True)
class Workload:
    name: str
    cfg: LayerConfig
    T: int
    seed: int
    bias: str = "uniform"          # "uniform" U(-0.1, 0.1) | "zipf"


K3 = LayerConfig(d_model=7168, d_latent=3584, n_experts=896, top_k=16,
                 d_expert_ff=3072, d_shared_ff=6144)
K3_TINY = LayerConfig(d_model=640, d_latent=320, n_experts=64, top_k=2,
                      d_expert_ff=256, d_shared_ff=512)
K2 = LayerConfig(d_model=7168, d_latent=0, n_experts=384, top_k=8,
                 d_expert_ff=2048, d_shared_ff=2048, use_latent_norm=False,
                 routed_scale=2.827, act="swiglu", expert_wfmt="fp8_block128")

# A mid-size latent layer used only by the parity tests: every GEMM spans
# several 128-row tiles and ends on a ragged tail, and T is not a multiple of
# any token tile.
K3_MID = LayerConfig(d_model=1152, d_latent=704, n_experts=160, top_k=6,
                     d_expert_ff=608, d_shared_ff=864)

WORKLOADS = {
    "k3_tiny_t16": Workload("k3_tiny_t16", K3_TINY, T=16, seed=0),
    "k3_decode_t64": Workload("k3_decode_t64", K3, T=64, seed=1),
    "k3_prefill_t8192": Workload("k3_prefill_t8192", K3, T=8192, seed=2, bias="zipf"),
    "k2_t4096": Workload("k2_t4096", K2, T=4096, seed=3),
}
# Kimi-K3 shapes with 64 experts (1.1 GB of expert weights): the small case
# for detailed profiler captures of the same kernels.
WORKLOADS["k3_e64_t8"] = Workload("k3_e64_t8", replace(K3, n_experts=64), T=8, seed=6)
# The same 64 experts at T = 1024 (256 assignments per expert): the prefill
# token tile (96) on a case small enough for a full profiler capture.
WORKLOADS["k3_e64_t1024"] = Workload("k3_e64_t1024", replace(K3, n_experts=64), T=1024, seed=7)
# Kimi-K2 shapes with 32 experts (1.4 GB of FP8 expert weights) and 96
# assignments per expert, near the 85 of the K2 T = 4096 batch.
WORKLOADS["k2_e32_t384"] = Workload("k2_e32_t384", replace(K2, n_experts=32), T=384, seed=8)
# The prefill batch with one E4M3 term per routed-expert activation (MXFP8,
# the walk-through's deployment precision): same weights and tokens.
WORKLOADS["k3_prefill_t8192_mxfp8"] = Workload("k3_prefill_t8192_mxfp8", replace(K3, act_terms=1), T=8192, seed=2,
                                               bias="zipf")
SWEEP_T = (1, 8, 32, 128, 512, 2048)
for _t in SWEEP_T:
    WORKLOADS[f"k3_sweep_t{_t}"] = Workload(f"k3_sweep_t{_t}", K3, T=_t, seed=4)


def workload(name: str, **overrides) -> Workload:
    w = WORKLOADS[name]
    return replace(w, **overrides) if overrides else w


def param_counts(cfg: LayerConfig) -> dict:
    """Learned parameters per layer instance, counted from the tensor shapes
    this project generates (quantisation scales excluded, as the pages do)."""
    d, l, E, F, Fs = cfg.d_model, cfg.d_latent, cfg.n_experts, cfg.d_expert_ff, cfg.d_shared_ff
    din = cfg.d_expert_in
    out = {
        "router": E * d + E,                      # weight [E, d] + fp32 selection bias [E]
        "routed_expert": 3 * din * F,             # gate, up [F, din]; down [din, F]
        "shared": 3 * d * Fs if Fs else 0,
    }
    if l:
        out["latent_down"] = d * l
        out["latent_up"] = l * d
        out["latent_norm"] = l if cfg.use_latent_norm else 0
    total = out["router"] + E * out["routed_expert"] + out["shared"]
    total += out.get("latent_down", 0) + out.get("latent_up", 0) + out.get("latent_norm", 0)
    out["total"] = total
    return out
