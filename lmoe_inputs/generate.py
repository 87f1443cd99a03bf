"""Seeded synthetic inputs for the Stable LatentMoE layer.

This is the one module that both the fp64 oracle and the CUDA library read
their inputs from.  It holds no arithmetic of the layer itself: it draws
numbers and stores them in the checkpoint formats the pages name.

Formats (Kimi K3 card, "Explanation"; NVFP4 port notes, first paragraph):
  * routed-expert weights in MXFP4: E2M1 codes, two per byte with the even K
    index in the low nibble, plus one E8M0 scale byte per 32 consecutive K
    values (K = the input dimension, the contiguous one of nn.Linear's
    [out, in] storage);
  * everything else bf16, the router's selection bias fp32;
  * Kimi K2 card, parameter table: FP8 E4M3 weights with one fp32 scale per
    128 x 128 block.

Random numbers come from a counter-based hash (Wellons' "lowbias32" 32-bit
integer mixer), so any slice of any tensor can be regenerated on any device
with identical bits: normals are read from a fixed table of 65536 N(0,1)
quantiles indexed by 16 hash bits.  Every float operation used here (one
fp32 multiply, exact power-of-two scalings, comparisons, RNE casts) is
IEEE-exact or correctly rounded, so CPU and CUDA produce the same bytes.

MXFP4 quantisation follows the OCP MX rule: shared exponent
X = floor(log2(amax_32)) - 2, element = RNE(w / 2^X) on the E2M1 grid,
saturating at +-6.  FP8: scale = amax_128x128 / 448, element =
RNE(w / scale) in E4M3, saturating.
"""
from __future__ import annotations

import math
from statistics import NormalDist

import numpy as np
import torch

from .configs import LayerConfig, Workload

_M32 = 0xFFFFFFFF
_TABLE_BITS = 16
_NORM_TABLE_CPU = None


def _norm_table(device) -> torch.Tensor:
    global _NORM_TABLE_CPU
    if _NORM_TABLE_CPU is None:
        nd = NormalDist()
        n = 1 << _TABLE_BITS
        vals = [nd.inv_cdf((i + 0.5) / n) for i in range(n)]
        _NORM_TABLE_CPU = torch.tensor(vals, dtype=torch.float64).to(torch.float32)
    return _NORM_TABLE_CPU.to(device)


def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2^32 for int64 tensors holding values in [0, 2^32),
    split into 16-bit halves of c so that no intermediate exceeds 2^49."""
    c_lo, c_hi = c & 0xFFFF, c >> 16
    return (x * c_lo + (((x * c_hi) & 0xFFFF) << 16)) & _M32


def hash32(x: torch.Tensor) -> torch.Tensor:
    """lowbias32 integer mixer on int64 tensors holding uint32 values."""
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def _hash32_int(v: int) -> int:
    return int(hash32(torch.tensor([v & _M32], dtype=torch.int64))[0])


def stream_key(seed: int, *tags: int) -> int:
    """Scalar key of one random stream: (seed, tensor tag, expert, ...)."""
    k = _hash32_int(seed * 0x9E3779B9 + 0x632BE5AB)
    for t in tags:
        k = _hash32_int(k ^ _hash32_int(t + 0x5BD1E995))
    return k


def _bits(n: int, key: int, device) -> torch.Tensor:
    idx = torch.arange(n, dtype=torch.int64, device=device)
    k2 = _hash32_int(key ^ 0x27D4EB2F)
    return hash32(hash32(idx ^ key) ^ k2)


def normal_f32(n: int, key: int, device, std: float = 1.0) -> torch.Tensor:
    """n draws of N(0, std^2) as float32 (table quantile times fp32 std)."""
    h = _bits(n, key, device)
    v = _norm_table(device)[h & ((1 << _TABLE_BITS) - 1)]
    if std != 1.0:
        v = v * torch.tensor(std, dtype=torch.float32, device=device)
    return v


def uniform_f32(n: int, key: int, device) -> torch.Tensor:
    """n draws of U[0, 1) with 24 random bits, float32."""
    h = _bits(n, key, device)
    return (h >> 8).to(torch.float32) * (1.0 / (1 << 24))


# ---------------------------------------------------------------- formats
def to_bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16)


def quantise_mxfp4(w: torch.Tensor):
    """float32 [N, K] -> (codes uint8 [N, K/2], scales uint8 [N, K/32])."""
    N, K = w.shape
    assert K % 32 == 0
    wb = w.view(N, K // 32, 32)
    amax = wb.abs().amax(-1)
    field = (amax.view(torch.int32).to(torch.int64) >> 23) & 0xFF
    sbyte = torch.where(amax > 0, (field - 2).clamp(0, 253), torch.zeros_like(field))
    # 2^(127 - sbyte) built from its bit pattern: an exact power of two.
    p2 = ((254 - sbyte) << 23).to(torch.int32).view(torch.float32)
    v = wb * p2[..., None]
    a = v.abs()
    code = torch.zeros_like(a, dtype=torch.int64)
    # Round to nearest, ties to even code, on the grid 0,.5,1,1.5,2,3,4,6.
    code = torch.where(a > 0.25, 1, code)
    code = torch.where(a >= 0.75, 2, code)
    code = torch.where(a > 1.25, 3, code)
    code = torch.where(a >= 1.75, 4, code)
    code = torch.where(a > 2.5, 5, code)
    code = torch.where(a >= 3.5, 6, code)
    code = torch.where(a > 5.0, 7, code)
    nib = code | ((v < 0).to(torch.int64) << 3)
    nib = nib.view(N, K)
    packed = (nib[:, 0::2] | (nib[:, 1::2] << 4)).to(torch.uint8)
    return packed.contiguous(), sbyte.to(torch.uint8).contiguous()


def quantise_fp8_block128(w: torch.Tensor):
    """float32 [N, K] -> (E4M3 bytes uint8 [N, K], fp32 scales [ceil(N/128), ceil(K/128)])."""
    N, K = w.shape
    nb, kb = -(-N // 128), -(-K // 128)
    pad = torch.zeros(nb * 128, kb * 128, dtype=torch.float32, device=w.device)
    pad[:N, :K] = w
    blk = pad.view(nb, 128, kb, 128)
    amax = blk.abs().amax(dim=(1, 3))
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (blk / scale[:, None, :, None]).clamp(-448.0, 448.0)
    q8 = q.to(torch.float8_e4m3fn).view(torch.uint8).view(nb * 128, kb * 128)[:N, :K]
    return q8.contiguous(), scale.contiguous()


# ---------------------------------------------------------------- tensors
# Tensor tags of the random streams.
TAG = dict(x=1, router_w=2, router_bias=3, w_down_latent=4, w_up_latent=5, norm_w=6,
           ex_gate=7, ex_up=8, ex_down=9, sh_gate=10, sh_up=11, sh_down=12, zipf_perm=13)


def _std(fan_in: int) -> float:
    return float(np.float32(1.0 / math.sqrt(fan_in)))


def gen_x(wl: Workload, device="cpu", T: int | None = None) -> torch.Tensor:
    """Tokens x ~ N(0, 1) in bf16, [T, d] (batch and positions flattened)."""
    T = wl.T if T is None else T
    d = wl.cfg.d_model
    return to_bf16(normal_f32(T * d, stream_key(wl.seed, TAG["x"]), device)).view(T, d)


def gen_router_bias(wl: Workload) -> torch.Tensor:
    """fp32 selection bias [E]: U(-0.1, 0.1), or the Zipf skew of the prefill
    workload (v_r = r^-1.1 over a seeded random permutation of the experts,
    mapped linearly so that min -> -0.5 and max -> +0.5)."""
    E = wl.cfg.n_experts
    if wl.bias == "zipf":
        r = np.arange(1, E + 1, dtype=np.float64)
        v = r ** -1.1
        h = _bits(E, stream_key(wl.seed, TAG["zipf_perm"]), "cpu").numpy()
        order = np.argsort(h, kind="stable")      # seeded permutation of experts
        b = np.empty(E, dtype=np.float64)
        b[order] = v
        b = (b - b.min()) / (b.max() - b.min()) - 0.5
        return torch.from_numpy(b.astype(np.float32))
    u = uniform_f32(E, stream_key(wl.seed, TAG["router_bias"]), "cpu")
    return (u * 0.2 - 0.1).to(torch.float32)


def gen_dense(wl: Workload, name: str, shape, fan_in: int, device="cpu") -> torch.Tensor:
    n = shape[0] * shape[1]
    w = normal_f32(n, stream_key(wl.seed, TAG[name]), device, _std(fan_in))
    return to_bf16(w).view(*shape)


def gen_expert(wl: Workload, name: str, e: int, device="cpu"):
    """One routed expert matrix in the workload's expert format.
    name in {"ex_gate", "ex_up", "ex_down"}; nn.Linear [out, in] storage."""
    cfg = wl.cfg
    din, F = cfg.d_expert_in, cfg.d_expert_ff
    N, K = (F, din) if name in ("ex_gate", "ex_up") else (din, F)
    w = normal_f32(N * K, stream_key(wl.seed, TAG[name], e), device, _std(K)).view(N, K)
    if cfg.expert_wfmt == "mxfp4":
        return quantise_mxfp4(w)
    return quantise_fp8_block128(w)


def gen_experts_mxfp4(wl: Workload, name: str, device, chunk: int = 16):
    """All experts of one MXFP4 matrix, `chunk` experts per batch of tensor
    ops: the same bytes as gen_expert one expert at a time (each expert keeps
    its own stream key), with far fewer kernel launches on a GPU."""
    cfg = wl.cfg
    din, F, E = cfg.d_expert_in, cfg.d_expert_ff, cfg.n_experts
    N, K = (F, din) if name in ("ex_gate", "ex_up") else (din, F)
    q_all = torch.empty((E, N, K // 2), dtype=torch.uint8, device=device)
    s_all = torch.empty((E, N, K // 32), dtype=torch.uint8, device=device)
    std = torch.tensor(_std(K), dtype=torch.float32, device=device)
    idx = torch.arange(N * K, dtype=torch.int64, device=device)
    table = _norm_table(device)
    for e0 in range(0, E, chunk):
        es = range(e0, min(E, e0 + chunk))
        keys = [stream_key(wl.seed, TAG[name], e) for e in es]
        k1 = torch.tensor(keys, dtype=torch.int64, device=device)[:, None]
        k2 = torch.tensor([_hash32_int(k ^ 0x27D4EB2F) for k in keys], dtype=torch.int64, device=device)[:, None]
        h = hash32(hash32(idx[None, :] ^ k1) ^ k2)
        w = (table[h & ((1 << _TABLE_BITS) - 1)] * std).view(len(es) * N, K)
        q, s = quantise_mxfp4(w)
        q_all[e0:e0 + len(es)] = q.view(len(es), N, K // 2)
        s_all[e0:e0 + len(es)] = s.view(len(es), N, K // 32)
        del h, w, q, s
    return q_all, s_all


def gen_shared_fp8(wl: Workload, name: str, device="cpu"):
    cfg = wl.cfg
    d, Fs = cfg.d_model, cfg.d_shared_ff
    N, K = (Fs, d) if name in ("sh_gate", "sh_up") else (d, Fs)
    w = normal_f32(N * K, stream_key(wl.seed, TAG[name]), device, _std(K)).view(N, K)
    return quantise_fp8_block128(w)


def gen_dense_weights(wl: Workload, device="cpu") -> dict:
    """The layer's non-expert weights on `device`: router, latent
    projections and norm, shared MLP (bf16, or FP8 block-128 for the FP8
    layer format)."""
    cfg = wl.cfg
    d, l, E, Fs = cfg.d_model, cfg.d_latent, cfg.n_experts, cfg.d_shared_ff
    W = {}
    W["router_w"] = gen_dense(wl, "router_w", (E, d), d, device)
    W["router_bias"] = gen_router_bias(wl).to(device)
    if l:
        W["w_down_latent"] = gen_dense(wl, "w_down_latent", (l, d), d, device)
        W["w_up_latent"] = gen_dense(wl, "w_up_latent", (d, l), l, device)
        if cfg.use_latent_norm:
            nw = 1.0 + normal_f32(l, stream_key(wl.seed, TAG["norm_w"]), "cpu", 0.02)
            W["norm_w"] = to_bf16(nw).to(device)
    if Fs:
        if cfg.expert_wfmt == "mxfp4":
            W["sh_gate"] = gen_dense(wl, "sh_gate", (Fs, d), d, device)
            W["sh_up"] = gen_dense(wl, "sh_up", (Fs, d), d, device)
            W["sh_down"] = gen_dense(wl, "sh_down", (d, Fs), Fs, device)
        else:
            for name in ("sh_gate", "sh_up", "sh_down"):
                W[name], W[name + "_s"] = gen_shared_fp8(wl, name, device)
    return W


def gen_weights(wl: Workload, device="cpu") -> dict:
    """All layer weights on `device`.  Keys mirror the C-ABI weight struct."""
    cfg = wl.cfg
    E = cfg.n_experts
    W = gen_dense_weights(wl, device)
    for name in ("ex_gate", "ex_up", "ex_down"):
        if device != "cpu" and cfg.expert_wfmt == "mxfp4":
            W[name + "_q"], W[name + "_s"] = gen_experts_mxfp4(wl, name, device)
            continue
        for e in range(E):
            q, s = gen_expert(wl, name, e, device)
            if e == 0:
                W[name + "_q"] = torch.empty((E,) + tuple(q.shape), dtype=q.dtype, device=device)
                W[name + "_s"] = torch.empty((E,) + tuple(s.shape), dtype=s.dtype, device=device)
            W[name + "_q"][e] = q
            W[name + "_s"][e] = s
    return W


def gen_inputs(wl: Workload, device="cpu") -> dict:
    out = gen_weights(wl, device)
    out["x"] = gen_x(wl, device)
    return out
