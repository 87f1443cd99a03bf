"""fp64 CPU oracle of the Stable LatentMoE feed-forward layer (forward pass).

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The CUDA library never calls it and shares no code with it; the two
meet only in the seeded input bytes of ``lmoe_inputs``.

What it computes, step by step in the pages' order and notation
(Kimi K3 card "Latent mixture of experts", equations under "All 23 steps",
and the ``KimiSparseMoeBlock.forward`` / ``moe_infer`` excerpt of
modeling_kimi_linear.py; Kimi K2 card "Mixture of experts", "All 19 steps"):

  router      z = x W_r,  s = sigma(z),  E_sel = top_k(s + b),
              G_i = scale * s_i E_sel_i / sum_j s_j E_sel_j
  latent down x^c = x W_down                          (K3 only)
  expert i    g = x^c W_gate, u = x^c W_up, h = SiTU(g, u), E_i = h W_down
  sum         u = sum_i G_i E_i                        (in the latent for K3)
  norm        u_hat = RMSNorm(u)                       (K3, before the up-projection)
  latent up   y_routed = u_hat W_up                    (K3 only)
  shared      y_shared = SiTU-GLU(x) (full width)      (SwiGLU for K2)
  output      Delta = y_routed + y_shared              (no residual inside the layer)

Everything runs in float64 on weights dequantised exactly from their stored
formats.  numpy's matmul serves as the one library primitive.

Readings of points the pages leave open:
  * top-k ties go to the lower expert index; a token whose k-th and
    (k+1)-th biased scores differ by less than 1e-6 is flagged, and either
    choice there is correct;
  * no epsilon in the renormalisation (every sigma > 0);
  * RMSNorm(u) = w * u / sqrt(mean(u^2) + eps), eps from the config;
  * SiTU: beta_1 = 4 caps the gate's linear factor, beta_2 = 25 caps the
    up branch, gate = first projection, up = second;
  * MXFP4 nibble order: the even K index sits in the low nibble;
  * FP8 blocks are 128 (out) x 128 (in), w = e4m3(q) * scale.
"""
from __future__ import annotations

import numpy as np

TIE_EPS = 1e-6


# ------------------------------------------------------------------ formats
def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 stored as uint16 bit patterns -> float64 (exact)."""
    b = np.asarray(bits).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def e2m1_value(nib: np.ndarray) -> np.ndarray:
    """E2M1 (OCP MX FP4): 1 sign, 2 exponent (bias 1), 1 mantissa bit.
    exponent 0 is subnormal: 0.5 * m; otherwise 2^(e-1) * (1 + m/2)."""
    nib = np.asarray(nib).astype(np.int64)
    sign = np.where(nib & 0x8, -1.0, 1.0)
    e = (nib >> 1) & 0x3
    m = (nib & 0x1).astype(np.float64)
    mag = np.where(e == 0, 0.5 * m, np.exp2(e.astype(np.float64) - 1.0) * (1.0 + 0.5 * m))
    return sign * mag


def e8m0_value(s: np.ndarray) -> np.ndarray:
    """E8M0 scale byte -> 2^(s - 127).  (0xFF is NaN in the format and is
    never produced by the input generator.)"""
    return np.exp2(np.asarray(s).astype(np.float64) - 127.0)


# Every value the two formats can hold, from the closed forms above: a code
# is dequantised by looking its value up (the same numbers, without
# re-evaluating the formula for each of a matrix's millions of codes).
E2M1_VALUES = e2m1_value(np.arange(16))
E8M0_VALUES = e8m0_value(np.arange(256))


def dequant_mxfp4(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """codes uint8 [N, K/2] (even K in the low nibble) and E8M0 scales
    uint8 [N, K/32] -> float64 [N, K]: w = e2m1(code) * 2^(scale - 127)
    for the 32 consecutive K values each scale covers."""
    q = np.asarray(q)
    N, Kh = q.shape
    K = 2 * Kh
    nib = np.stack([q & 0x0F, q >> 4], axis=-1).reshape(N, K)   # even K index = low nibble
    nb = -(-K // 32)
    w = np.zeros((N, nb * 32), dtype=np.float64)
    w[:, :K] = E2M1_VALUES[nib]
    w = w.reshape(N, nb, 32) * E8M0_VALUES[np.asarray(s)[:, :nb]][:, :, None]
    return w.reshape(N, nb * 32)[:, :K]


def e4m3_value(b: np.ndarray) -> np.ndarray:
    """OCP FP8 E4M3 (fn variant): 1 sign, 4 exponent (bias 7), 3 mantissa;
    exponent 0 is subnormal m/8 * 2^-6; S.1111.111 is NaN."""
    b = np.asarray(b).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, np.exp2(e.astype(np.float64) - 7.0) * (1.0 + m / 8.0))
    mag = np.where((e == 15) & ((b & 7) == 7), np.nan, mag)
    return sign * mag


E4M3_VALUES = e4m3_value(np.arange(256))


def dequant_fp8_block128(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """E4M3 bytes [N, K] and fp32 scales [ceil(N/128), ceil(K/128)] -> float64:
    w = e4m3(q) * scale of the 128 x 128 block holding (n, k)."""
    q = np.asarray(q)
    N, K = q.shape
    scale = np.repeat(np.repeat(np.asarray(s, dtype=np.float64), 128, 0), 128, 1)[:N, :K]
    return E4M3_VALUES[q] * scale


# ------------------------------------------- block-scaled FP8 activations
# The deployment precision of the routed experts' activations is MXFP8
# (walk-through "Kimi K3 模型结构（5）", section "参数账": weights MXFP4,
# activations MXFP8): E4M3 elements, one E8M0 scale per 32 consecutive
# values along the contraction.  The emulation below quantises as the
# library does, so that its one-term (MXFP8) and two-term (E4M3 hi + lo)
# activation modes can be checked at the layer tolerance.
E4M3_MAX = 448.0


def e4m3_round(y: np.ndarray) -> np.ndarray:
    """Round to the nearest E4M3 value, ties to even, saturating at +-448:
    3 fraction bits at binade 2^e (e >= -6), steps of 2^-9 below 2^-6."""
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    step = np.exp2(e - 3.0)
    q = np.rint(a / step) * step
    return np.sign(y) * np.minimum(q, E4M3_MAX)


def e4m3_block_exponent(amax: np.ndarray) -> np.ndarray:
    """p of a 32-value block's scale 2^p: the smallest power of two with
    amax / 2^p <= 448 (no element saturates), kept to the normal range
    [-126, 126]; p = -126 for an all-zero block."""
    amax = np.asarray(amax, dtype=np.float64)
    with np.errstate(divide="ignore"):
        p = np.ceil(np.log2(amax / E4M3_MAX))
    p = np.where(amax > 0, p, -126.0)
    # log2 of an exact power of two times 448 can round either way: settle on the definition
    p = np.where((amax > 0) & (amax / np.exp2(p - 1) <= E4M3_MAX), p - 1, p)
    return np.clip(p, -126, 126)


def mx_e4m3_terms(v: np.ndarray, terms: int) -> np.ndarray:
    """v [..., K] (K a multiple of 32) as the sum of `terms` block-scaled E4M3
    terms: each term quantises what the previous ones left (the first, v
    itself) with its own per-32 scale.  Returns the represented values."""
    v = np.asarray(v, dtype=np.float64)
    shp = v.shape
    blocks = v.reshape(shp[:-1] + (shp[-1] // 32, 32))
    total = np.zeros_like(blocks)
    rest = blocks
    for _ in range(terms):
        p = e4m3_block_exponent(np.abs(rest).max(axis=-1))[..., None]
        term = e4m3_round(rest / np.exp2(p)) * np.exp2(p)
        total = total + term
        rest = rest - term
    return total.reshape(shp)


E2M1_MAX = 6.0


def e2m1_round(y: np.ndarray) -> np.ndarray:
    """Round to the nearest E2M1 value (0, 0.5, 1, 1.5, 2, 3, 4, 6 and
    negatives), ties to the even code, saturating at +-6."""
    y = np.asarray(y, dtype=np.float64)
    grid = E2M1_VALUES[:8]                                   # codes 0..7, ascending magnitudes
    a = np.minimum(np.abs(y), E2M1_MAX)[..., None]
    dist = np.abs(a - grid)
    best = dist.min(axis=-1, keepdims=True)
    cand = dist == best                                      # one code, or two at a midpoint
    even = cand & (np.arange(8) % 2 == 0)
    code = np.where(even.any(-1), np.argmax(even, -1), np.argmax(cand, -1))
    return np.sign(y) * grid[code]


def e2m1_block_exponent(amax: np.ndarray) -> np.ndarray:
    """p of a 32-value block's scale 2^p for E2M1 terms: the smallest power of
    two with amax / 2^p <= 6 (no element saturates), within [-126, 126];
    p = -126 for an all-zero block."""
    amax = np.asarray(amax, dtype=np.float64)
    with np.errstate(divide="ignore"):
        p = np.ceil(np.log2(amax / E2M1_MAX))
    p = np.where(amax > 0, p, -126.0)
    p = np.where((amax > 0) & (amax / np.exp2(p - 1) <= E2M1_MAX), p - 1, p)
    return np.clip(p, -126, 126)


def mx_e2m1_terms(v: np.ndarray, terms: int) -> np.ndarray:
    """v [..., K] (K a multiple of 32) as the sum of `terms` MXFP4 terms, each
    quantising what the previous ones left with its own E8M0 scale per 32."""
    v = np.asarray(v, dtype=np.float64)
    shp = v.shape
    blocks = v.reshape(shp[:-1] + (shp[-1] // 32, 32))
    total = np.zeros_like(blocks)
    rest = blocks
    for _ in range(terms):
        p = e2m1_block_exponent(np.abs(rest).max(axis=-1))[..., None]
        term = e2m1_round(rest / np.exp2(p)) * np.exp2(p)
        total = total + term
        rest = rest - term
    return total.reshape(shp)


def act_encode(v: np.ndarray, terms: int, fmt: str = "e4m3") -> np.ndarray:
    """The block-scaled encoding of the routed experts' inputs: E4M3 or E2M1 terms."""
    return mx_e2m1_terms(v, terms) if fmt == "e2m1" else mx_e4m3_terms(v, terms)


def mx_e4m3_valid_range(v: np.ndarray, rel: float = 1e-4):
    """The one-term encodings a computation of v can produce when it errs by
    at most rel times its 32-value block's largest magnitude (the scale of a
    dot product's rounding error): (lo, hi) per element, the smallest and
    largest encoding of any value within that distance, under either block
    scale when the block maximum itself lies that close to a scale
    threshold.  lo == hi where the encoding is unambiguous.  Rounding a value
    computed in lower precision is a decision taken near such boundaries, like
    a near tie of the router; any encoding in the range is correct."""
    v = np.asarray(v, dtype=np.float64)
    shp = v.shape
    blocks = v.reshape(shp[:-1] + (shp[-1] // 32, 32))
    amax = np.abs(blocks).max(axis=-1, keepdims=True)
    d = rel * amax
    lo, hi = None, None
    for pa in (amax * (1 - rel), amax * (1 + rel)):
        s = np.exp2(e4m3_block_exponent(pa))
        a = e4m3_round((blocks - d) / s) * s
        b = e4m3_round((blocks + d) / s) * s
        lo = a if lo is None else np.minimum(lo, a)
        hi = b if hi is None else np.maximum(hi, b)
    return lo.reshape(shp), hi.reshape(shp)


# ------------------------------------------------------------ activations
def sigmoid(z):
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-np.asarray(z, dtype=np.float64)))


def situ(g, u, beta=4.0, linear_beta=25.0):
    """SiTU-GLU (Kimi K3 card, routed-expert steps; SituAndMul):
    a = beta * tanh(g / beta) * sigma(g);  u_bar = linear_beta * tanh(u / linear_beta);
    h = a * u_bar."""
    a = beta * np.tanh(g / beta) * sigmoid(g)
    ubar = linear_beta * np.tanh(u / linear_beta)
    return a * ubar


def swiglu(g, u):
    """Kimi K2 card, routed-expert steps: a = g * sigma(g), h = a * u."""
    return g * sigmoid(g) * u


def rms_norm(u, w, eps):
    """RMSNorm over the last axis: w * u / sqrt(mean(u^2) + eps)."""
    return w * u / np.sqrt(np.mean(u * u, axis=-1, keepdims=True) + eps)


# ---------------------------------------------------------------- routing
def route_from_logits(z: np.ndarray, bias: np.ndarray, k: int, scale: float = 1.0):
    """Router steps after the logits.  z fp64 [T, E], bias [E].

    Returns dict: idx [T, k] (by biased score descending, ties to the lower
    index), G [T, k] (raw sigmoid renormalised over the selection, times
    `scale`), s, c (= s + b), and flag [T] (k-th and (k+1)-th biased scores
    within TIE_EPS)."""
    z = np.asarray(z, dtype=np.float64)
    T, E = z.shape
    s = sigmoid(z)
    c = s + np.asarray(bias, dtype=np.float64)[None, :]
    idx = np.empty((T, k), dtype=np.int64)
    flag = np.zeros(T, dtype=bool)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-c[t, e], e))
        idx[t] = order[:k]
        if k < E:
            flag[t] = (c[t, order[k - 1]] - c[t, order[k]]) < TIE_EPS
    G = weights_for(s, idx, scale)
    return dict(idx=idx, G=G, s=s, c=c, flag=flag, z=z)


def weights_for(s: np.ndarray, idx: np.ndarray, scale: float = 1.0) -> np.ndarray:
    """G_i = scale * s_i / sum_{j in selection} s_j (raw sigmoid, not s + b)."""
    sel = np.take_along_axis(s, idx, axis=1)
    return scale * sel / sel.sum(axis=1, keepdims=True)


def router(x: np.ndarray, Wr: np.ndarray, bias: np.ndarray, k: int, scale: float = 1.0):
    """z = x W_r^T with W_r in nn.Linear [E, d] storage, then route."""
    return route_from_logits(x @ Wr.T, bias, k, scale)


def dispatch(idx: np.ndarray, E: int):
    """Token -> expert dispatch of moe_infer, written as a counting sort.

    The flattened assignment a = t*k + j goes to expert idx[t, j].  Returns
    counts [E], offsets [E+1] (exclusive prefix sum), perm [T*k] (assignments
    grouped by expert, in increasing a inside each expert) and inv [T*k]
    (position of assignment a in perm)."""
    flat = np.asarray(idx).reshape(-1)
    counts = np.zeros(E, dtype=np.int64)
    for e in flat:
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    fill = offsets[:-1].copy()
    perm = np.empty(flat.size, dtype=np.int64)
    inv = np.empty(flat.size, dtype=np.int64)
    for a, e in enumerate(flat):
        perm[fill[e]] = a
        inv[a] = fill[e]
        fill[e] += 1
    return dict(counts=counts, offsets=offsets, perm=perm, inv=inv)


# ------------------------------------------------------------- the layer
class Layer:
    """Weights of one layer instance in fp64, dequantised on first use.

    W maps the C-ABI weight names to numpy arrays: bf16 tensors as uint16 bit
    patterns, expert codes / scales as uint8 [E, N, K/2] / [E, N, K/32]
    (MXFP4) or uint8 [E, N, K] / fp32 [E, N/128, K/128] (FP8).  Instead of
    stacked arrays, W may carry ``expert_fn(name, e) -> (q, s)`` to fetch one
    expert at a time."""

    def __init__(self, cfg, W: dict, cache_experts: bool = True):
        self.cfg = cfg
        self.W = W
        self.cache_experts = cache_experts   # False: dequantise an expert afresh on every use
        self._cache = {}

    def dense(self, name):
        if name not in self._cache:
            self._cache[name] = bf16_bits_to_f64(self.W[name])
        return self._cache[name]

    def expert(self, name, e):
        key = (name, e)
        if key in self._cache:
            return self._cache[key]
        if "expert_fn" in self.W:
            q, s = self.W["expert_fn"](name, e)
        else:
            q, s = self.W[name + "_q"][e], self.W[name + "_s"][e]
        if self.cfg.expert_wfmt == "mxfp4":
            w = dequant_mxfp4(q, s)
        else:
            w = dequant_fp8_block128(q, s)
        if self.cache_experts:
            self._cache[key] = w
        return w

    def shared(self, name):
        if self.cfg.expert_wfmt == "mxfp4":
            return self.dense(name)
        key = (name, "fp8")
        if key not in self._cache:
            self._cache[key] = dequant_fp8_block128(self.W[name], self.W[name + "_s"])
        return self._cache[key]

    def act(self, g, u):
        c = self.cfg
        if c.act == "situ":
            return situ(g, u, c.situ_beta, c.situ_linear_beta)
        return swiglu(g, u)


def forward(layer: Layer, x_bits: np.ndarray, routes: dict | None = None,
            idx: np.ndarray | None = None, act_terms: int | None = None,
            x_in: np.ndarray | None = None, h_in: np.ndarray | None = None, act_format: str = "e4m3") -> dict:
    """Delta for the tokens in x (bf16 bits [T, d]).

    routes: a dict from `router` to reuse; idx: a given selection [T, k]
    (its G is recomputed from this run's raw sigmoid); act_terms: None keeps
    the routed experts' inputs exact, 1 or 2 emulates their block-scaled
    E4M3 (act_format "e4m3") or E2M1 ("e2m1") encoding (x^c before the
    gate/up projections, h before the down projection) with that many terms;
    x_in: the encoded expert inputs [T][dx]
    to use instead of encoding x^c here (a choice among the encodings
    mx_e4m3_valid_range allows, checked by the caller); h_in: likewise the
    encoded hidden activations [T*k][F] per assignment a = t*k + j (the gate
    and up projections are then not evaluated).  Returns Delta and the
    intermediates (h: the hidden activations the down projections take; h_pre:
    before their encoding)."""
    cfg = layer.cfg
    x = bf16_bits_to_f64(x_bits)
    T = x.shape[0]
    k = cfg.top_k
    if routes is None:
        routes = router(x, layer.dense("router_w"), layer.W["router_bias"], k, cfg.routed_scale)
    if idx is not None:
        routes = dict(routes)
        routes["idx"] = np.asarray(idx, dtype=np.int64)
        routes["G"] = weights_for(routes["s"], routes["idx"], cfg.routed_scale)
    sel, G = routes["idx"], routes["G"]

    # Latent down-projection (K3); the K2 experts take x itself.
    xe = x @ layer.dense("w_down_latent").T if cfg.d_latent else x
    if x_in is not None:
        xin = np.asarray(x_in, dtype=np.float64)
    else:
        xin = act_encode(xe, act_terms, act_format) if act_terms else xe

    # moe_infer: group the assignments by expert, run each selected expert once
    # on its tokens, put the outputs back in assignment order.
    disp = dispatch(sel, cfg.n_experts)
    out = np.zeros((T * k, xe.shape[1]), dtype=np.float64)
    h_all = np.zeros((T * k, cfg.d_expert_ff), dtype=np.float64)
    h_pre = np.zeros((T * k, cfg.d_expert_ff), dtype=np.float64)
    for e in range(cfg.n_experts):
        lo, hi = disp["offsets"][e], disp["offsets"][e + 1]
        if hi == lo:
            continue
        assign = disp["perm"][lo:hi]
        toks = assign // k
        if h_in is not None:
            h = np.asarray(h_in, dtype=np.float64)[assign]
        else:
            g = xin[toks] @ layer.expert("ex_gate", e).T
            u = xin[toks] @ layer.expert("ex_up", e).T
            h = layer.act(g, u)
            h_pre[assign] = h
            if act_terms:
                h = act_encode(h, act_terms, act_format)
        h_all[assign] = h
        out[assign] = h @ layer.expert("ex_down", e).T
    # Weighted sum over each token's selection (u in the pages' notation).
    u_sum = (out.reshape(T, k, -1) * G[:, :, None]).sum(axis=1)

    if cfg.d_latent:
        u_hat = rms_norm(u_sum, layer.dense("norm_w"), cfg.norm_eps) if cfg.use_latent_norm else u_sum
        y_routed = u_hat @ layer.dense("w_up_latent").T
    else:
        u_hat = None
        y_routed = u_sum

    if cfg.d_shared_ff:
        gs = x @ layer.shared("sh_gate").T
        us = x @ layer.shared("sh_up").T
        h_s = layer.act(gs, us)
        y_shared = h_s @ layer.shared("sh_down").T
    else:
        h_s = None
        y_shared = np.zeros_like(y_routed)
    delta = y_routed + y_shared
    return dict(delta=delta, routes=routes, xc=xe if cfg.d_latent else None, x_in=xin, h=h_all, h_pre=h_pre,
                u=u_sum,
                u_hat=u_hat, y_routed=y_routed, y_shared=y_shared, h_s=h_s, dispatch=disp)


# ------------------------------------------------------- input conversion
def numpy_inputs(tensors: dict) -> dict:
    """torch tensors from lmoe_inputs -> numpy arrays the oracle reads
    (bf16 as uint16 bit patterns).  Only the representation changes."""
    import torch
    out = {}
    for k, v in tensors.items():
        if not isinstance(v, torch.Tensor):
            out[k] = v
            continue
        v = v.detach().cpu()
        if v.dtype == torch.bfloat16:
            out[k] = v.view(torch.int16).numpy().view(np.uint16)
        else:
            out[k] = v.numpy()
    return out


# ------------------------------------------------------- quantile balancing
# The selection-bias update of Stable LatentMoE (tutorial "Stable LatentMoE",
# section "Quantile Balancing: giving every expert a fair shot"; walk-through
# "Kimi K3 模型结构（5）", section "Stable 之三：Quantile Balancing", with its
# appendix-C derivation and the appendix-D histogram estimator).  Scores s are
# the raw sigmoids [m, n] of a batch routed with the current biases b.
def qb_cutoffs(s: np.ndarray, b: np.ndarray, k: int) -> np.ndarray:
    """alpha_i: the (k+1)-th largest biased score s_i + b of token i, the
    line an expert must cross to enter token i's top-k."""
    c = np.asarray(s, dtype=np.float64) + np.asarray(b, dtype=np.float64)[None, :]
    assert k < c.shape[1], "the cutoff needs k + 1 <= n experts"
    return -np.sort(-c, axis=1)[:, k]


def qb_required_bias(s: np.ndarray, b: np.ndarray, k: int) -> np.ndarray:
    """r_ij = alpha_i - s_ij: the bias expert j would need to cross token i's
    cutoff (token i selects j under a new bias b_j exactly when b_j > r_ij)."""
    return qb_cutoffs(s, b, k)[:, None] - np.asarray(s, dtype=np.float64)


def quantile_higher(v: np.ndarray, num: int, den: int) -> np.ndarray:
    """(num/den)-quantile along axis 0 with the 'higher' convention: the sorted
    value at index ceil(num/den * (m - 1)), the index in exact integers."""
    v = np.sort(np.asarray(v, dtype=np.float64), axis=0)
    i = -(-(num * (v.shape[0] - 1)) // den)
    return v[i]


def qb_update(s: np.ndarray, b: np.ndarray, k: int) -> dict:
    """Exact update: b_new_j = the (k/n)-quantile of r_{:,j} (its target share
    q = m k / n of the m tokens), then centred (a common offset does not
    change any top-k).  Returns the centred biases and the raw quantiles."""
    r = qb_required_bias(s, b, k)
    n = r.shape[1]
    raw = quantile_higher(r, k, n)
    return dict(bias=raw - raw.mean(), raw=raw, r=r)


def qb_range(b: np.ndarray):
    """Histogram range of the required biases: s lies in (0, 1) and every
    cutoff is some expert's biased score, so r lies in [min b - 1, max b + 1]."""
    b = np.asarray(b, dtype=np.float64)
    return b.min() - 1.0, b.max() + 1.0


def qb_histogram(s: np.ndarray, b: np.ndarray, k: int, bins: int) -> np.ndarray:
    """n x B integer counts of the required biases r_ij in B uniform bins of
    the range (values on the upper edge go to the last bin)."""
    r = qb_required_bias(s, b, k)
    lo, hi = qb_range(b)
    w = (hi - lo) / bins
    counts = np.zeros((r.shape[1], bins), dtype=np.int64)
    for j in range(r.shape[1]):
        for v in r[:, j]:
            c = min(max(int(np.floor((v - lo) / w)), 0), bins - 1)
            counts[j, c] += 1
    return counts


def qb_update_from_histogram(counts: np.ndarray, b: np.ndarray, k: int) -> dict:
    """Quantile of each expert's histogram: the first bin whose cumulative
    count reaches ceil(q), q = m k / n (m = the tokens counted, each expert
    counts every token once), with linear interpolation inside that bin; then
    centred."""
    counts = np.asarray(counts, dtype=np.int64)
    n, B = counts.shape
    lo, hi = qb_range(b)
    w = (hi - lo) / B
    raw = np.empty(n, dtype=np.float64)
    for j in range(n):
        m = counts[j].sum()
        target = int(np.ceil(m * k / n))
        cum = 0
        for c in range(B):
            if counts[j, c] and cum + counts[j, c] >= target:
                raw[j] = lo + w * (c + (target - cum) / counts[j, c])
                break
            cum += counts[j, c]
        else:
            raw[j] = hi
    return dict(bias=raw - raw.mean(), raw=raw)
