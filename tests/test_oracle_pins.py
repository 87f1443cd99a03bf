"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: numbers
printed on the pages, closed forms, brute force on tiny inputs, library
routines for the special cases that reduce to one, and invariants the method
guarantees.  A plausible slip in the oracle (a dropped term, a swapped beta,
a transposed operand, the norm in the wrong place, weighting by s+b instead of
s) fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from lmoe_inputs import configs as C
from lmoe_inputs import generate as G

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------ parameter counts
def test_param_counts_k3():
    """Kimi K3 card, "Exact per-instance accounting" table."""
    p = C.param_counts(C.K3)
    assert p["router"] == 6_423_424
    assert p["latent_down"] == 25_690_112
    assert p["routed_expert"] == 33_030_144
    assert C.K3.n_experts * p["routed_expert"] == 29_595_009_024
    assert p["latent_norm"] == 3_584
    assert p["latent_up"] == 25_690_112
    assert p["shared"] == 132_120_576
    assert p["total"] == 29_784_936_832


def test_param_counts_k2():
    """Kimi K2 card, "Exact per-instance accounting" table."""
    p = C.param_counts(C.K2)
    assert p["router"] == 2_752_896
    assert p["routed_expert"] == 44_040_192
    assert C.K2.n_experts * p["routed_expert"] == 16_911_433_728
    assert p["shared"] == 44_040_192
    assert p["total"] == 16_958_226_816


def test_generated_shapes_match_counts():
    """The generator's tensors hold exactly the counted parameters (tiny
    layer in full, one full-size K3 and K2 expert)."""
    wl = C.workload("k3_tiny_t16")
    W = G.gen_weights(wl)
    cfg = wl.cfg
    n = W["router_w"].numel() + W["router_bias"].numel()
    assert n == C.param_counts(cfg)["router"] == 41_024
    per_expert = sum(2 * W[f"{m}_q"][0].numel() for m in ("ex_gate", "ex_up", "ex_down"))
    assert per_expert == C.param_counts(cfg)["routed_expert"] == 245_760
    sh = W["sh_gate"].numel() + W["sh_up"].numel() + W["sh_down"].numel()
    assert sh == C.param_counts(cfg)["shared"] == 983_040
    for m in ("ex_gate", "ex_up", "ex_down"):
        assert W[f"{m}_s"][0].numel() * 32 == 2 * W[f"{m}_q"][0].numel()
    q, s = G.gen_expert(C.workload("k3_decode_t64"), "ex_gate", 0)
    assert tuple(q.shape) == (3072, 1792) and tuple(s.shape) == (3072, 112)
    q, s = G.gen_expert(C.workload("k3_decode_t64"), "ex_down", 5)
    assert tuple(q.shape) == (3584, 1536) and tuple(s.shape) == (3584, 96)


# ------------------------------------------------------------------- formats
E2M1_GRID = {0: 0.0, 1: 0.5, 2: 1.0, 3: 1.5, 4: 2.0, 5: 3.0, 6: 4.0, 7: 6.0}


def test_mxfp4_dequant_exhaustive():
    """16 codes x 255 scale bytes against sign * grid * 2^(s-127) taken from
    the E2M1 value table and math.ldexp, with the even index in the low
    nibble of each byte."""
    codes = np.arange(16, dtype=np.uint8)
    for s in range(255):
        q = np.zeros((1, 16), dtype=np.uint8)
        q[0, :8] = codes[0::2] | (codes[1::2] << 4)     # 16 codes in order
        q[0, 8:] = codes[1::2] | (codes[0::2] << 4)     # pairs swapped
        sc = np.full((1, 1), s, dtype=np.uint8)
        w = O.dequant_mxfp4(q, sc)[0]
        order = list(codes) + [c for pair in zip(codes[1::2], codes[0::2]) for c in pair]
        for i, c in enumerate(order):
            mag = E2M1_GRID[int(c) & 7]
            want = math.ldexp(-mag if c & 8 else mag, s - 127)
            assert w[i] == want, (s, i, c)


def test_mxfp4_quantiser_roundtrip_exact_values():
    """Values already on the E2M1 grid times 2^X (X from the block's amax)
    survive quantise -> dequantise exactly; a block's amax lands on 4 or 6."""
    rng = np.random.default_rng(7)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)
    vals = rng.choice(grid, size=(8, 64)) * rng.choice([-1, 1], size=(8, 64))
    vals[:, 0] = 6.0
    vals[:, 32] = -4.0
    w = torch.from_numpy((vals * 2.0 ** -7).astype(np.float32))
    q, s = G.quantise_mxfp4(w)
    back = O.dequant_mxfp4(q.numpy(), s.numpy())
    assert np.array_equal(back, vals * 2.0 ** -7)


def test_e4m3_all_bytes_against_torch():
    b = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = O.e4m3_value(b)
    both_nan = np.isnan(ref) & np.isnan(mine)
    assert np.array_equal(mine[~both_nan], ref[~both_nan])
    assert np.array_equal(np.isnan(ref), np.isnan(mine))


def test_bf16_bits_against_torch():
    x = torch.randn(4096, dtype=torch.float32).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.bf16_bits_to_f64(bits), x.to(torch.float64).numpy())


def test_fp8_block_dequant_orientation():
    """Block (i, j) of the fp32 scale multiplies rows 128i.. and columns 128j.."""
    q = np.full((256, 384), 0x38, dtype=np.uint8)   # e4m3 1.0
    s = np.arange(6, dtype=np.float32).reshape(2, 3) + 1
    w = O.dequant_fp8_block128(q, s)
    assert w[0, 0] == 1 and w[0, 128] == 2 and w[0, 256] == 3
    assert w[128, 0] == 4 and w[255, 383] == 6


# ---------------------------------------------------------------- activations
def test_situ_bounded_by_100():
    """Appendix B property quoted on the K3 walk-through: |h| <= beta1*beta2 = 100."""
    g = np.concatenate([-np.logspace(-3, 4, 200), np.logspace(-3, 4, 200)])
    gg, uu = np.meshgrid(g, g)
    h = O.situ(gg, uu)
    assert np.all(np.abs(h) <= 100.0)
    assert abs(O.situ(1e4, 1e4) - 100.0) < 1e-9          # saturates at the bound
    assert abs(O.situ(1e4, -1e4) + 100.0) < 1e-9


def test_situ_first_order_swiglu():
    """beta*tanh(z/beta) = z - z^3/(3 beta^2) + O(z^5): near 0 the gap to
    SwiGLU is sigma(g)*(|g|^3 |u| / 48 + |g| |u|^3 / 1875) to leading order
    (48 = 3*4^2 pins beta1 = 4 on the gate, 1875 = 3*25^2 pins beta2 = 25
    on the up branch)."""
    pts = [(0.01, 0.1), (0.1, 0.01), (-0.05, 0.08), (0.08, -0.1), (0.1, 0.1), (-0.1, -0.1), (0.003, 0.09)]
    for g, u in pts:
        gap = abs(O.situ(g, u) - O.swiglu(g, u))
        sig = 1 / (1 + math.exp(-g))
        lead = sig * (abs(g) ** 3 * abs(u) / 48 + abs(g) * abs(u) ** 3 / 1875)
        assert gap <= lead * 1.01, (g, u, gap, lead)
        assert gap >= lead * 0.98, (g, u, gap, lead)


def test_situ_converges_to_swiglu():
    g = np.linspace(-8, 8, 97)
    gg, uu = np.meshgrid(g, g)
    ref = torch.nn.functional.silu(torch.from_numpy(gg)).numpy() * uu
    got = O.situ(gg, uu, beta=1e7, linear_beta=1e7)
    assert np.allclose(got, ref, rtol=1e-10, atol=1e-12)
    assert np.allclose(O.swiglu(gg, uu), ref, rtol=1e-13, atol=1e-14)


def test_sigmoid_and_rmsnorm_library():
    z = np.linspace(-30, 30, 1001)
    ref = torch.sigmoid(torch.from_numpy(z)).numpy()
    assert np.allclose(O.sigmoid(z), ref, rtol=1e-14, atol=0)
    u = np.random.default_rng(1).standard_normal((5, 320))
    w = 1 + 0.02 * np.random.default_rng(2).standard_normal(320)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(u), (320,), torch.from_numpy(w), eps=1e-6).numpy()
    assert np.allclose(O.rms_norm(u, w, 1e-6), ref, rtol=1e-13, atol=1e-14)


# -------------------------------------------------------------------- routing
def _logit(p):
    p = np.asarray(p, dtype=np.float64)
    return np.log(p / (1 - p))


def test_worked_routing_example():
    """Stable LatentMoE tutorial: four experts, raw scores 0.90/0.80/0.65/0.20,
    biases -0.40 and +0.25 -> experts 3 and 2 (0-based 2, 1), mixed at about
    45% / 55% with the raw scores."""
    ex = json.load(open(os.path.join(GOLDEN, "routing_worked_example.json")))
    z = _logit([ex["raw_scores"]])
    r0 = O.route_from_logits(z, np.zeros(4), ex["k"])
    assert list(r0["idx"][0]) == ex["selected_without_bias"]
    r = O.route_from_logits(z, np.array(ex["bias"]), ex["k"])
    assert np.allclose(r["c"][0], ex["selection_scores"], atol=1e-12)
    assert list(r["idx"][0]) == ex["selected"]
    for j, e in enumerate(r["idx"][0]):
        assert abs(r["G"][0, j] - ex["mixing_weights"][str(e)]) < 1e-12
        assert round(100 * r["G"][0, j]) == ex["mixing_weights_page_rounded_percent"][str(e)]


def test_topk_brute_force_small():
    """Top-k of s + b equals the k-subset with the largest sum of biased
    scores (ties: the lexicographically smallest index set), for E <= 10."""
    rng = np.random.default_rng(3)
    for trial in range(60):
        E = int(rng.integers(2, 11))
        k = int(rng.integers(1, E + 1))
        z = rng.normal(size=(1, E))
        b = rng.uniform(-0.1, 0.1, size=E)
        if trial % 3 == 0:      # exact ties in the biased score
            z[0, :] = 0.0
            b = rng.choice([-0.05, 0.0, 0.05], size=E)
        c = 1 / (1 + np.exp(-z[0])) + b
        best = max(itertools.combinations(range(E), k), key=lambda S: (round(sum(c[list(S)]), 12), [-i for i in S]))
        r = O.route_from_logits(z, b, k)
        assert sorted(r["idx"][0]) == list(best), (E, k, c)
        sel = c[r["idx"][0]]
        assert np.all(np.diff(sel) <= 0)


def test_weights_use_raw_sigmoid_not_biased_score():
    """Kimi K3 card router steps and the port notes (3): selection by s + b,
    weighting by the raw s renormalised to 1."""
    z = _logit([[0.6, 0.6, 0.1, 0.2]])
    b = np.array([0.0, 0.3, 0.0, 0.0])
    r = O.route_from_logits(z, b, 2)
    assert list(r["idx"][0]) == [1, 0]
    assert np.allclose(r["G"][0], [0.5, 0.5])
    r1 = O.route_from_logits(z, np.zeros(4), 1)
    assert r1["G"][0, 0] == 1.0
    rk = O.route_from_logits(z, b, 2, scale=2.827)
    assert np.allclose(rk["G"][0].sum(), 2.827)


def test_tie_flag():
    z = np.zeros((2, 5))
    b = np.array([0.3, 0.2, 0.1, 0.1 - 5e-7, 0.0])
    b2 = np.array([0.3, 0.2, 0.1, 0.1 - 2e-6, 0.0])
    r = O.route_from_logits(z, b, 3)
    assert r["flag"][0] and r["flag"][1]
    r2 = O.route_from_logits(z, b2, 3)
    assert not r2["flag"][0]
    assert not O.route_from_logits(z, b2, 5)["flag"].any()


def test_dispatch_against_stable_argsort():
    rng = np.random.default_rng(5)
    for E, T, k in [(8, 5, 3), (64, 16, 2), (896, 9, 16)]:
        idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)])
        d = O.dispatch(idx, E)
        flat = idx.reshape(-1)
        assert np.array_equal(d["counts"], np.bincount(flat, minlength=E))
        assert np.array_equal(d["perm"], np.argsort(flat, kind="stable"))
        assert np.array_equal(d["inv"][d["perm"]], np.arange(flat.size))
        assert d["offsets"][-1] == T * k


# --------------------------------------------------------------- whole layer
def _tiny(**cfg_over):
    wl = C.workload("k3_tiny_t16")
    if cfg_over:
        from dataclasses import replace
        wl = replace(wl, cfg=replace(wl.cfg, **cfg_over))
    W = O.numpy_inputs(G.gen_weights(wl))
    x = O.numpy_inputs({"x": G.gen_x(wl)})["x"]
    return wl, W, x


def _dense_reference(layer, x_bits):
    """P1's sum u = sum_{i=1}^{E} G_i E_i written literally: every expert on
    every token, G_i = 0 for the unselected ones, no dispatch at all."""
    cfg = layer.cfg
    x = O.bf16_bits_to_f64(x_bits)
    r = O.router(x, layer.dense("router_w"), layer.W["router_bias"], cfg.top_k, cfg.routed_scale)
    T = x.shape[0]
    Gfull = np.zeros((T, cfg.n_experts))
    for t in range(T):
        Gfull[t, r["idx"][t]] = r["G"][t]
    xc = x @ layer.dense("w_down_latent").T
    u = np.zeros((T, cfg.d_latent))
    for e in range(cfg.n_experts):
        h = layer.act(xc @ layer.expert("ex_gate", e).T, xc @ layer.expert("ex_up", e).T)
        u += Gfull[:, e:e + 1] * (h @ layer.expert("ex_down", e).T)
    uh = layer.dense("norm_w") * u / np.sqrt((u * u).mean(-1, keepdims=True) + cfg.norm_eps)
    y = uh @ layer.dense("w_up_latent").T
    hs = layer.act(x @ layer.dense("sh_gate").T, x @ layer.dense("sh_up").T)
    return y + hs @ layer.dense("sh_down").T


def test_forward_matches_dense_formulation():
    wl, W, x = _tiny()
    layer = O.Layer(wl.cfg, W)
    got = O.forward(layer, x)["delta"]
    ref = _dense_reference(layer, x)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)
    assert got.shape == (16, 640)


def test_norm_sits_after_the_sum():
    """Port notes (4) and K3 card code: routed_expert_norm between the expert
    sum and the up-projection.  Doubling every expert's down weights (scale
    byte + 1) or every G leaves Delta unchanged up to the eps effect; a norm
    before the experts would not cancel them."""
    from dataclasses import replace
    wl, W, x = _tiny()
    base = O.forward(O.Layer(wl.cfg, W), x)
    W2 = dict(W)
    W2["ex_down_s"] = W["ex_down_s"] + 1
    d2 = O.forward(O.Layer(wl.cfg, W2), x)
    assert np.allclose(d2["u"], 2 * base["u"], rtol=1e-14)
    # closed form of the eps effect: RMSNorm(2u) = RMSNorm(u) * 2 sqrt(m+eps) / sqrt(4m+eps)
    m = (base["u"] ** 2).mean(-1, keepdims=True)
    eps = wl.cfg.norm_eps
    f = 2 * np.sqrt(m + eps) / np.sqrt(4 * m + eps)
    assert np.allclose(d2["u_hat"], base["u_hat"] * f, rtol=1e-12)
    assert np.allclose(d2["y_routed"], base["y_routed"] * f, rtol=1e-10, atol=1e-13)
    # with eps = 0 the doubling cancels exactly (up to rounding)
    cfg0 = replace(wl.cfg, norm_eps=0.0)
    a0 = O.forward(O.Layer(cfg0, W), x)
    assert np.allclose(O.forward(O.Layer(cfg0, W2), x)["delta"], a0["delta"], rtol=1e-12, atol=1e-12)
    d3 = O.forward(O.Layer(replace(cfg0, routed_scale=2.0), W), x)
    assert np.allclose(d3["delta"], a0["delta"], rtol=1e-12, atol=1e-12)
    # without the norm, the doubling passes straight through
    d4 = O.forward(O.Layer(replace(wl.cfg, use_latent_norm=False), W2), x)
    d5 = O.forward(O.Layer(replace(wl.cfg, use_latent_norm=False), W), x)
    assert np.allclose(d4["y_routed"], 2 * d5["y_routed"], rtol=1e-12)
    # u_hat has unit RMS up to the norm weight
    rms = np.sqrt((base["u_hat"] / O.bf16_bits_to_f64(W["norm_w"])) ** 2).mean(-1)
    assert np.all(rms > 0)
    uh = base["u_hat"] / O.bf16_bits_to_f64(W["norm_w"])
    assert np.allclose(np.sqrt((uh * uh).mean(-1)), 1.0, atol=1e-3)


def test_token_permutation_equivariance():
    wl, W, x = _tiny()
    layer = O.Layer(wl.cfg, W)
    base = O.forward(layer, x)["delta"]
    p = np.random.default_rng(0).permutation(x.shape[0])
    got = O.forward(layer, x[p])["delta"]
    assert np.allclose(got, base[p], rtol=1e-13, atol=1e-13)


def test_selection_bias_only_moves_the_choice():
    wl, W, x = _tiny()
    layer = O.Layer(wl.cfg, W)
    base = O.forward(layer, x)
    # a constant shift of b changes nothing
    W2 = dict(W)
    W2["router_bias"] = (W["router_bias"].astype(np.float64) + 0.37)
    d2 = O.forward(O.Layer(wl.cfg, W2), x)
    assert np.array_equal(d2["routes"]["idx"], base["routes"]["idx"])
    assert np.array_equal(d2["delta"], base["delta"])
    # lowering the bias of experts nobody selected changes nothing either
    unused = np.setdiff1d(np.arange(wl.cfg.n_experts), base["routes"]["idx"].reshape(-1))
    W3 = dict(W)
    b3 = W["router_bias"].astype(np.float64).copy()
    b3[unused] -= 0.5
    W3["router_bias"] = b3
    d3 = O.forward(O.Layer(wl.cfg, W3), x)
    assert np.array_equal(d3["delta"], base["delta"])


def test_equal_experts_make_routing_irrelevant():
    """With every expert identical, sum_i G_i E_i = E(x^c) since the G sum to
    1: Delta does not depend on the bias."""
    wl, W, x = _tiny()
    W1 = dict(W)
    for m in ("ex_gate", "ex_up", "ex_down"):
        W1[m + "_q"] = np.repeat(W[m + "_q"][:1], wl.cfg.n_experts, axis=0)
        W1[m + "_s"] = np.repeat(W[m + "_s"][:1], wl.cfg.n_experts, axis=0)
    a = O.forward(O.Layer(wl.cfg, W1), x)["delta"]
    W2 = dict(W1)
    W2["router_bias"] = np.random.default_rng(9).uniform(-1, 1, wl.cfg.n_experts)
    b = O.forward(O.Layer(wl.cfg, W2), x)
    assert np.allclose(a, b["delta"], rtol=1e-12, atol=1e-12)


def test_k_equals_E_is_dense_sigmoid_mixture():
    from dataclasses import replace
    wl, W, x = _tiny()
    cfg = replace(wl.cfg, n_experts=6, top_k=6)
    W6 = {k: (v[:6] if k.startswith("ex_") or k.startswith("router") else v) for k, v in W.items()}
    layer = O.Layer(cfg, W6)
    out = O.forward(layer, x)
    s = O.sigmoid(O.bf16_bits_to_f64(x) @ layer.dense("router_w").T)
    Gd = s / s.sum(1, keepdims=True)
    got = np.take_along_axis(out["routes"]["G"], np.argsort(out["routes"]["idx"], 1), 1)
    assert np.allclose(got, Gd, rtol=1e-14)
    assert not out["routes"]["flag"].any()


def test_k2_routed_scale_is_linear():
    """K2 card: G = 2.827 * s / sum s and no norm, so the routed output scales
    linearly with the factor."""
    from dataclasses import replace
    cfg = replace(C.K2, d_model=256, n_experts=12, top_k=3, d_expert_ff=256, d_shared_ff=256)
    wl = C.Workload("k2_small", cfg, T=5, seed=11)
    W = O.numpy_inputs(G.gen_weights(wl))
    x = O.numpy_inputs({"x": G.gen_x(wl)})["x"]
    a = O.forward(O.Layer(cfg, W), x)
    b = O.forward(O.Layer(replace(cfg, routed_scale=1.0), W), x)
    assert np.allclose(a["y_routed"], 2.827 * b["y_routed"], rtol=1e-12)
    assert np.allclose(a["delta"] - a["y_routed"], b["delta"] - b["y_routed"], rtol=1e-14)
    # SwiGLU experts: the literal per-token formula for one token
    layer = O.Layer(cfg, W)
    xt = O.bf16_bits_to_f64(x)[0]
    acc = 0
    for j, e in enumerate(a["routes"]["idx"][0]):
        g = layer.expert("ex_gate", e) @ xt
        u = layer.expert("ex_up", e) @ xt
        acc = acc + a["routes"]["G"][0, j] * (layer.expert("ex_down", e) @ (g / (1 + np.exp(-g)) * u))
    assert np.allclose(acc, a["y_routed"][0], rtol=1e-12, atol=1e-12)


def test_batched_expert_generation_matches_per_expert():
    """The batched generator (used on GPUs) yields the bytes of the
    one-expert-at-a-time generator the oracle's inputs come from."""
    wl = C.workload("k3_tiny_t16")
    for name in ("ex_gate", "ex_down"):
        qa, sa = G.gen_experts_mxfp4(wl, name, "cpu", chunk=5)
        for e in (0, 7, 63):
            q, s = G.gen_expert(wl, name, e)
            assert torch.equal(qa[e], q) and torch.equal(sa[e], s)
