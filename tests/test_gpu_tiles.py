"""Every token-tile size of the grouped expert GEMMs against the fp64 oracle.

The tile is chosen from the mean assignments per expert (16 and 32 with
interleaved hi/lo activation columns, 64 and 96 with split hi/lo operands for
MXFP4 weights; 16 to 96, all split, for FP8 weights), so a small layer run at
several token counts reaches each tile, with ragged last tiles, at sizes the
oracle checks token by token."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle as O
from lmoe_inputs import configs as C
from tests._harness import (assert_delta_close, check_expert_io, forward_checked, gpu_inputs, make_layer,
                            oracle_layer, rel_l2_per_token, x_bits)

pytestmark = pytest.mark.gpu

K3_TINY = C.Workload("k3_tiny_tiles", C.K3_TINY, T=3001, seed=51)         # E 64, k 2
K3_MID = C.Workload("k3_mid_tiles", C.K3_MID, T=1800, seed=52)            # E 160, k 6, F 608 (padded K)
K2_SMALL = C.Workload("k2_small_tiles", replace(C.K2, d_model=1024, n_experts=48, top_k=4, d_expert_ff=384,
                                                d_shared_ff=256), T=1001, seed=53)
CASES = [(K3_TINY, (100, 400, 1500, 3001)),    # tiles 16, 32, 64, 96
         (K3_MID, (1000, 1800)),               # tiles 64, 96 with a 608-row (padded) contraction
         (K2_SMALL, (100, 300, 600, 1001))]    # FP8 tiles 16, 32, 64, 96


@pytest.mark.parametrize("wl,Ts", CASES, ids=[c[0].name for c in CASES])
def test_all_token_tiles(wl, Ts):
    W, x = gpu_inputs(wl)
    layer = make_layer(wl, W, max_tokens=wl.T)
    olayer = oracle_layer(wl, W)
    try:
        for T in Ts:
            xt = x[:T].contiguous()
            got, got32, idx, _ = forward_checked(layer, xt)
            ref = O.forward(olayer, x_bits(xt), idx=idx)
            check_expert_io(layer, T, wl.cfg.top_k, ref["x_in"], ref["h"], 2, label=f"{wl.name} T={T}")
            u = layer.lmoe_debug_tensor("u", T).cpu().double().numpy()
            assert rel_l2_per_token(u, ref["u"]).max() <= 1e-2, T
            assert_delta_close(got, ref["delta"], got32, label=f"{wl.name} T={T}")
        # repeated forwards of the largest batch are bit-identical
        a = layer.lmoe_forward(x).cpu()
        b = layer.lmoe_forward(x).cpu()
        assert torch.equal(a, b)
    finally:
        layer.close()


# d = 1024, Fs = 1024 at T = 10,000 (40 tiles of 256 tokens): the shared
# gate/up GEMM (8 gate/up tile pairs, SiTU in the epilogue) and the
# K-concatenated output GEMM (4 paired tiles, bf16 in the epilogue) run wide,
# two 128-row accumulators per CTA, while the router and the latent GEMM keep
# one tile per CTA.
# The routing uses the top-k of the model each layer is shaped after (K3:
# 16, K2: 8).
WIDE = C.Workload("k3_wide_dense", replace(C.K3_TINY, d_model=1024, d_latent=512, n_experts=64, top_k=16,
                                           d_expert_ff=256, d_shared_ff=1024), T=10000, seed=54)
# K2-shaped: its shared expert runs on the FP8 expert GEMMs (tiles of 96
# tokens), all tokens checked.
WIDE_K2 = C.Workload("k2_wide_dense", replace(C.K2, d_model=1024, n_experts=48, top_k=8, d_expert_ff=384,
                                              d_shared_ff=1024), T=10000, seed=55)


@pytest.mark.parametrize("wl", [WIDE, WIDE_K2], ids=["k3_shape", "k2_shape"])
def test_wide_dense_tiles_all_tokens(wl):
    W, x = gpu_inputs(wl)
    layer = make_layer(wl, W, max_tokens=wl.T)
    olayer = oracle_layer(wl, W)
    try:
        got, got32, idx, _ = forward_checked(layer, x)
        ref = O.forward(olayer, x_bits(x), idx=idx)
        if wl.cfg.expert_wfmt == "mxfp4":
            hs = layer.lmoe_debug_tensor("h_shared", wl.T).cpu().double().numpy()
            assert rel_l2_per_token(hs, ref["h_s"]).max() <= 1e-2
        else:
            ys = layer.lmoe_debug_tensor("y_shared", wl.T).cpu().double().numpy()
            assert rel_l2_per_token(ys, ref["y_shared"]).max() <= 1e-2
        assert_delta_close(got, ref["delta"], got32, label=f"{wl.name} T={wl.T}")
    finally:
        layer.close()


# Decode-sized batches of a d = 4096 layer: every dense GEMM splits K across
# CTAs (up to 19 splits) and sums fp32 partials; every token is checked.
WIDE_SPLITK = C.Workload("k3_wide_splitk", replace(C.K3_TINY, d_model=4096, d_latent=2048, n_experts=32, top_k=4,
                                                   d_expert_ff=256, d_shared_ff=4096), T=64, seed=56)


def test_split_k_dense_all_tokens():
    wl = WIDE_SPLITK
    W, x = gpu_inputs(wl)
    layer = make_layer(wl, W, max_tokens=wl.T)
    olayer = oracle_layer(wl, W)
    try:
        for T in (8, 64):
            xt = x[:T].contiguous()
            got, got32, idx, _ = forward_checked(layer, xt)
            ref = O.forward(olayer, x_bits(xt), idx=idx)
            xc = layer.lmoe_debug_tensor("xc", T).cpu().double().numpy()
            assert np.abs(xc - ref["xc"]).max() <= 1e-4 * (1 + np.abs(ref["xc"]).max())
            hs = layer.lmoe_debug_tensor("h_shared", T).cpu().double().numpy()
            assert rel_l2_per_token(hs, ref["h_s"]).max() <= 1e-2
            assert_delta_close(got, ref["delta"], got32, label=f"{wl.name} T={T}")
    finally:
        layer.close()
