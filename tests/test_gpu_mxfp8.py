"""The one-term activation mode (act_terms = 1: MXFP8, one E4M3 code per
value with an E8M0 scale per 32, the deployment precision the walk-through's
"参数账" section names) against the fp64 oracle emulating the same encoding
of the routed experts' inputs (x^c before gate/up, h before down), at the
layer tolerances: per-token relative L2 <= 1e-2 and max-abs <= 2e-2 RMS on
Delta before its bf16 rounding.  Where an fp32 x^c falls within 1e-4 of an
E4M3 rounding midpoint or block-scale threshold, either encoding is correct
(a decision like the router's near ties): the GPU's is checked to be one of
the valid encodings and the oracle then continues from it.  The same holds
for h, whose fp32 value the epilogue computes with the hardware tanh and exp
approximations (relative error ~2^-11): every GPU h is checked to encode a
value within 2e-3 of its block's largest magnitude of the exact h, and the
down projection then continues from it.

Against the exact oracle the mode is off by the encoding itself; that error
is printed and bounded by the encoding's worst case (half an E4M3 step,
2^-4 of each value, on each of the two quantised inputs of the routed path,
1/8 in all)."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle as O
from lmoe_inputs import configs as C
from tests._harness import (assert_delta_close, check_expert_io, forward_checked, gpu_inputs, make_layer,
                            oracle_layer, rel_l2_per_token, validated_one_term_hidden, validated_one_term_inputs,
                            x_bits)
from tests._oracle_workers import OracleWorkers
from tests.test_gpu_parity import full_size_check

pytestmark = pytest.mark.gpu

TILES = [(C.Workload("k3_tiny_mxfp8", replace(C.K3_TINY, act_terms=1), T=3001, seed=51), (3, 100, 400, 1500, 3001)),
         (C.Workload("k3_mid_mxfp8", replace(C.K3_MID, act_terms=1), T=1800, seed=52), (37, 1000, 1800))]


@pytest.mark.parametrize("wl,Ts", TILES, ids=[c[0].name for c in TILES])
def test_one_term_all_tiles(wl, Ts):
    """Tiles 16 and 32 (interleaved: the lo column holds an exact zero),
    64 and 96 (split: only the hi rows are loaded and multiplied), every
    token."""
    W, x = gpu_inputs(wl)
    layer = make_layer(wl, W, max_tokens=wl.T)
    olayer = oracle_layer(wl, W)
    try:
        for T in Ts:
            xt = x[:T].contiguous()
            got, got32, idx, _ = forward_checked(layer, xt)
            exact = O.forward(olayer, x_bits(xt), idx=idx)
            x_in, other = validated_one_term_inputs(layer, T, wl.cfg.top_k, exact["xc"])
            pre = O.forward(olayer, x_bits(xt), idx=idx, act_terms=1, x_in=x_in)
            h_in, other_h = validated_one_term_hidden(layer, T, pre["h_pre"])
            emu = O.forward(olayer, x_bits(xt), idx=idx, act_terms=1, x_in=x_in, h_in=h_in)
            check_expert_io(layer, T, wl.cfg.top_k, emu["x_in"], emu["h"], 1, label=f"{wl.name} T={T}")
            assert_delta_close(got, emu["delta"], got32,
                               label=f"{wl.name} T={T} vs 1-term emulation (other valid encodings: "
                                     f"{other:.1e} of x, {other_h:.1e} of h)")
            rel = rel_l2_per_token(got32, exact["delta"]).max()
            print(f"{wl.name} T={T}: rel-L2 max {rel:.3e} against the exact oracle")
            assert rel <= 0.125
        a = layer.lmoe_forward(x).cpu()
        b = layer.lmoe_forward(x).cpu()
        assert torch.equal(a, b)
    finally:
        layer.close()


def test_one_term_small_batch_k_split():
    """Kimi-K3 shapes at 2 tokens (K-split expert GEMMs) in the one-term mode."""
    wl = replace(C.workload("k3_decode_t64"), cfg=replace(C.K3, act_terms=1), name="k3_decode_mxfp8")
    W, x = gpu_inputs(wl)
    layer = make_layer(wl, W, max_tokens=wl.T)
    try:
        with OracleWorkers(wl, W) as workers:
            for T in (2, 64):
                full_size_check(wl, layer, oracle_layer(wl, W), workers, x[:T].contiguous(), act_terms=1)
    finally:
        layer.close()


def test_one_term_prefill_full_size():
    wl = C.workload("k3_prefill_t8192_mxfp8")
    W, x = gpu_inputs(wl)
    layer = make_layer(wl, W, max_tokens=wl.T)
    try:
        with OracleWorkers(wl, W) as workers:
            full_size_check(wl, layer, oracle_layer(wl, W), workers, x, act_terms=1)
    finally:
        layer.close()
