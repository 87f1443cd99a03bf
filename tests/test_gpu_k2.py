"""Parity of the non-latent FP8 path (Kimi K2 card: 384 experts, top-8, routed
scale 2.827, SwiGLU experts on the full width, one shared expert, FP8 E4M3
weights with fp32 scales per 128 x 128 block) with the fp64 oracle.

A small K2-shaped layer is checked step by step and as a whole; the full K2
workload (T = 4096) is checked on every token's routing and on 16 sampled
tokens' outputs."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle as O
from lmoe_inputs import configs as C
from tests._harness import (assert_delta_close, forward_checked, gpu_inputs, make_layer, oracle_layer,
                            rel_l2_per_token, x_bits)
from tests._oracle_workers import OracleWorkers
from tests.test_gpu_parity import _check_routes, full_size_check

pytestmark = pytest.mark.gpu

K2_SMALL = C.Workload("k2_small_t50", replace(C.K2, d_model=1024, n_experts=48, top_k=4, d_expert_ff=384,
                                              d_shared_ff=256), T=50, seed=31)


@pytest.fixture(scope="module")
def k2_small():
    W, x = gpu_inputs(K2_SMALL)
    layer = make_layer(K2_SMALL, W, max_tokens=64)
    return K2_SMALL, W, x, layer, oracle_layer(K2_SMALL, W)


def test_k2_small_steps_and_layer(k2_small):
    wl, W, x, layer, olayer = k2_small
    T = x.shape[0]
    got, got32, idx, Gw = forward_checked(layer, x)
    r = _check_routes(wl, layer, olayer, x, idx, Gw)
    assert np.allclose(r["G"].sum(1), 2.827)
    ref = O.forward(olayer, x_bits(x), idx=idx)
    d = O.dispatch(idx, wl.cfg.n_experts)
    assert np.array_equal(layer.lmoe_debug_tensor("perm", T).cpu().numpy(), d["perm"])
    u = layer.lmoe_debug_tensor("u", T).cpu().double().numpy()      # y_routed: no latent, no norm
    assert rel_l2_per_token(u, ref["y_routed"]).max() <= 1e-2
    ys = layer.lmoe_debug_tensor("y_shared", T).cpu().double().numpy()   # shared expert on the FP8 GEMMs
    assert rel_l2_per_token(ys, ref["y_shared"]).max() <= 1e-2
    assert_delta_close(got, ref["delta"], got32, label=f"{wl.name} T={T}")


def test_k2_small_token_tiles(k2_small):
    """T = 1 (16-assignment tiles) and T = 50 with 32-token tiles agree with
    the oracle; repeated forwards are bit-identical."""
    wl, W, x, layer, olayer = k2_small
    for T in (1, 7):
        got, got32, _, _ = forward_checked(layer, x[:T].contiguous())
        ref = O.forward(olayer, x_bits(x[:T]))
        assert_delta_close(got, ref["delta"], got32, label=f"{wl.name} T={T}")
    a = layer.lmoe_forward(x).cpu()
    b = layer.lmoe_forward(x).cpu()
    assert torch.equal(a, b)


def test_k2_full_size():
    """The K2 workload (T = 4096, seed 3): every token's routing, Delta on 16
    sampled tokens."""
    wl = C.workload("k2_t4096")
    W, x = gpu_inputs(wl)
    layer = make_layer(wl, W, max_tokens=wl.T)
    try:
        with OracleWorkers(wl, W) as workers:
            full_size_check(wl, layer, oracle_layer(wl, W), workers, x)
    finally:
        layer.close()
