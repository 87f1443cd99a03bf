"""Parity of the non-latent FP8 path (Kimi K2 card: 384 experts, top-8, routed
scale 2.827, SwiGLU experts on the full width, one shared expert, FP8 E4M3
weights with fp32 scales per 128 x 128 block) with the fp64 oracle.

A small K2-shaped layer is checked step by step and as a whole; the full K2
workload (T = 4096) is checked on every token's routing and on sampled
tokens' outputs."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle as O
from lmoe_inputs import configs as C
from tests._harness import assert_delta_close, gpu_inputs, make_layer, oracle_layer, rel_l2_per_token, x_bits
from tests.test_gpu_parity import _check_routes

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
    out, idx, Gw = layer.lmoe_forward(x, return_routing=True)
    torch.cuda.synchronize()
    layer.lmoe_sync_status()
    idx = idx.cpu().numpy()
    r = _check_routes(wl, layer, olayer, x, idx, Gw.cpu().numpy())
    assert np.allclose(r["G"].sum(1), 2.827)
    ref = O.forward(olayer, x_bits(x), idx=idx)
    d = O.dispatch(idx, wl.cfg.n_experts)
    assert np.array_equal(layer.lmoe_debug_tensor("perm", T).cpu().numpy(), d["perm"])
    u = layer.lmoe_debug_tensor("u", T).cpu().double().numpy()      # y_routed: no latent, no norm
    assert rel_l2_per_token(u, ref["y_routed"]).max() <= 1e-2
    ys = layer.lmoe_debug_tensor("y_shared", T).cpu().double().numpy()   # shared expert on the FP8 GEMMs
    assert rel_l2_per_token(ys, ref["y_shared"]).max() <= 1e-2
    assert_delta_close(out.cpu().double().numpy(), ref["delta"])


def test_k2_small_token_tiles(k2_small):
    """T = 1 (16-assignment tiles) and T = 50 with 32-token tiles agree with
    the oracle; repeated forwards are bit-identical."""
    wl, W, x, layer, olayer = k2_small
    for T in (1, 7):
        out = layer.lmoe_forward(x[:T].contiguous())
        ref = O.forward(olayer, x_bits(x[:T]))
        assert_delta_close(out.cpu().double().numpy(), ref["delta"])
    a = layer.lmoe_forward(x).cpu()
    b = layer.lmoe_forward(x).cpu()
    assert torch.equal(a, b)


def test_k2_full_size():
    wl = C.workload("k2_t4096")
    W, x = gpu_inputs(wl)
    layer = make_layer(wl, W, max_tokens=wl.T)
    olayer = oracle_layer(wl, W)
    out, idx, Gw = layer.lmoe_forward(x, return_routing=True)
    torch.cuda.synchronize()
    layer.lmoe_sync_status()
    idx = idx.cpu().numpy()
    sample = [0, 1000, 2047, 4095]
    _check_routes(wl, layer, olayer, x, idx, Gw.cpu().numpy(), tokens=sample)
    ref = O.forward(olayer, x_bits(x)[sample], idx=idx[sample])
    assert_delta_close(out.cpu().double().numpy()[sample], ref["delta"])
    layer.close()
