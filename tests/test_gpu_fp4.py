"""The packed 4-bit expert GEMMs (act_format e2m1: MXFP4 weights as stored x
activations as three MXFP4 terms, tcgen05 kind::mxf4 with E8M0 scales per
32) against the fp64 oracle at the layer tolerances (per-token relative L2
<= 1e-2, max-abs <= 2e-2 RMS on Delta before its bf16 rounding).

Every token tile (16 and 32 with 256-row weight items, 64 and 96 with
128-row items), K padded to the 256-value groups of packed rows (tiny l = 320,
mid l = 704 and F = 608), the K split of one- to four-token batches, and the
full Kimi-K3 decode and prefill batches.  The expert inputs and hidden
activations the MMAs multiply are checked per assignment against the exact
values (three E2M1 terms hold them to ~1e-3) and the E2M1 emulation of the
oracle is printed beside."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle as O
from lmoe_inputs import configs as C
from tests._harness import (assert_delta_close, check_expert_io, forward_checked, gpu_inputs, make_layer,
                            oracle_layer, rel_l2_per_token, x_bits)
from tests._oracle_workers import OracleWorkers
from tests.test_gpu_parity import full_size_check

pytestmark = pytest.mark.gpu

E2M1 = dict(act_format="e2m1", act_terms=3)
TILES = [(C.Workload("k3_tiny_fp4", replace(C.K3_TINY, **E2M1), T=3001, seed=51), (3, 100, 400, 1500, 3001)),
         (C.Workload("k3_mid_fp4", replace(C.K3_MID, **E2M1), T=1800, seed=52), (37, 1000, 1800))]
IO_TOL = (5e-3, 1e-2)   # per-row rel-L2 of three E2M1 terms against the exact inputs / hidden activations


@pytest.mark.parametrize("wl,Ts", TILES, ids=[c[0].name for c in TILES])
def test_fp4_all_tiles(wl, Ts):
    W, x = gpu_inputs(wl)
    layer = make_layer(wl, W, max_tokens=wl.T)
    olayer = oracle_layer(wl, W)
    try:
        for T in Ts:
            xt = x[:T].contiguous()
            got, got32, idx, _ = forward_checked(layer, xt)
            ref = O.forward(olayer, x_bits(xt), idx=idx)
            check_expert_io(layer, T, wl.cfg.top_k, ref["x_in"], ref["h"], 3, label=f"{wl.name} T={T}", tol=IO_TOL)
            assert_delta_close(got, ref["delta"], got32, label=f"{wl.name} T={T}")
            emu = O.forward(olayer, x_bits(xt), idx=idx, act_terms=3, act_format="e2m1")
            print(f"{wl.name} T={T}: rel-L2 max {rel_l2_per_token(got32, emu['delta']).max():.3e} "
                  "against the oracle emulating three E2M1 terms")
        a = layer.lmoe_forward(x).cpu()
        b = layer.lmoe_forward(x).cpu()
        assert torch.equal(a, b)
    finally:
        layer.close()


@pytest.fixture(scope="module")
def k3_fp4():
    wl = replace(C.workload("k3_decode_t64"), cfg=replace(C.K3, **E2M1), name="k3_decode_fp4")
    W, x = gpu_inputs(wl)
    layer = make_layer(wl, W, max_tokens=wl.T)
    workers = OracleWorkers(wl, W)
    yield wl, W, x, layer, oracle_layer(wl, W), workers
    workers.close()
    layer.close()
    del W
    torch.cuda.empty_cache()


@pytest.mark.parametrize("T", [1, 2, 4, 64])
def test_fp4_k3_decode(k3_fp4, T):
    """Kimi-K3 shapes: 1-4 tokens run the K-split form, 64 the decode batch."""
    wl, W, x, layer, olayer, workers = k3_fp4
    xs = x[:T].contiguous()
    got, idx, _ = full_size_check(wl, layer, olayer, workers, xs, io_tol=IO_TOL)
    again = layer.lmoe_forward(xs)
    torch.cuda.synchronize()
    assert np.array_equal(again.cpu().double().numpy(), got)


def test_fp4_k3_prefill():
    wl = replace(C.workload("k3_prefill_t8192"), cfg=replace(C.K3, **E2M1), name="k3_prefill_fp4")
    W, x = gpu_inputs(wl)
    layer = make_layer(wl, W, max_tokens=wl.T)
    try:
        with OracleWorkers(wl, W) as workers:
            full_size_check(wl, layer, oracle_layer(wl, W), workers, x, io_tol=IO_TOL)
    finally:
        layer.close()
