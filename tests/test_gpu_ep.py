"""Expert parallelism through the library's device phases (lmoe_ep_dispatch,
lmoe_ep_experts, lmoe_ep_combine) against the fp64 oracle.

On one GPU, R ranks are emulated by R handles, each holding its contiguous
range of E / R experts and its own tokens: every phase runs for all ranks,
and the host moves the buffers between phases the way the all-to-alls
would (counts: each rank's slice of every source's counts, source-major;
rows: each source's block for each rank, in rank order; then back).  No
kernel waits on another rank's.  Each rank's Delta must meet the layer
tolerances against the oracle's forward of its tokens with all experts."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle as O
from lmoe_inputs import configs as C
from lmoe_inputs import generate as G
from latent_mixture_experts_gb300.expert_parallel import ep_forward, local_experts
from tests._harness import assert_delta_close, built_library, gpu_inputs, oracle_layer, x_bits

pytestmark = pytest.mark.gpu

CASES = [("k3_tiny_t16", C.K3_TINY, 2), ("k3_tiny_t16", C.K3_TINY, 4), ("k3_mid", C.K3_MID, 2),
         ("k2_small", replace(C.K2, d_model=1024, n_experts=48, top_k=4, d_expert_ff=384, d_shared_ff=256), 2)]


def _handles(wl, W, R, Tm):
    from latent_mixture_experts_gb300 import LatentMoE
    built_library()
    locs = [local_experts(W, r, R) for r in range(R)]
    layers = [LatentMoE(wl.cfg, locs[r], max_tokens=Tm, ep_size=R, ep_rank=r) for r in range(R)]
    for layer in layers:
        layer.lmoe_keep_f32_output(True)
    return layers, locs


def emulated_ep(layers, xs):
    """The phases of every rank with the exchanges done by the host."""
    R = len(layers)
    sends, counts = zip(*[layers[r].lmoe_ep_dispatch(xs[r]) for r in range(R)])
    E = counts[0].numel()
    El = E // R
    splits = [c.view(R, El).sum(1).tolist() for c in counts]           # splits[s][r]: rows s -> r
    starts = [np.concatenate([[0], np.cumsum(sp)]) for sp in splits]
    outs = []
    for r in range(R):
        rc = torch.stack([counts[s][r * El:(r + 1) * El] for s in range(R)])
        recv = torch.cat([sends[s][starts[s][r]:starts[s][r + 1]] for s in range(R)])
        outs.append(layers[r].lmoe_ep_experts(recv.contiguous(), rc.contiguous()))
    deltas = []
    for s in range(R):
        pieces, off = [], [0] * R
        for r in range(R):
            before = sum(splits[q][r] for q in range(s))                # rows of earlier sources in r's receive
            pieces.append(outs[r][before:before + splits[s][r]])
        ret = torch.cat(pieces).contiguous()
        deltas.append(layers[s].lmoe_ep_combine(ret, xs[s].shape[0]))
    torch.cuda.synchronize()
    for layer in layers:
        layer.lmoe_sync_status()
    d32 = [layers[s].lmoe_debug_tensor("delta_f32", xs[s].shape[0]).cpu().double().numpy() for s in range(R)]
    return deltas, d32


@pytest.mark.parametrize("name,cfg,R", CASES, ids=[f"{c[0]}_R{c[2]}" for c in CASES])
def test_expert_parallel_ranks_match_oracle(name, cfg, R):
    wl = C.Workload(name, cfg, T=24, seed=71)
    W, _ = gpu_inputs(wl, T=1)
    layers, _ = _handles(wl, W, R, Tm=wl.T)
    olayer = oracle_layer(wl, W)
    try:
        xs = [G.gen_x(replace(wl, seed=wl.seed + 13 * r), device="cuda", T=wl.T - 5 * r) for r in range(R)]
        deltas, d32 = emulated_ep(layers, xs)
        for r in range(R):
            ref = O.forward(olayer, x_bits(xs[r]))
            assert_delta_close(deltas[r].cpu().double().numpy(), ref["delta"], d32[r],
                               label=f"{name} R={R} rank {r}")
        again, _ = emulated_ep(layers, xs)
        assert all(torch.equal(a, b) for a, b in zip(deltas, again))
    finally:
        for layer in layers:
            layer.close()


def test_single_rank_phases_match_forward():
    """ep_size 1: the three phases (no exchange) against lmoe_forward of a
    plain handle on the same tokens (bf16 transport of the latent rows and
    of the expert outputs is their only difference)."""
    from latent_mixture_experts_gb300 import LatentMoE
    wl = C.workload("k3_tiny_t16")
    W, x = gpu_inputs(wl)
    built_library()
    ep = LatentMoE(wl.cfg, W, max_tokens=wl.T, ep_size=1)
    plain = LatentMoE(wl.cfg, W, max_tokens=wl.T)
    try:
        a = ep_forward(ep, x).cpu().double().numpy()
        b = plain.lmoe_forward(x).cpu().double().numpy()
        ref = O.forward(oracle_layer(wl, W), x_bits(x))
        assert_delta_close(a, ref["delta"], label="ep_size 1 phases")
        assert np.abs(a - b).max() <= 2e-2 * np.sqrt((b ** 2).mean())
        from latent_mixture_experts_gb300 import LmoeError
        two = LatentMoE(wl.cfg, local_experts(W, 0, 2), max_tokens=wl.T, ep_size=2, ep_rank=0)
        with pytest.raises(LmoeError):
            two.lmoe_forward(x)                       # an expert-parallel handle runs the phases only
        two.close()
    finally:
        ep.close()
        plain.close()
