"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Each step of the hot path is checked on its own, then the whole layer:
  router logits and top-k (indices bit-exact except oracle-flagged near
  ties, where the GPU's choice must still be a valid top-k), dispatch
  (bit-exact), latent down-projection, expert sum u and u_hat, shared
  h, and Delta at the layer tolerances (per-token relative L2 <= 1e-2,
  max-abs <= 2e-2 * RMS(Delta)).
Workloads: the tiny layer, a mid-size layer whose every GEMM spans several
tiles with ragged tails (and K padding in the expert GEMMs), the full
Kimi-K3 decode batch and the full prefill batch (sampled tokens).
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle as O
from lmoe_inputs import configs as C
from lmoe_inputs import generate as G
from tests._harness import (assert_delta_close, gpu_inputs, make_layer, oracle_layer, rel_l2_per_token,
                            valid_selection, x_bits)

pytestmark = pytest.mark.gpu

MID = C.Workload("k3_mid_t200", C.K3_MID, T=200, seed=21)


@pytest.fixture(scope="module")
def tiny():
    wl = C.workload("k3_tiny_t16")
    W, x = gpu_inputs(wl)
    layer = make_layer(wl, W, max_tokens=64)
    return wl, W, x, layer, oracle_layer(wl, W)


@pytest.fixture(scope="module")
def mid():
    W, x = gpu_inputs(MID)
    layer = make_layer(MID, W, max_tokens=256)
    return MID, W, x, layer, oracle_layer(MID, W)


def _check_routes(wl, layer, olayer, x, idx_gpu, G_gpu, tokens=None):
    xb = x_bits(x)
    if tokens is not None:
        xb = xb[tokens]
        idx_gpu = idx_gpu[tokens]
        G_gpu = G_gpu[tokens]
    xo = O.bf16_bits_to_f64(xb)
    r = O.router(xo, olayer.dense("router_w"), olayer.W["router_bias"], wl.cfg.top_k, wl.cfg.routed_scale)
    for t in range(xo.shape[0]):
        if r["flag"][t]:
            assert valid_selection(r["c"][t], idx_gpu[t]), t
        else:
            assert list(idx_gpu[t]) == list(r["idx"][t]), (t, idx_gpu[t], r["idx"][t])
            assert np.allclose(G_gpu[t], r["G"][t], rtol=2e-5, atol=1e-6)
    return r


@pytest.mark.parametrize("which", ["tiny", "mid"])
def test_router_and_topk(which, request):
    wl, W, x, layer, olayer = request.getfixturevalue(which)
    idx, Gw = layer.lmoe_route(x)
    torch.cuda.synchronize()
    _check_routes(wl, layer, olayer, x, idx.cpu().numpy(), Gw.cpu().numpy())


@pytest.mark.parametrize("which", ["tiny", "mid"])
def test_router_logits(which, request):
    wl, W, x, layer, olayer = request.getfixturevalue(which)
    layer.lmoe_forward(x)
    z = layer.lmoe_debug_tensor("logits", x.shape[0]).cpu().double().numpy()
    zo = O.bf16_bits_to_f64(x_bits(x)) @ olayer.dense("router_w").T
    assert np.abs(z - zo).max() <= 2e-5 * (1 + np.abs(zo).max())


def test_dispatch_bit_exact_random():
    wl = C.workload("k3_tiny_t16")
    W, x = gpu_inputs(wl)
    rng = np.random.default_rng(0)
    for E, T, k in [(64, 16, 2), (64, 300, 2), (64, 1, 2)]:
        idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
        layer = make_layer(wl, W, max_tokens=max(T, 16))
        counts, offsets, perm = layer.lmoe_dispatch(torch.from_numpy(idx).cuda())
        torch.cuda.synchronize()
        d = O.dispatch(idx, E)
        assert np.array_equal(counts.cpu().numpy(), d["counts"])
        assert np.array_equal(offsets.cpu().numpy(), d["offsets"])
        assert np.array_equal(perm.cpu().numpy(), d["perm"])
        layer.lmoe_sync_status()
        layer.close()


def test_dispatch_skewed_and_full_size():
    """All tokens on the same few experts; and a Kimi-K3-sized assignment set
    (T = 2048, k = 16, E = 896) spanning many counting chunks."""
    wl = C.workload("k3_tiny_t16")
    W, x = gpu_inputs(wl)
    rng = np.random.default_rng(1)
    layer = make_layer(wl, W, max_tokens=4096)
    idx = np.tile(np.array([[5, 9]], dtype=np.int32), (4096, 1))
    counts, offsets, perm = layer.lmoe_dispatch(torch.from_numpy(idx).cuda())
    d = O.dispatch(idx, 64)
    assert np.array_equal(perm.cpu().numpy(), d["perm"]) and np.array_equal(counts.cpu().numpy(), d["counts"])
    layer.close()
    # full-size routing table through a K3-shaped dispatch (no weights needed beyond the tiny layer's)
    E, T, k = 896, 2048, 16
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    big = C.Workload("dispatch_only", replace(C.K3_TINY, n_experts=E, top_k=k), T=T, seed=5)
    Wb, _ = gpu_inputs(big, T=1)
    layer = make_layer(big, Wb, max_tokens=T)
    counts, offsets, perm = layer.lmoe_dispatch(torch.from_numpy(idx).cuda())
    d = O.dispatch(idx, E)
    assert np.array_equal(counts.cpu().numpy(), d["counts"])
    assert np.array_equal(offsets.cpu().numpy(), d["offsets"])
    assert np.array_equal(perm.cpu().numpy(), d["perm"])
    layer.close()


def test_dispatch_rejects_out_of_range_expert(tiny):
    wl, W, x, layer, olayer = tiny
    idx = torch.tensor([[0, 64], [1, 2]], dtype=torch.int32, device="cuda")
    layer.lmoe_dispatch(idx)
    from latent_mixture_experts_gb300 import LmoeError, LMOE_ERR_INVALID_ARG
    with pytest.raises(LmoeError) as ei:
        layer.lmoe_sync_status()
    assert ei.value.status == LMOE_ERR_INVALID_ARG
    layer.lmoe_sync_status()   # flag cleared


@pytest.mark.parametrize("which", ["tiny", "mid"])
def test_steps_and_layer(which, request):
    wl, W, x, layer, olayer = request.getfixturevalue(which)
    T = x.shape[0]
    out, idx, Gw = layer.lmoe_forward(x, return_routing=True)
    torch.cuda.synchronize()
    layer.lmoe_sync_status()
    idx = idx.cpu().numpy()
    _check_routes(wl, layer, olayer, x, idx, Gw.cpu().numpy())
    ref = O.forward(olayer, x_bits(x), idx=idx)          # oracle run with the GPU's selection
    # latent down-projection (fp32 accumulation of bf16 products)
    xc = layer.lmoe_debug_tensor("xc", T).cpu().double().numpy()
    assert np.abs(xc - ref["xc"]).max() <= 1e-4 * (1 + np.abs(ref["xc"]).max())
    # dispatch of this forward
    d = O.dispatch(idx, wl.cfg.n_experts)
    assert np.array_equal(layer.lmoe_debug_tensor("perm", T).cpu().numpy(), d["perm"])
    assert np.array_equal(layer.lmoe_debug_tensor("offsets", T).cpu().numpy(), d["offsets"])
    # expert sum and its norm
    u = layer.lmoe_debug_tensor("u", T).cpu().double().numpy()
    assert rel_l2_per_token(u, ref["u"]).max() <= 1e-2
    uh = layer.lmoe_debug_tensor("u_hat", T).cpu().double().numpy()
    assert rel_l2_per_token(uh, ref["u_hat"]).max() <= 1e-2
    # shared experts
    hs = layer.lmoe_debug_tensor("h_shared", T).cpu().double().numpy()
    assert rel_l2_per_token(hs, ref["h_s"]).max() <= 1e-2
    # the layer
    assert_delta_close(out.cpu().double().numpy(), ref["delta"])


def test_ragged_T_and_edge_cases(mid):
    wl, W, x, layer, olayer = mid
    full = layer.lmoe_forward(x).cpu()
    for T in (1, 37):
        out = layer.lmoe_forward(x[:T].contiguous())
        torch.cuda.synchronize()
        ref = O.forward(olayer, x_bits(x[:T]))
        assert_delta_close(out.cpu().double().numpy(), ref["delta"])
        # per-token independence: the first T rows do not depend on the others
        assert torch.equal(out.cpu(), full[:T]) or \
            rel_l2_per_token(out.cpu().double().numpy(), full[:T].double().numpy()).max() < 1e-2
    empty = torch.empty(0, wl.cfg.d_model, dtype=torch.bfloat16, device="cuda")
    assert layer.lmoe_forward(empty).shape == (0, wl.cfg.d_model)
    from latent_mixture_experts_gb300 import LmoeError
    too_many = torch.zeros(257, wl.cfg.d_model, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(LmoeError):
        layer.lmoe_forward(too_many)


def test_deterministic_and_host_path(mid):
    wl, W, x, layer, olayer = mid
    a = layer.lmoe_forward(x).cpu()
    b = layer.lmoe_forward(x).cpu()
    assert torch.equal(a, b)
    xh = x.cpu().pin_memory()
    oh = torch.empty(x.shape[0], wl.cfg.d_model, dtype=torch.bfloat16).pin_memory()
    layer.lmoe_forward_host(xh, oh)
    assert torch.equal(oh, a)


def test_stage_timing_period(mid):
    """Stage timing records one event pair per timed call and stage: with a
    period of 3, forwards 0, 3 and 6 of seven; outputs are unchanged by it."""
    wl, W, x, layer, olayer = mid
    ref = layer.lmoe_forward(x).cpu()
    layer.lmoe_set_profiling(8, stages=["expert_gate_up", "combine_norm"])
    layer.lmoe_set_profiling_period(3)
    for _ in range(7):
        out = layer.lmoe_forward(x)
    prof = layer.lmoe_profile_get()
    assert prof["expert_gate_up"][1] == 3 and prof["combine_norm"][1] == 3
    assert prof["expert_down"][1] == 0
    assert prof["expert_gate_up"][0] > 0
    assert torch.equal(out.cpu(), ref)
    with pytest.raises(RuntimeError):
        layer.lmoe_set_profiling_period(0)
    layer.lmoe_set_profiling_period(1)
    layer.lmoe_set_profiling(0)
    layer.lmoe_sync_status()


def test_generator_bytes_match_cpu():
    wl = C.workload("k3_decode_t64")
    for name, e in (("ex_gate", 0), ("ex_down", 895)):
        qc, sc = G.gen_expert(wl, name, e, "cpu")
        qg, sg = G.gen_expert(wl, name, e, "cuda")
        assert torch.equal(qc, qg.cpu()) and torch.equal(sc, sg.cpu())
    assert torch.equal(G.gen_x(wl, "cpu"), G.gen_x(wl, "cuda").cpu())


@pytest.fixture(scope="module")
def k3_decode():
    wl = C.workload("k3_decode_t64")
    W, x = gpu_inputs(wl)
    layer = make_layer(wl, W, max_tokens=wl.T)
    yield wl, W, x, layer, oracle_layer(wl, W)
    layer.close()
    del W
    torch.cuda.empty_cache()


def test_k3_decode_full_size(k3_decode):
    """Kimi-K3 shapes, T = 64, in the launch configuration the benchmark
    times: routing of every token against the oracle, Delta on sampled
    tokens the oracle computes one by one."""
    wl, W, x, layer, olayer = k3_decode
    out, idx, Gw = layer.lmoe_forward(x, return_routing=True)
    torch.cuda.synchronize()
    layer.lmoe_sync_status()
    idx = idx.cpu().numpy()
    _check_routes(wl, layer, olayer, x, idx, Gw.cpu().numpy())
    sample = [0, 17, 42, 63]
    ref = O.forward(olayer, x_bits(x)[sample], idx=idx[sample])
    assert_delta_close(out.cpu().double().numpy()[sample], ref["delta"])


@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_k3_small_batch_k_split(k3_decode, T):
    """Kimi-K3 shapes at 1-4 tokens, where the expert GEMMs split each
    weight-row item's K range across CTAs (gate/up partials finished by the
    last split to arrive, down partials added by the combine): every token
    against the oracle, and repeated forwards bit-identical (the partials are
    added in split order whatever the arrival order)."""
    wl, W, x, layer, olayer = k3_decode
    xs = x[:T].contiguous()
    out, idx, Gw = layer.lmoe_forward(xs, return_routing=True)
    again = layer.lmoe_forward(xs)
    torch.cuda.synchronize()
    layer.lmoe_sync_status()
    assert torch.equal(out, again)
    idx = idx.cpu().numpy()
    _check_routes(wl, layer, olayer, xs, idx, Gw.cpu().numpy())
    ref = O.forward(olayer, x_bits(xs), idx=idx)
    assert_delta_close(out.cpu().double().numpy(), ref["delta"])


def test_k3_prefill_full_size():
    """T = 8192 with the Zipf-skewed bias: every token's routing checked
    for validity, sampled tokens (one on the most loaded expert) against
    the oracle."""
    wl = C.workload("k3_prefill_t8192")
    W, x = gpu_inputs(wl)
    layer = make_layer(wl, W, max_tokens=wl.T)
    olayer = oracle_layer(wl, W)
    out, idx, Gw = layer.lmoe_forward(x, return_routing=True)
    torch.cuda.synchronize()
    layer.lmoe_sync_status()
    idx = idx.cpu().numpy()
    counts = np.bincount(idx.reshape(-1), minlength=wl.cfg.n_experts)
    hot = int(np.argmax(counts))
    t_hot = int(np.nonzero((idx == hot).any(1))[0][0])
    sample = sorted({0, 4095, 8191, t_hot})
    _check_routes(wl, layer, olayer, x, idx, Gw.cpu().numpy(), tokens=sample)
    ref = O.forward(olayer, x_bits(x)[sample], idx=idx[sample])
    assert_delta_close(out.cpu().double().numpy()[sample], ref["delta"])
    layer.close()
