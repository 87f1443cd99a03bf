"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Each step of the hot path is checked on its own, then the whole layer:
  router logits and top-k (indices bit-exact except oracle-flagged near
  ties, where the GPU's choice must still be a valid top-k), dispatch
  (bit-exact), latent down-projection, expert sum u and u_hat, shared
  h, and Delta at the layer tolerances (per-token relative L2 <= 1e-2,
  max-abs <= 2e-2 * RMS(Delta)).
Workloads: the tiny layer, a mid-size layer whose every GEMM spans several
tiles with ragged tails (and K padding in the expert GEMMs), and every
full-size Kimi-K3 configuration: the decode batch (T = 64, seed 1), the
token-count sweep (T = 8 .. 2048, seed 4) and the Zipf-skewed prefill batch
(T = 8192, seed 2), each with every token's routing checked and Delta on
every token (T <= 16) or 16 sampled ones.  The max-abs bound applies to
Delta before its final bf16 rounding (the forward keeps that fp32 value as
a debug tensor); the bf16 output's own raw figure is printed beside it.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle as O
from lmoe_inputs import configs as C
from lmoe_inputs import generate as G
from tests._harness import (assert_delta_close, check_expert_io, forward_checked, gpu_inputs, make_layer,
                            oracle_layer, rel_l2_per_token, sample_tokens, valid_selection,
                            validated_one_term_hidden, validated_one_term_inputs, x_bits)
from tests._oracle_workers import OracleWorkers

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
    """Every token's selection against the oracle's: the same set of experts
    (bit-exact) unless the oracle flags the k-th / (k+1)-th biased scores as
    a near tie, where the GPU's set must still be a valid top-k; the GPU's
    order must be descending in biased score (selected experts whose scores
    lie within 1e-6 may come in either order); and each expert's weight must
    be the raw sigmoid renormalised over the GPU's own selection."""
    xb = x_bits(x)
    if tokens is not None:
        xb = xb[tokens]
        idx_gpu = idx_gpu[tokens]
        G_gpu = G_gpu[tokens]
    xo = O.bf16_bits_to_f64(xb)
    r = O.router(xo, olayer.dense("router_w"), olayer.W["router_bias"], wl.cfg.top_k, wl.cfg.routed_scale)
    G_own = O.weights_for(r["s"], np.asarray(idx_gpu, dtype=np.int64), wl.cfg.routed_scale)
    for t in range(xo.shape[0]):
        if r["flag"][t]:
            assert valid_selection(r["c"][t], idx_gpu[t]), t
        else:
            assert sorted(idx_gpu[t]) == sorted(r["idx"][t]), (t, idx_gpu[t], r["idx"][t])
        c_sel = r["c"][t][idx_gpu[t]]
        assert np.all(np.diff(c_sel) <= O.TIE_EPS), (t, idx_gpu[t], c_sel)
        assert np.allclose(G_gpu[t], G_own[t], rtol=2e-5, atol=1e-6), t
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
    got, got32, idx, Gw = forward_checked(layer, x)
    _check_routes(wl, layer, olayer, x, idx, Gw)
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
    assert_delta_close(got, ref["delta"], got32, label=f"{wl.name} T={T}")


def test_f32_output_leaves_the_bf16_output_unchanged(mid):
    """Keeping the fp32 Delta adds stores only: the bf16 output of a handle
    without it is bit-identical."""
    wl, W, x, layer, olayer = mid
    plain = make_layer(wl, W, max_tokens=256, keep_f32=False)
    try:
        a = plain.lmoe_forward(x).cpu()
        b = layer.lmoe_forward(x).cpu()
        plain.lmoe_sync_status()
        assert torch.equal(a, b)
        from latent_mixture_experts_gb300 import LmoeError
        with pytest.raises(LmoeError):
            plain.lmoe_debug_tensor("delta_f32", x.shape[0])
    finally:
        plain.close()


def test_ragged_T_and_edge_cases(mid):
    wl, W, x, layer, olayer = mid
    full = layer.lmoe_forward(x).cpu()
    for T in (1, 37):
        got, got32, idx, _ = forward_checked(layer, x[:T].contiguous())
        out = torch.from_numpy(got).to(torch.bfloat16)
        ref = O.forward(olayer, x_bits(x[:T]))
        assert_delta_close(got, ref["delta"], got32, label=f"{wl.name} T={T}")
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


def test_bounded_wait_reports_timeout(tiny):
    """A kernel waiting on a barrier nothing arrives at gives up after its
    limit: the next status check reports the timeout and clears it, and the
    handle keeps working."""
    wl, W, x, layer, olayer = tiny
    from latent_mixture_experts_gb300 import LmoeError, LMOE_ERR_INVALID_ARG, LMOE_ERR_TIMEOUT
    before = layer.lmoe_forward(x).cpu()
    layer.lmoe_sync_status()
    layer.lmoe_selftest_timeout(5_000)              # 5 us
    with pytest.raises(LmoeError) as ei:
        layer.lmoe_sync_status()
    assert ei.value.status == LMOE_ERR_TIMEOUT
    layer.lmoe_sync_status()                          # flag cleared
    assert torch.equal(layer.lmoe_forward(x).cpu(), before)
    layer.lmoe_sync_status()
    for bad in (10, 2_000_000_000):
        with pytest.raises(LmoeError) as ei:
            layer.lmoe_selftest_timeout(bad)
        assert ei.value.status == LMOE_ERR_INVALID_ARG


def full_size_check(wl, layer, olayer, workers, x, n_sample=16, seed=0, act_terms=None, io_tol=(2e-3, 5e-3)):
    """Every token's routing against the oracle (indices bit-exact, near
    ties flagged and checked for validity), then Delta on every token (T <=
    n_sample) or n_sample tokens including flagged ones and one on the most
    loaded expert, computed by the oracle with the GPU's selection."""
    T = x.shape[0]
    got, got32, idx, Gw = forward_checked(layer, x)
    r = _check_routes(wl, layer, olayer, x, idx, Gw)
    sample = sample_tokens(T, n_sample, r, idx, seed)
    x_in = h_in = None
    other = other_h = 0.0
    k = wl.cfg.top_k
    rows = (np.asarray(sample)[:, None] * k + np.arange(k)[None, :]).reshape(-1)
    if act_terms == 1:   # the oracle continues from the GPU's encodings once checked to be valid ones
        xe = O.bf16_bits_to_f64(x_bits(x)[sample]) @ olayer.dense("w_down_latent").T   # the oracle's x^c
        x_in, other = validated_one_term_inputs(layer, T, k, xe, rows=sample)
        pre = workers.forward(x_bits(x)[sample], idx[sample], act_terms=1, x_in=x_in, keep=("h_pre",))
        h_in, other_h = validated_one_term_hidden(layer, T, pre["h_pre"], rows=rows)
    ref = workers.forward(x_bits(x)[sample], idx[sample], act_terms=act_terms, keep=("delta", "x_in", "h"),
                          x_in=x_in, h_in=h_in)
    xin_full = np.zeros((T, ref["x_in"].shape[1]))
    xin_full[sample] = ref["x_in"]
    check_expert_io(layer, T, k, xin_full, ref["h"], act_terms or 2, rows=rows, label=f"{wl.name} T={T}",
                    tol=io_tol)
    assert_delta_close(got[sample], ref["delta"], got32[sample],
                       label=f"{wl.name} T={T} ({len(sample)} tokens, {int(r['flag'].sum())} flagged)"
                             + (f" vs the oracle emulating {act_terms}-term activations (other valid "
                                f"encodings: {other:.1e} of x, {other_h:.1e} of h)" if act_terms else ""))
    return got, idx, sample


@pytest.fixture(scope="module")
def k3_decode():
    wl = C.workload("k3_decode_t64")
    W, x = gpu_inputs(wl)
    layer = make_layer(wl, W, max_tokens=wl.T)
    workers = OracleWorkers(wl, W)
    yield wl, W, x, layer, oracle_layer(wl, W), workers
    workers.close()
    layer.close()
    del W
    torch.cuda.empty_cache()


def test_k3_decode_full_size(k3_decode):
    """Kimi-K3 shapes, T = 64, seed 1, in the launch configuration the
    benchmark times."""
    wl, W, x, layer, olayer, workers = k3_decode
    full_size_check(wl, layer, olayer, workers, x)


@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_k3_small_batch_k_split(k3_decode, T):
    """Kimi-K3 shapes at 1-4 tokens, where the expert GEMMs split each
    weight-row item's K range across CTAs (gate/up partials finished by the
    last split to arrive, down partials added by the combine): every token
    against the oracle, and repeated forwards bit-identical (the partials are
    added in split order whatever the arrival order)."""
    wl, W, x, layer, olayer, workers = k3_decode
    xs = x[:T].contiguous()
    got, idx, _ = full_size_check(wl, layer, olayer, workers, xs)
    again = layer.lmoe_forward(xs)
    torch.cuda.synchronize()
    assert np.array_equal(again.cpu().double().numpy(), got)


@pytest.fixture(scope="module")
def k3_sweep():
    """The token-count sweep configuration: Kimi-K3 shapes, seed 4, uniform
    bias; one layer serves every T (the tokens of a smaller T are the first
    rows of the largest batch)."""
    wl = C.workload("k3_sweep_t2048")
    W, x = gpu_inputs(wl)
    layer = make_layer(wl, W, max_tokens=wl.T)
    workers = OracleWorkers(wl, W)
    yield wl, W, x, layer, oracle_layer(wl, W), workers
    workers.close()
    layer.close()
    del W
    torch.cuda.empty_cache()


@pytest.mark.parametrize("T", [8, 32, 128, 512, 2048])
def test_k3_sweep_full_size(k3_sweep, T):
    wl, W, x, layer, olayer, workers = k3_sweep
    assert torch.equal(x[:T].cpu(), G.gen_x(C.workload(f"k3_sweep_t{T}"), "cpu"))
    full_size_check(replace(wl, T=T, name=f"k3_sweep_t{T}"), layer, olayer, workers, x[:T].contiguous(), seed=T)


def test_k3_prefill_full_size():
    """T = 8192 with the Zipf-skewed bias (seed 2): every token's routing,
    Delta on 16 sampled tokens (flagged ones and one on the most loaded
    expert among them)."""
    wl = C.workload("k3_prefill_t8192")
    W, x = gpu_inputs(wl)
    layer = make_layer(wl, W, max_tokens=wl.T)
    try:
        with OracleWorkers(wl, W) as workers:
            full_size_check(wl, layer, oracle_layer(wl, W), workers, x)
    finally:
        layer.close()
