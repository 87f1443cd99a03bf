"""Quantile Balancing on the GPU (lmoe_qb_update, lmoe_qb_histogram,
lmoe_qb_update_from_histogram) against the fp64 oracle on the same fp32
router logits.

The exact update is compared as values (the GPU works in fp32, so a
quantile between two required biases closer than ~1e-7 may resolve to
either); the histogram counts are integers decided by fp32 comparisons
against the bin edges, so they are checked edge by edge: the GPU's count
below each edge must lie between the oracle's counts below the edge minus
and plus 1e-5.  The update read from the histogram is compared on the GPU's
own counts."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle as O
from lmoe_inputs import configs as C
from tests._harness import gpu_inputs, make_layer

pytestmark = pytest.mark.gpu

SHAPES = [(896, 16, 4096), (64, 2, 1000), (384, 8, 8192), (896, 16, 1)]


@pytest.fixture(scope="module", params=SHAPES, ids=[f"E{e}_k{k}_T{t}" for e, k, t in SHAPES])
def qb_case(request):
    E, k, T = request.param
    wl = C.Workload("qb_layer", replace(C.K3_TINY, n_experts=E, top_k=k), T=max(T, 16), seed=61)
    W, _ = gpu_inputs(wl, T=1)
    layer = make_layer(wl, W, max_tokens=max(T, 16), keep_f32=False)
    g = torch.Generator(device="cuda").manual_seed(E + T)
    z = (torch.randn(T, E, device="cuda", generator=g) * 1.5).contiguous()
    bias = ((torch.rand(E, device="cuda", generator=g) - 0.5) * 0.2).contiguous()
    yield E, k, T, layer, z, bias
    layer.close()


def _scores(z):
    return 1.0 / (1.0 + np.exp(-z.cpu().double().numpy()))


def test_exact_update(qb_case):
    E, k, T, layer, z, bias = qb_case
    nb = layer.lmoe_qb_update(T, logits=z, bias=bias)
    torch.cuda.synchronize()
    layer.lmoe_sync_status()
    ref = O.qb_update(_scores(z), bias.cpu().double().numpy(), k)
    got = nb.cpu().double().numpy()
    assert np.abs(got - ref["bias"]).max() <= 2e-6, np.abs(got - ref["bias"]).max()
    assert abs(got.mean()) <= 1e-6


def test_histogram_counts_and_update(qb_case):
    E, k, T, layer, z, bias = qb_case
    B = 1000
    counts = torch.zeros(E, B, dtype=torch.int32, device="cuda")
    layer.lmoe_qb_histogram(T, counts, logits=z, bias=bias)
    nb = layer.lmoe_qb_update_from_histogram(counts, bias=bias)
    torch.cuda.synchronize()
    layer.lmoe_sync_status()
    h = counts.cpu().numpy().astype(np.int64)
    assert np.all(h.sum(1) == T)
    b64 = bias.cpu().double().numpy()
    r = O.qb_required_bias(_scores(z), b64, k)
    lo, hi = O.qb_range(b64)
    edges = lo + (hi - lo) / B * np.arange(1, B)
    below = np.cumsum(h, axis=1)[:, :-1]                     # GPU count below each inner edge
    eps = 1e-5
    for j in range(E):
        rs = np.sort(r[:, j])
        lo_n = np.searchsorted(rs, edges - eps, side="left")
        hi_n = np.searchsorted(rs, edges + eps, side="right")
        assert np.all(below[j] >= lo_n) and np.all(below[j] <= hi_n), j
    ref = O.qb_update_from_histogram(h, b64, k)
    got = nb.cpu().double().numpy()
    assert np.abs(got - ref["bias"]).max() <= 2e-6, np.abs(got - ref["bias"]).max()
    # the estimator's error bound against the exact update (one bin plus one order-statistic gap)
    if T >= 1000:
        exact = O.qb_update(_scores(z), b64, k)
        rsort = np.sort(r, axis=0)
        tgt = -(-(T * k) // E)
        gap = rsort[min(tgt, T - 1)] - rsort[tgt - 1]
        assert np.all(np.abs(ref["raw"] - exact["raw"]) <= (hi - lo) / B + gap + 1e-9)


def test_histogram_micro_batches_add_up(qb_case):
    E, k, T, layer, z, bias = qb_case
    if T < 2:
        pytest.skip("one token")
    B = 257
    whole = torch.zeros(E, B, dtype=torch.int32, device="cuda")
    parts = torch.zeros(E, B, dtype=torch.int32, device="cuda")
    layer.lmoe_qb_histogram(T, whole, logits=z, bias=bias)
    h = T // 3
    layer.lmoe_qb_histogram(h, parts, logits=z[:h].contiguous(), bias=bias)
    layer.lmoe_qb_histogram(T - h, parts, logits=z[h:].contiguous(), bias=bias)
    torch.cuda.synchronize()
    assert torch.equal(whole, parts)


def test_update_from_the_last_forward():
    """logits = NULL and bias = NULL read the handle's last forward's router
    logits and its own router bias."""
    wl = C.workload("k3_tiny_t16")
    W, x = gpu_inputs(wl)
    layer = make_layer(wl, W, max_tokens=64, keep_f32=False)
    try:
        layer.lmoe_forward(x)
        z = layer.lmoe_debug_tensor("logits", wl.T)
        a = layer.lmoe_qb_update(wl.T)
        b = layer.lmoe_qb_update(wl.T, logits=z, bias=W["router_bias"])
        torch.cuda.synchronize()
        layer.lmoe_sync_status()
        assert torch.equal(a, b)
        from latent_mixture_experts_gb300 import LmoeError
        with pytest.raises(LmoeError):
            layer.lmoe_qb_update(wl.T + 1)          # not the last forward's token count
    finally:
        layer.close()
