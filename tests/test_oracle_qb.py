"""Pins of the oracle's Quantile Balancing update (tutorial "Stable
LatentMoE", section "Quantile Balancing: giving every expert a fair shot";
walk-through "Kimi K3 模型结构（5）", section "Stable 之三：Quantile
Balancing", its appendix-C derivation and appendix-D histogram estimator)
against what the pages and the mathematics fix: the library quantile the
tutorial's code calls, the exact target load the walk-through derives, the
closed forms of the coordinate descent on the LP dual, centring invariance,
and the histogram estimator's bin-width error bound and additivity."""
import numpy as np
import pytest
import torch

import oracle as O


def _batch(m, n, seed, spread=1.0):
    rng = np.random.default_rng(seed)
    s = 1.0 / (1.0 + np.exp(-spread * rng.standard_normal((m, n))))
    b = rng.uniform(-0.1, 0.1, n)
    return s, b


def test_cutoff_is_the_k_plus_first_biased_score():
    s, b = _batch(40, 9, 0)
    a = O.qb_cutoffs(s, b, 3)
    for i in range(40):
        c = sorted(s[i] + b, reverse=True)
        assert a[i] == c[3]


@pytest.mark.parametrize("m,n,k", [(64, 8, 2), (200, 16, 3), (97, 12, 5)])
def test_exact_update_is_the_higher_quantile_the_code_takes(m, n, k):
    """The tutorial's update: quantile(relative_thresh, k/n, interpolation
    'higher') along the tokens, then the mean removed."""
    s, b = _batch(m, n, m + n)
    u = O.qb_update(s, b, k)
    r = torch.from_numpy(O.qb_cutoffs(s, b, k)[:, None] - s)
    ref = torch.quantile(r, k / n, dim=0, interpolation="higher").numpy()
    if float(k * (m - 1) / n).is_integer():
        pytest.skip("index exactly integral: float rounding of p (m-1) may land either side")
    assert np.array_equal(u["raw"], ref)
    assert np.array_equal(u["raw"], np.quantile(r.numpy(), k / n, axis=0, method="higher"))
    assert abs(u["bias"].mean()) < 1e-15
    assert np.allclose(u["bias"], ref - ref.mean(), rtol=0, atol=1e-15)


@pytest.mark.parametrize("m,n,k", [(64, 8, 2), (96, 12, 3), (160, 16, 4)])
def test_new_bias_gives_each_expert_exactly_its_target_load(m, n, k):
    """Walk-through: with every cutoff fixed, token i picks expert j exactly
    when s_ij + b_j > alpha_i, and the new bias is the (q+1)-th smallest
    required bias, q = m k / n.  So at most q tokens clear it strictly and
    at least q + 1 reach it; where no required bias ties with it (a tie
    arises when j is itself token i's (k+1)-th choice, r_ij = b_j), exactly
    q tokens pick j."""
    assert m * k % n == 0
    q = m * k // n
    s, b = _batch(m, n, 7 * m)
    u = O.qb_update(s, b, k)
    alpha = O.qb_cutoffs(s, b, k)
    strict = (s + u["raw"][None, :] > alpha[:, None]).sum(0)
    weak = (s + u["raw"][None, :] >= alpha[:, None]).sum(0)
    assert np.all(strict <= q) and np.all(weak >= q + 1)
    r = O.qb_required_bias(s, b, k)
    untied = np.array([(r[:, j] == u["raw"][j]).sum() == 1 for j in range(n)])
    assert untied.any()
    assert np.all(strict[untied] == q)


def _dual_expert_side(s, alpha, q, beta):
    """Expert-side part of the LP dual of the balanced assignment:
    q beta + sum_i max(0, s_i - alpha_i - beta)."""
    return q * beta + np.maximum(0.0, s - alpha - beta).sum()


def _dual_token_side(s_row, beta, k, a):
    return k * a + np.maximum(0.0, s_row - beta - a).sum()


def test_closed_forms_minimise_the_lp_dual():
    """Appendix C: fixing the token multipliers alpha, the expert multiplier
    beta_j = -b_j minimising the dual is the (q+1)-th largest of s_:j -
    alpha; fixing beta, alpha_i is the (k+1)-th largest of s_i: - beta.  Both
    checked against every breakpoint of the piecewise-linear objective."""
    m, n, k = 120, 10, 3
    q = m * k // n
    s, b = _batch(m, n, 11)
    alpha = O.qb_cutoffs(s, b, k)
    u = O.qb_update(s, b, k)
    for j in range(n):
        beta = -u["raw"][j]
        f = _dual_expert_side(s[:, j], alpha, q, beta)
        cand = s[:, j] - alpha
        assert all(f <= _dual_expert_side(s[:, j], alpha, q, c) + 1e-12 for c in cand)
        assert all(f <= _dual_expert_side(s[:, j], alpha, q, c) + 1e-12 for c in np.linspace(-2, 2, 401))
    beta = -b
    a = O.qb_cutoffs(s, b, k)
    for i in range(0, m, 7):
        g = _dual_token_side(s[i], beta, k, a[i])
        cand = s[i] - beta
        assert all(g <= _dual_token_side(s[i], beta, k, c) + 1e-12 for c in cand)


def test_centred_update_ignores_a_common_bias_offset():
    s, b = _batch(80, 8, 3)
    u0 = O.qb_update(s, b, 2)["bias"]
    u1 = O.qb_update(s, b + 0.37, 2)["bias"]
    assert np.allclose(u0, u1, rtol=0, atol=1e-12)


def test_histogram_counts_brute_force_and_additivity():
    """Every (token, expert) counted once in the bin whose edges bracket r;
    counts of micro-batches add up to the counts of the whole batch."""
    s, b = _batch(90, 6, 5)
    B = 37
    h = O.qb_histogram(s, b, 2, B)
    assert np.all(h.sum(1) == 90)
    lo, hi = O.qb_range(b)
    edges = lo + (hi - lo) / B * np.arange(B + 1)
    r = O.qb_required_bias(s, b, 2)
    for j in range(6):
        ref = np.histogram(r[:, j], bins=edges)[0]
        assert np.array_equal(h[j], ref)
    parts = O.qb_histogram(s[:40], b, 2, B) + O.qb_histogram(s[40:], b, 2, B)
    assert np.array_equal(parts, h)
    assert r.min() >= lo and r.max() <= hi        # the range the walk-through derives


@pytest.mark.parametrize("B", [50, 1000])
def test_histogram_quantile_within_one_bin_of_the_exact_order_statistic(B):
    """Appendix D: the estimate lies in the bin of the ceil(q)-th smallest
    required bias, so its error is below one bin width; at B = 1000 and
    biases of +-0.1 that width is a few 1e-3."""
    m, n, k = 3000, 16, 2
    s, b = _batch(m, n, B)
    h = O.qb_histogram(s, b, k, B)
    est = O.qb_update_from_histogram(h, b, k)
    r = np.sort(O.qb_required_bias(s, b, k), axis=0)
    lo, hi = O.qb_range(b)
    w = (hi - lo) / B
    target = -(-(m * k) // n)
    assert np.all(np.abs(est["raw"] - r[target - 1]) <= w * (1 + 1e-12))
    exact = O.qb_update(s, b, k)
    assert np.all(np.abs(est["raw"] - exact["raw"]) <= w + (r[target] - r[target - 1]) + 1e-12)
    if B == 1000:
        assert 1e-3 <= w <= 1e-2
