"""Pins of the oracle's block-scaled E4M3 activation emulation (the MXFP8
activations of the walk-through's "参数账" section, one or two terms):
rounding against torch's float8_e4m3fn cast, the block exponent against its
definition by exhaustive search, the per-element error bound of one term,
and the layer-level effect of the emulation."""
import numpy as np
import torch

import oracle as O
from lmoe_inputs import configs as C
from lmoe_inputs import generate as G


def test_e4m3_rounding_matches_torch_cast():
    rng = np.random.default_rng(0)
    v = (rng.standard_normal(300000) * 10.0 ** rng.uniform(-5, 2.65, 300000)).astype(np.float32)
    v = np.clip(v, -448, 448)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    assert np.array_equal(O.e4m3_round(v.astype(np.float64)), ref)
    assert O.e4m3_round(np.array([500.0, -1e6]))[0] == 448.0 and O.e4m3_round(np.array([-1e6]))[0] == -448.0


def test_block_exponent_is_the_smallest_non_saturating_power_of_two():
    rng = np.random.default_rng(1)
    a = np.abs(rng.standard_normal(20000)) * 10.0 ** rng.uniform(-30, 30, 20000)
    a[:5] = [448.0, 224.0, 1.75 * 256, 1.7500001 * 256, 2.0 ** -100 * 448]
    p = O.e4m3_block_exponent(a)
    for v, e in zip(a, p):
        best = next(q for q in range(-126, 127) if v / 2.0 ** q <= 448.0)
        assert e == best
    assert O.e4m3_block_exponent(np.array([0.0]))[0] == -126


def test_one_term_error_bound_and_two_terms():
    """One term: every element whose scaled value is a normal E4M3 number is
    within half a step (2^-4 of its binade) of itself; two terms cut the
    per-GEMM-input error by more than an order of magnitude."""
    rng = np.random.default_rng(2)
    v = rng.standard_normal((64, 3584)) * np.exp(rng.standard_normal((64, 1)))
    one = O.mx_e4m3_terms(v, 1)
    two = O.mx_e4m3_terms(v, 2)
    blocks = v.reshape(64, -1, 32)
    p = O.e4m3_block_exponent(np.abs(blocks).max(-1))[..., None]
    normal = (np.abs(blocks) / np.exp2(p) >= 2.0 ** -6).reshape(v.shape)
    rel = np.abs(one - v) / np.abs(v)
    assert rel[normal].max() <= 2.0 ** -4 * (1 + 1e-12)
    e1 = np.linalg.norm(one - v) / np.linalg.norm(v)
    e2 = np.linalg.norm(two - v) / np.linalg.norm(v)
    assert 0.01 < e1 < 0.04 and e2 < e1 / 10


def test_layer_emulation_modes():
    """act_terms=None is the exact layer; two terms stay within 1e-2 of it,
    one term (MXFP8) does not — the reason the library keeps two terms by
    default and checks its one-term mode against this emulation."""
    wl = C.workload("k3_tiny_t16")
    W = G.gen_weights(wl)
    x = G.gen_x(wl)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    L = O.Layer(wl.cfg, O.numpy_inputs(W))
    ref = O.forward(L, xb)
    assert np.array_equal(O.forward(L, xb, act_terms=None)["delta"], ref["delta"])

    def rel(a):
        return (np.linalg.norm(a - ref["delta"], axis=1) / np.linalg.norm(ref["delta"], axis=1)).max()
    r2 = rel(O.forward(L, xb, act_terms=2)["delta"])
    r1 = rel(O.forward(L, xb, act_terms=1)["delta"])
    assert r2 < 3e-3 and r1 > 1e-2, (r1, r2)


def test_valid_range_holds_the_encoding_and_its_boundary_neighbours():
    """The range holds the oracle's own encoding; away from boundaries it is
    that encoding alone; a value on a rounding midpoint admits both
    neighbours; a block maximum on a scale threshold admits both scales."""
    rng = np.random.default_rng(3)
    v = rng.standard_normal((8, 64))
    lo, hi = O.mx_e4m3_valid_range(v)
    enc = O.mx_e4m3_terms(v, 1)
    assert np.all((lo <= enc) & (enc <= hi))
    big = np.abs(v) > 0.1 * np.abs(v).max()
    assert (lo[big] != hi[big]).mean() < 2e-2
    w = np.zeros((1, 32))
    w[0, 0] = 448.0                     # block maximum exactly on the scale threshold
    w[0, 1] = 1.0625                    # midpoint of 1.0 and 1.125 at scale 1
    lo, hi = O.mx_e4m3_valid_range(w)
    assert lo[0, 1] <= 1.0 and hi[0, 1] >= 1.125
    assert lo[0, 0] <= 448.0 <= hi[0, 0]


def test_e2m1_rounding_is_nearest_with_ties_to_even_codes():
    """Against the grid the format defines (pinned code by code elsewhere):
    every result is a nearest grid point; at midpoints, the even code."""
    grid = O.E2M1_VALUES[:8]
    rng = np.random.default_rng(4)
    v = rng.uniform(-7, 7, 100000)
    r = O.e2m1_round(v)
    d = np.abs(np.minimum(np.abs(v), 6.0)[:, None] - grid[None, :]).min(1)
    assert np.allclose(np.abs(np.minimum(np.abs(v), 6.0) - np.abs(r)), d, rtol=0, atol=1e-15)
    mids = (grid[:-1] + grid[1:]) / 2                      # 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5
    assert list(O.e2m1_round(mids)) == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]
    assert O.e2m1_round(np.array([-9.0]))[0] == -6.0


def test_e2m1_terms_converge():
    """Each MXFP4 term shrinks the residual: three terms reach ~1e-3 relative
    error per GEMM input (two E4M3 terms' precision), four a few 1e-4; the
    block exponent is the smallest non-saturating one."""
    rng = np.random.default_rng(5)
    v = rng.standard_normal((32, 3584)) * np.exp(rng.standard_normal((32, 1)))
    errs = [np.linalg.norm(O.mx_e2m1_terms(v, t) - v) / np.linalg.norm(v) for t in (1, 2, 3, 4)]
    assert errs[0] > errs[1] > errs[2] > errs[3]
    assert 3e-4 < errs[2] < 5e-3 and errs[3] < 1e-3
    a = np.abs(rng.standard_normal(5000)) * 10.0 ** rng.uniform(-20, 20, 5000)
    for x, p in zip(a, O.e2m1_block_exponent(a)):
        assert p == next(q for q in range(-126, 127) if x / 2.0 ** q <= 6.0)
