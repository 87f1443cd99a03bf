"""Shared helpers of the GPU tests: build and load the library, place a
workload's seeded inputs on the GPU, run the oracle on the same bytes."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle as O
from lmoe_inputs import generate as G


@functools.lru_cache(maxsize=1)
def built_library() -> str:
    from latent_mixture_experts_gb300 import build
    return build.build()


def gpu_inputs(wl, T=None):
    """Seeded weights and tokens of `wl`, generated on the GPU (same bytes
    as on the CPU)."""
    W = G.gen_weights(wl, device="cuda")
    x = G.gen_x(wl, device="cuda", T=T)
    return W, x


def make_layer(wl, W, max_tokens):
    from latent_mixture_experts_gb300 import LatentMoE
    built_library()
    return LatentMoE(wl.cfg, W, max_tokens=max_tokens)


def oracle_layer(wl, W_gpu):
    """Oracle view of the generated weights: dense tensors copied to the
    host, experts fetched one at a time on first use."""
    dense = {k: v for k, v in W_gpu.items() if not k.startswith("ex_")}
    Wn = O.numpy_inputs(dense)

    def expert_fn(name, e):
        q = W_gpu[name + "_q"][e].cpu().numpy()
        s = W_gpu[name + "_s"][e].cpu().numpy()
        return q, s

    Wn["expert_fn"] = expert_fn
    return O.Layer(wl.cfg, Wn)


def x_bits(x: torch.Tensor) -> np.ndarray:
    return x.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def rel_l2_per_token(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    num = np.sqrt(((got - ref) ** 2).sum(-1))
    den = np.sqrt((ref ** 2).sum(-1))
    return num / np.maximum(den, 1e-30)


def bf16_half_ulp(v: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers at |v| (8 significant bits): the
    largest error of rounding v to the nearest bf16."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def assert_delta_close(got, ref, rel_tol=1e-2, abs_frac=2e-2):
    """Tolerances of the layer output: per-token relative L2 <= 1e-2 and
    max-abs <= 2e-2 * RMS(oracle output).  The layer returns Delta in bf16,
    which cannot hold an element closer than half a bf16 spacing at its
    magnitude (0.03 at |Delta| ~ 10), so each element's error is taken
    beyond that unavoidable rounding before the max-abs bound."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rel = rel_l2_per_token(got, ref)
    rms = np.sqrt((ref ** 2).mean())
    err = np.abs(got - ref)
    beyond = np.maximum(err - bf16_half_ulp(ref), 0.0)
    i = np.unravel_index(np.argmax(beyond), beyond.shape)
    assert rel.max() <= rel_tol, f"per-token rel L2 max {rel.max():.3e} (token {rel.argmax()})"
    assert beyond[i] <= abs_frac * rms, (
        f"max abs err beyond bf16 rounding {beyond[i]:.3e} > {abs_frac} * RMS {rms:.3e} "
        f"(element {i}: |ref| {abs(ref[i]):.3e}, err {err[i]:.3e}; max raw err {err.max():.3e})")
    return rel.max(), beyond[i] / rms


def valid_selection(c_row: np.ndarray, sel, tol=1e-6) -> bool:
    """A selection is valid when no unselected expert beats a selected one
    by more than `tol` in biased score."""
    sel = np.asarray(sel)
    mask = np.zeros(c_row.shape[0], dtype=bool)
    mask[sel] = True
    if mask.all():
        return True
    return c_row[mask].min() >= c_row[~mask].max() - tol
