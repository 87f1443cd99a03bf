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


def make_layer(wl, W, max_tokens, keep_f32=True):
    """The layer through the C ABI; keep_f32 also keeps each forward's Delta
    before its bf16 rounding (debug tensor "delta_f32")."""
    from latent_mixture_experts_gb300 import LatentMoE
    built_library()
    layer = LatentMoE(wl.cfg, W, max_tokens=max_tokens)
    if keep_f32:
        layer.lmoe_keep_f32_output(True)
    return layer


def forward_checked(layer, x):
    """One forward: (bf16 Delta, its fp32 value before rounding, idx, G) as
    numpy, after the deferred-error check."""
    out, idx, Gw = layer.lmoe_forward(x, return_routing=True)
    torch.cuda.synchronize()
    layer.lmoe_sync_status()
    out32 = layer.lmoe_debug_tensor("delta_f32", x.shape[0])
    return (out.cpu().double().numpy(), out32.cpu().double().numpy(), idx.cpu().numpy(), Gw.cpu().numpy())


def check_expert_io(layer, T, k, x_in, h_ref, terms, rows=None, label="", tol=(2e-3, 5e-3)):
    """Step-level check of the routed experts: the inputs ("x_expert") and
    hidden activations ("h") the expert GEMMs multiplied, decoded from their
    E4M3 terms, against the oracle's x_in [T][dx] (per token) and h
    [T*k][F] (per assignment).  rows: the assignments to compare (default
    all).  Two terms: within their resolution of the exact values (rel-L2 per
    row <= 2e-3 for x, 5e-3 for h, whose g and u carry x's encoding).  One
    term, against the oracle continuing from the GPU's validated encodings
    (validated_one_term_inputs / _hidden): identical."""
    xg = layer.lmoe_debug_tensor("x_expert", T).cpu().double().numpy()
    hg = layer.lmoe_debug_tensor("h", T).cpu().double().numpy()
    rows = np.arange(T * k) if rows is None else np.asarray(rows)
    xw = np.asarray(x_in)[rows // k]
    xg, hg, hw = xg[rows], hg[rows], np.asarray(h_ref)
    rx, rh = rel_l2_per_token(xg, xw).max(), rel_l2_per_token(hg, hw).max()
    fx, fh = (xg != xw).mean(), (hg != hw).mean()
    print(f"{label}: expert inputs rel-L2 max {rx:.2e} ({fx:.1e} of codes differ), "
          f"hidden rel-L2 max {rh:.2e} ({fh:.1e} differ)")
    if terms == 1:
        assert fx == 0 and fh == 0, (fx, fh)
    else:
        assert rx <= tol[0] and rh <= tol[1], (rx, rh)


def validated_one_term_hidden(layer, T, h_exact, rows=None, rel=2e-3):
    """The GPU's one-term hidden activations h [T*k][F] (rows: the
    assignments to take), each element checked to be an encoding of a value
    within rel x its 32-block's largest magnitude of the oracle's exact h
    (rel = 2e-3 covers the hardware tanh and exp approximations the epilogue
    uses, relative error ~2^-11 each).  Returns them for
    oracle.forward(h_in=...) and the fraction that differ from the oracle's
    own rounding."""
    hg = layer.lmoe_debug_tensor("h", T).cpu().double().numpy()
    if rows is not None:
        hg = hg[np.asarray(rows)]
    h_exact = np.asarray(h_exact, dtype=np.float64)
    lo, hi = O.mx_e4m3_valid_range(h_exact, rel=rel)
    ok = (lo <= hg) & (hg <= hi)
    assert ok.all(), f"{(~ok).sum()} hidden activations outside the valid encodings"
    return hg, (hg != O.mx_e4m3_terms(h_exact, 1)).mean()


def validated_one_term_inputs(layer, T, k, xe_exact, rows=None):
    """The GPU's one-term expert inputs, checked element by element to be one
    of the encodings the oracle allows for the exact x^c (the encoding
    itself, or at a rounding or scale boundary that an fp32 x^c can fall on
    either side of, the other valid ones: O.mx_e4m3_valid_range).  Every
    assignment of a token must carry the same encoding.  Returns the
    per-token rows [len(rows)][dx] for oracle.forward(x_in=...) and the
    fraction of elements where the GPU took another valid encoding than
    the oracle's own rounding."""
    xg = layer.lmoe_debug_tensor("x_expert", T).cpu().double().numpy().reshape(T, k, -1)
    assert (xg == xg[:, :1]).all(), "assignments of one token carry different encodings"
    xt = xg[:, 0] if rows is None else xg[np.asarray(rows), 0]
    xe_exact = np.asarray(xe_exact, dtype=np.float64)
    lo, hi = O.mx_e4m3_valid_range(xe_exact)
    ok = (lo <= xt) & (xt <= hi)
    assert ok.all(), f"{(~ok).sum()} encoded inputs outside the valid encodings"
    other = (xt != O.mx_e4m3_terms(xe_exact, 1)).mean()
    return xt, other


def sample_tokens(T, n, routes, idx, seed=0):
    """Every token for T <= n; else n tokens: the first and last, up to four
    the oracle flags as near ties, one on the most loaded expert, the rest
    drawn at random."""
    if T <= n:
        return list(range(T))
    pick = {0, T - 1}
    pick.update(int(t) for t in np.nonzero(routes["flag"])[0][:4])
    counts = np.bincount(idx.reshape(-1), minlength=int(idx.max()) + 1)
    pick.add(int(np.nonzero((idx == int(np.argmax(counts))).any(1))[0][0]))
    rng = np.random.default_rng(seed)
    for t in rng.permutation(T):
        if len(pick) >= n:
            break
        pick.add(int(t))
    return sorted(pick)


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


def max_abs_over_rms(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.abs(got - ref).max() / np.sqrt((ref ** 2).mean()))


def assert_delta_close(got, ref, got_f32=None, rel_tol=1e-2, abs_frac=2e-2, label=""):
    """Tolerances of the layer output, as stated: per-token relative L2 <=
    1e-2 and max-abs <= 2e-2 * RMS(oracle output), both raw.

    `got` is the layer's bf16 output.  `got_f32`, when given, is the same
    forward's output before that final bf16 rounding (the "delta_f32" debug
    tensor); the max-abs bound is then applied to it as well, since a bf16
    element cannot come closer to the exact value than half a bf16 spacing
    (0.03 at |Delta| ~ 10).  Prints the raw figures of both and the bf16
    error beyond that rounding; returns (rel max, raw max-abs / RMS of the
    bf16 output, raw of the fp32 output or None)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rel = rel_l2_per_token(got, ref)
    rms = np.sqrt((ref ** 2).mean())
    err = np.abs(got - ref)
    raw16 = err.max() / rms
    beyond = (np.maximum(err - bf16_half_ulp(ref), 0.0)).max() / rms
    raw32 = None
    if got_f32 is not None:
        f = np.asarray(got_f32, dtype=np.float64)
        raw32 = np.abs(f - ref).max() / rms
        assert np.array_equal(bf16_round(f), got), "bf16 output is not the rounding of the fp32 output"
    print(f"{label}: rel-L2 max {rel.max():.3e}, max-abs/RMS raw {raw16:.3e} (bf16 out), "
          + (f"{raw32:.3e} (fp32 before rounding), " if raw32 is not None else "")
          + f"{beyond:.3e} beyond bf16 rounding")
    assert rel.max() <= rel_tol, f"per-token rel L2 max {rel.max():.3e} (token {rel.argmax()})"
    bound_on = raw32 if raw32 is not None else raw16
    assert bound_on <= abs_frac, (f"max-abs/RMS {bound_on:.3e} > {abs_frac} "
                                  f"({'fp32 output before rounding' if raw32 is not None else 'bf16 output'})")
    return rel.max(), raw16, raw32


def bf16_round(v: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even of float64 values that are fp32 numbers to bf16."""
    f = np.asarray(v, dtype=np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint32) << 16
    return r.view(np.float32).astype(np.float64)


def valid_selection(c_row: np.ndarray, sel, tol=1e-6) -> bool:
    """A selection is valid when no unselected expert beats a selected one
    by more than `tol` in biased score."""
    sel = np.asarray(sel)
    mask = np.zeros(c_row.shape[0], dtype=bool)
    mask[sel] = True
    if mask.all():
        return True
    return c_row[mask].min() >= c_row[~mask].max() - tol
