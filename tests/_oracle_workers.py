"""The fp64 oracle's forward over many tokens, in spawned worker processes.

The layer is per-token (each token's Delta depends on that token and the
weights only), so a large parity check splits its tokens into chunks and
runs ``oracle.forward`` on each chunk in its own process.  The weights reach
the workers as .npy files in a temporary directory (dense weights once; each
selected expert's codes and scales once), which the workers map read-only.
Workers are started with the "spawn" method and import numpy and the oracle
only, never torch or CUDA.
"""
from __future__ import annotations

import multiprocessing
import os
import shutil
import tempfile
import types

import numpy as np

_CFG_FIELDS = ("d_model", "d_latent", "n_experts", "top_k", "d_expert_ff", "d_shared_ff", "use_latent_norm",
               "norm_eps", "routed_scale", "situ_beta", "situ_linear_beta", "act", "expert_wfmt")


def _forward_chunk(args):
    """Worker: oracle forward of one chunk of tokens with the given selection."""
    import oracle as O
    wdir, cfgd, x_bits, idx, keep, act_terms, x_in, h_in = args
    cfg = types.SimpleNamespace(**cfgd)
    W = {}
    for f in os.listdir(wdir):
        if f.startswith("dense_"):
            W[f[len("dense_"):-len(".npy")]] = np.load(os.path.join(wdir, f), mmap_mode="r")

    def expert_fn(name, e):
        return (np.load(os.path.join(wdir, f"{name}_q_{e}.npy")), np.load(os.path.join(wdir, f"{name}_s_{e}.npy")))

    W["expert_fn"] = expert_fn
    layer = O.Layer(cfg, W, cache_experts=False)
    r = O.forward(layer, x_bits, idx=idx, act_terms=act_terms, x_in=x_in, h_in=h_in)
    return {k: r[k] for k in keep if r.get(k) is not None}


class OracleWorkers:
    """Pool of spawned processes running the oracle on token chunks.

    wl: the workload (its layer config); W_gpu: the layer weights as the
    tests hold them (torch tensors, experts stacked [E, ...])."""

    def __init__(self, wl, W_gpu: dict, workers: int | None = None):
        import oracle as O
        self.cfg = {f: getattr(wl.cfg, f) for f in _CFG_FIELDS}
        self.W = W_gpu
        # RAM-backed /dev/shm when it has room, else the default temp directory
        base = None
        if os.path.isdir("/dev/shm") and shutil.disk_usage("/dev/shm").free > 16 << 30:
            base = "/dev/shm"
        self.dir = tempfile.mkdtemp(prefix="lmoe_oracle_", dir=base)
        dense = {k: v for k, v in W_gpu.items() if not k.startswith("ex_")}
        for k, v in O.numpy_inputs(dense).items():
            np.save(os.path.join(self.dir, f"dense_{k}.npy"), v)
        self.saved = set()
        n = workers or min(8, os.cpu_count() or 1)
        self.n = n
        self.pool = multiprocessing.get_context("spawn").Pool(n)

    def _save_experts(self, experts):
        for e in experts:
            e = int(e)
            if e in self.saved:
                continue
            for m in ("ex_gate", "ex_up", "ex_down"):
                np.save(os.path.join(self.dir, f"{m}_q_{e}.npy"), self.W[m + "_q"][e].cpu().numpy())
                np.save(os.path.join(self.dir, f"{m}_s_{e}.npy"), self.W[m + "_s"][e].cpu().numpy())
            self.saved.add(e)

    def forward(self, x_bits: np.ndarray, idx: np.ndarray, keep=("delta",), act_terms=None, x_in=None,
                h_in=None) -> dict:
        """Oracle forward of tokens x_bits (bf16 bits [T, d]) with the given
        selection idx [T, k] (act_terms: the activation emulation of
        oracle.forward); returns the `keep` outputs stacked over tokens."""
        x_bits = np.asarray(x_bits)
        idx = np.asarray(idx)
        self._save_experts(np.unique(idx))
        T = x_bits.shape[0]
        chunks = [c for c in np.array_split(np.arange(T), min(T, 2 * self.n)) if len(c)]
        try:
            k = idx.shape[1]
            res = self.pool.map(_forward_chunk, [
                (self.dir, self.cfg, x_bits[c], idx[c], keep, act_terms, None if x_in is None else x_in[c],
                 None if h_in is None else h_in.reshape(-1, k, h_in.shape[-1])[c].reshape(-1, h_in.shape[-1]))
                for c in chunks])
        finally:
            self._drop_experts()
        return {k: np.concatenate([r[k] for r in res]) for k in keep}

    def _drop_experts(self):
        """Expert files are written per call (a full-size expert is 17.5 MB)."""
        for e in self.saved:
            for m in ("ex_gate", "ex_up", "ex_down"):
                for part in ("q", "s"):
                    f = os.path.join(self.dir, f"{m}_{part}_{e}.npy")
                    if os.path.exists(f):
                        os.unlink(f)
        self.saved.clear()

    def close(self):
        self.pool.terminate()
        self.pool.join()
        shutil.rmtree(self.dir, ignore_errors=True)

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
