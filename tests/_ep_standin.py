"""CPU stand-in of an expert-parallel handle for the multi-process tests of
the exchange logic: the three device phases of lmoe_ep_dispatch /
lmoe_ep_experts / lmoe_ep_combine restated with the fp64 oracle on CPU
tensors (test infrastructure; the library's kernels run in the GPU tests)."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O


class OracleEPLayer:
    """Rank `rank` of `world`: the full dense weights and the routed experts
    [rank E/R, (rank+1) E/R) of a layer, the layer's phases in fp64."""

    def __init__(self, cfg, weights_np: dict, rank: int, world: int):
        self.cfg, self.rank, self.world = cfg, rank, world
        self.E_loc = cfg.n_experts // world
        self.layer = O.Layer(cfg, weights_np)
        self.state = {}

    def lmoe_ep_dispatch(self, x: torch.Tensor):
        cfg, L = self.cfg, self.layer
        xb = x.view(torch.int16).numpy().view(np.uint16)
        xf = O.bf16_bits_to_f64(xb)
        r = O.router(xf, L.dense("router_w"), L.W["router_bias"], cfg.top_k, cfg.routed_scale)
        xe = xf @ L.dense("w_down_latent").T if cfg.d_latent else xf
        d = O.dispatch(r["idx"], cfg.n_experts)
        self.state = dict(x=xf, G=r["G"], perm=d["perm"], T=x.shape[0])
        send = torch.from_numpy(xe[d["perm"] // cfg.top_k].copy())
        return send, torch.from_numpy(d["counts"].astype(np.int32))

    def lmoe_ep_experts(self, recv: torch.Tensor, recv_counts: torch.Tensor) -> torch.Tensor:
        rows = recv.numpy()
        cnt = recv_counts.numpy().reshape(self.world, self.E_loc)
        out = np.zeros_like(rows)
        pos = 0
        for s in range(self.world):                      # source-major, local experts inside
            for e in range(self.E_loc):
                n = int(cnt[s, e])
                ge = self.rank * self.E_loc + e
                blk = rows[pos:pos + n]
                g = blk @ self.layer.expert("ex_gate", ge).T
                u = blk @ self.layer.expert("ex_up", ge).T
                out[pos:pos + n] = self.layer.act(g, u) @ self.layer.expert("ex_down", ge).T
                pos += n
        assert pos == rows.shape[0]
        return torch.from_numpy(out)

    def lmoe_ep_combine(self, ret: torch.Tensor, T: int) -> torch.Tensor:
        cfg, L, st = self.cfg, self.layer, self.state
        assert T == st["T"]
        k = cfg.top_k
        y = np.zeros((T * k, ret.shape[1]))
        y[st["perm"]] = ret.numpy()
        u = (y.reshape(T, k, -1) * st["G"][:, :, None]).sum(1)
        if cfg.d_latent:
            uh = O.rms_norm(u, L.dense("norm_w"), cfg.norm_eps) if cfg.use_latent_norm else u
            yr = uh @ L.dense("w_up_latent").T
        else:
            yr = u
        ys = L.act(st["x"] @ L.shared("sh_gate").T, st["x"] @ L.shared("sh_up").T) @ L.shared("sh_down").T
        return torch.from_numpy(yr + ys)
