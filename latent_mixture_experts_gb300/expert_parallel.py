"""Expert-parallel forward of the layer: one process per GPU, the routed
experts split into contiguous ranges of E / R per rank (Kimi K2 card,
``moe_infer`` under ``ep_size > 1``; at the latent width for Stable
LatentMoE, so both exchanges move l-wide rows).

    send, counts = lmoe_ep_dispatch(x)             # router, grouping by global expert, x^c rows
    all_to_all(counts)  -> recv_counts             # rows every source sends to each local expert
    all_to_all(send, splits) -> recv               # the token exchange
    out = lmoe_ep_experts(recv, recv_counts)       # local regrouping, grouped expert GEMMs
    all_to_all(out, splits reversed) -> ret        # back to the source ranks
    Delta = lmoe_ep_combine(ret)                   # x G, slot-ordered sum, RMSNorm, output GEMM

The exchanges go through torch.distributed (NCCL on GPUs); the split sizes
are read on the host between them, as the K2 card's code does.  The device
work is the library's; this module only moves buffers between the calls.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def exchange_plan(counts: torch.Tensor, recv_counts: torch.Tensor, world: int):
    """Row splits of the token exchange: send_splits[r] = rows this rank sends
    to rank r (its experts' counts), recv_splits[s] = rows it receives from
    rank s (the counts s sent for this rank's experts)."""
    E = counts.numel()
    if E % world:
        raise ValueError(f"{E} experts do not split over {world} ranks")
    send_splits = counts.view(world, E // world).sum(1).tolist()
    recv_splits = recv_counts.view(world, E // world).sum(1).tolist()
    return send_splits, recv_splits


def ep_forward(layer, x: torch.Tensor, group=None) -> torch.Tensor:
    """Delta [T][d] of this rank's tokens x [T][d] (bf16) through an
    expert-parallel handle (ep_size = the group's size).  Every rank of the
    group calls it with its own tokens at the same time."""
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    send, counts = layer.lmoe_ep_dispatch(x)
    if world == 1:
        out = layer.lmoe_ep_experts(send, counts.view(1, -1))
        return layer.lmoe_ep_combine(out, x.shape[0])
    recv_counts = torch.empty_like(counts)
    dist.all_to_all_single(recv_counts, counts, group=group)
    send_splits, recv_splits = exchange_plan(counts, recv_counts, world)
    recv = send.new_empty(sum(recv_splits), send.shape[1])
    dist.all_to_all_single(recv, send, recv_splits, send_splits, group=group)
    out = layer.lmoe_ep_experts(recv, recv_counts.view(world, -1))
    ret = torch.empty_like(send)
    dist.all_to_all_single(ret, out, send_splits, recv_splits, group=group)
    return layer.lmoe_ep_combine(ret, x.shape[0])


def local_experts(weights: dict, rank: int, world: int) -> dict:
    """The weights of an expert-parallel rank: every dense tensor, and the
    contiguous range of routed experts [rank E/R, (rank+1) E/R) of each
    ex_* tensor (leading dimension E)."""
    out = {}
    for k, v in weights.items():
        if k.startswith("ex_"):
            E = v.shape[0]
            if E % world:
                raise ValueError(f"{E} experts do not split over {world} ranks")
            n = E // world
            out[k] = v[rank * n:(rank + 1) * n].contiguous()
        else:
            out[k] = v
    return out
