"""The expert-parallel exchange (latent_mixture_experts_gb300.expert_parallel)
on two gloo ranks on CPU: each rank routes its own tokens, ships every
assignment's latent row to the rank owning the expert (count all-to-all,
token all-to-all), computes its experts' outputs and sends them back; each
rank's Delta must equal the single-process oracle forward of its tokens.
The device phases are stood in by the fp64 oracle (tests/_ep_standin.py);
the split sizes, orders and buffers are the module's own."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle as O
from lmoe_inputs import configs as C
from lmoe_inputs import generate as G


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, wl_name, q):
    from dataclasses import replace
    from latent_mixture_experts_gb300.expert_parallel import ep_forward, exchange_plan
    from tests._ep_standin import OracleEPLayer
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.set_num_threads(max(1, (os.cpu_count() or 1) // world))   # ranks share the host's cores
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = C.workload(wl_name)
        W = O.numpy_inputs(G.gen_weights(wl))
        x = G.gen_x(replace(wl, seed=wl.seed + 101 * rank), T=wl.T - 3 * rank)   # ranks hold different counts
        layer = OracleEPLayer(wl.cfg, W, rank, world)
        got = ep_forward(layer, x).numpy()
        ref = O.forward(O.Layer(wl.cfg, W), x.view(torch.int16).numpy().view(np.uint16))["delta"]
        err = np.abs(got - ref).max() / np.abs(ref).max()
        # the split plan: what rank r sends to s is what s receives from r
        send, counts = layer.lmoe_ep_dispatch(x)
        rc = torch.empty_like(counts)
        dist.all_to_all_single(rc, counts)
        ss, rs = exchange_plan(counts, rc, world)
        allss = [None] * world
        dist.all_gather_object(allss, ss)
        ok_plan = all(allss[s][rank] == rs[s] for s in range(world))
        q.put((rank, float(err), ok_plan, int(send.shape[0])))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_expert_parallel_exchange_matches_oracle(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, "k3_tiny_t16", q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=180) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, err, ok_plan, nsend in res:
        assert ok_plan, rank
        assert err < 1e-12, (rank, err)
