"""Host-side parts of bench.py: the reference arm's per-assignment restatement
of the oracle gives oracle.forward's Delta, and the byte / FLOP accounting
matches the layer shapes of both model cards."""
from dataclasses import replace

import numpy as np
import pytest

import bench
import oracle as O
from lmoe_inputs import configs as C

K2_TINY = C.Workload("k2_tiny_t6", replace(C.K2, d_model=256, n_experts=12, top_k=3, d_expert_ff=128,
                                           d_shared_ff=128), T=6, seed=41)


@pytest.mark.parametrize("wl", [C.workload("k3_tiny_t16"), K2_TINY], ids=["k3_tiny", "k2_tiny"])
def test_reference_arm_matches_oracle_forward(wl):
    k = wl.cfg.top_k
    arm = bench.ReferenceArm(wl, n_assign=3 * k)
    for s in range(3 * k):
        arm.step(s)
    arm.layer.W["expert_fn"] = lambda name, e: arm.need[(name, e)]     # the codes the arm generated
    ref = O.forward(arm.layer, arm.x_bits[:3], routes={n: v[:3] for n, v in arm.routes.items()})
    got = np.stack([arm.delta[t] for t in range(3)])
    assert np.allclose(got, ref["delta"], rtol=1e-12, atol=1e-12 * np.abs(ref["delta"]).max())


def test_accounting_k3():
    a = bench.accounting(C.K3)
    assert a["expert"] == 3 * (3584 * 3072 // 2 + 3584 * 3072 // 32)            # 17,547,264
    assert a["dense"] == 896 * 7168 * 2 + 896 * 4 + 2 * 3584 * 7168 * 2 + 3584 * 2 + 3 * 6144 * 7168 * 2
    assert a["flops_per_token"] == 1_436_811_264


def test_accounting_k2():
    a = bench.accounting(C.K2)
    blk = 4 * 16 * 56                                           # fp32 scale per 128 x 128 block
    assert a["expert"] == 3 * (2048 * 7168 + blk)
    assert a["dense"] == 384 * 7168 * 2 + 384 * 4 + 3 * (2048 * 7168 + blk)
    assert a["flops_per_token"] == 2 * 384 * 7168 + 8 * 6 * 2048 * 7168 + 6 * 2048 * 7168


def test_expert_tile_rule():
    """bench.py's copy of the library's token-tile rule picks the tiles the
    profiler captures were taken on."""
    assert bench.expert_tile(C.K3, 64) == 16
    assert bench.expert_tile(C.workload("k3_e64_t8").cfg, 8) == 16
    assert bench.expert_tile(C.K3, 8192) == 96
    assert bench.expert_tile(C.K2, 4096) == 96
    assert bench.expert_tile(C.workload("k2_e32_t384").cfg, 384) == 96


def test_gate_up_ksplit_rule():
    """bench.py's copy of the library's K-split rule: the full K3 layer splits
    the gate/up pass at one token only (16 expert tiles x 12 weight items is
    under two items per SM; two tokens may select 32 experts), the 64-expert
    profiling case at one token, FP8 never."""
    assert [t for t in range(1, 17) if bench.gate_up_ksplit(C.K3, t)] == [1]
    assert bench.gate_up_ksplit(C.workload("k3_e64_t8").cfg, 1)
    assert not bench.gate_up_ksplit(C.K3, 64)
    assert not bench.gate_up_ksplit(C.K2, 1)
