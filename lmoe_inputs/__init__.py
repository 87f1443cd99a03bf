"""Seeded synthetic inputs (shapes, seeds, checkpoint formats) shared by the
fp64 oracle and the CUDA library's tests and benchmark."""
from .configs import (LayerConfig, Workload, WORKLOADS, SWEEP_T, K3, K3_TINY, K3_MID, K2,
                      workload, param_counts)
from .generate import gen_inputs, gen_weights, gen_x, gen_expert, gen_router_bias
