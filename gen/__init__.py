"""Seeded synthetic input generators shared by the oracle side and the CUDA side.

Holds no arithmetic of the layer itself; see gen.inputs.
"""
from .inputs import (LayerShape, WORKLOADS, WORKLOAD_ORDER, WORKLOAD_SEEDS, SKEW_GAMMA,
                     act_dtype, expert_weights, make_inputs, skewed_router_bias, workload, workload_seed)
