"""fp64 CPU oracle of the top-1 Switch MoE layer forward pass.

TEST INFRASTRUCTURE ONLY: tests/, __graft_entry__.smoke() and bench.py's CPU
baseline may use it; the CUDA library never does.  See oracle.switch_oracle.
"""
from . import switch_oracle
from .switch_oracle import (capacity, router_logits, softmax, top1, assign_slots, load_balance,
                            route, dispatch, expert_ffn, expert_outputs, combine, forward,
                            ties_within, groups_with_near_ties, Route)
