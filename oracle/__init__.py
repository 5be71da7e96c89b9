"""CPU oracle of the sparse MoE FFN forward pass (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package; the CUDA library never does.
"""
from .moe_oracle import (capacity, expert_ffn, forward, gate_logits, gelu,  # noqa: F401
                         load_balance, permute, renormalise, route, select_topk,
                         softmax)
