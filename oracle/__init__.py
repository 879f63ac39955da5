"""CPU float64 oracle of the MoE training update (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package; the product path never does.
"""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import (worked_example, rmsnorm, rmsnorm_backward, rope_tables, rope,
                         rope_backward, causal_attention, causal_attention_backward, causal_logsumexp,
                         token_topk, route_order, moe_forward, forward_backward,
                         clip_adamw, global_norm, train_update, loss_only, Dims,
                         UpdateResult, n_targets, to64, softmax, silu, silu_grad,
                         selective_updates, SelectiveResult, EXPERT_TENSORS)
