"""fp64 CPU oracle of the Mixtral-style sparse MoE feed-forward layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``sparse_mixture_experts_56_b300``) never imports it and shares no code with
it; the two meet only in the seeded input generators of ``workloads``.

Every function here is the plain definition of one step of the layer, written
in float64 NumPy, with a citation of the page and section it follows.  See
``oracle/moe.py``.
"""
from .moe import (  # noqa: F401
    router_logits, topk_select, topk_mask, masked_softmax, gate, gate_softmax_then_topk,
    silu, expert_swiglu, group_by_expert, moe_layer, moe_layer_dense, rmsnorm,
    stacked_layer, near_tie_tokens, param_counts, consecutive_same_expert_rate,
    routing_statistics, sigmoid, silu_grad, softmax_backward, expert_swiglu_backward,
    moe_layer_backward, attention_gqa, attention_gqa_rows, decoder_layer,
)
from .ep import ep_experts_of, ep_send_counts, ep_exchange_plan, ep_load, ep_regroup  # noqa: F401
