"""CPU oracle for the MoE layer forward (test infrastructure only).

Importable by ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference arm; never by the product path.
"""
from .moe_oracle import (DEFAULT, RENORMALIZE, DEEPSEEKV3, LLAMA4, RENORMALIZE_NAIVE, MINIMAX2,
                         SIGMOID_RENORM, GROUPED_TOPK, GROUPED_TOPK_SOFTMAX, METHODS, topk_desc,
                         softmax64, sigmoid64, deepseek_keys, group_select, group_totals_fp32,
                         grouped_topk, route, permute, swiglu, expert_ffn, gate, forward,
                         forward_partial, forward_permuted)

__all__ = ["DEFAULT", "RENORMALIZE", "DEEPSEEKV3", "LLAMA4", "RENORMALIZE_NAIVE", "MINIMAX2",
           "SIGMOID_RENORM", "GROUPED_TOPK", "GROUPED_TOPK_SOFTMAX", "METHODS", "topk_desc",
           "softmax64", "sigmoid64", "deepseek_keys", "group_select", "group_totals_fp32",
           "grouped_topk", "route", "permute", "swiglu", "expert_ffn", "gate", "forward",
           "forward_partial", "forward_permuted"]
