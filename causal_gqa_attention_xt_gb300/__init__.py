"""GB300-native causal grouped-query attention core (QK-RMSNorm + RoPE + causal
GQA SDPA, forward and backward) behind a C-ABI library of sm_103a kernels.

``causal_gqa_attention_xt_gb300.xt`` is the thin Python binding of that
library; ``causal_gqa_attention_xt_gb300.inputs`` draws seeded inputs.
Importing this package loads nothing: the CUDA library is loaded on first use
and its absence is an error, never a fallback.
"""
__all__ = ["inputs", "xt", "build"]
