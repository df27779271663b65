"""exact_attention_69_gb300: the fused exact-attention forward pass,
softmax(scale * Q K^T [+ mask]) V, as hand-written sm_103a (GB300) kernels
behind a small C ABI (include/attn.h, libattn.so).

Masks: none, causal (tiles above the diagonal skipped), 2-D neighbourhood
attention with clamped or circular ("wrap") windows (tiles no window touches
skipped). Outputs: O in bf16 and the fp32 log-sum-exp.
"""
from .api import (  # noqa: F401
    attention, attn_bwd, attn_fwd, device_status, na2d, na3d, sm_count, workspace_bytes)
from ._lib import AttnError  # noqa: F401

__all__ = ["attn_fwd", "attn_bwd", "attention", "na2d", "na3d", "device_status", "sm_count",
           "workspace_bytes", "AttnError"]
