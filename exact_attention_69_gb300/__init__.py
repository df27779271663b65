"""exact_attention_69_gb300: the fused exact-attention forward pass,
softmax(scale * Q K^T [+ mask]) V, as hand-written sm_103a (GB300) kernels
behind a small C ABI (include/attn.h, libattn.so).

Masks: none, causal (tiles above the diagonal skipped), neighbourhood attention
on 2-D grids and 3-D volumes with clamped or circular ("wrap") windows chosen
per axis, and dilation (tiles no window touches skipped). Outputs: O in bf16
and the fp32 log-sum-exp. attn_bwd / attention: the backward pass for every
mask. tune: the split-KV schedule chosen by measurement.
"""
from .api import (  # noqa: F401
    attention, attn_bwd, attn_fwd, device_status, na2d, na3d, sm_count, tune, workspace_bytes)
from ._lib import AttnError  # noqa: F401

__all__ = ["attn_fwd", "attn_bwd", "attention", "na2d", "na3d", "tune", "device_status", "sm_count",
           "workspace_bytes", "AttnError"]
