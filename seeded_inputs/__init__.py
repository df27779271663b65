"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no attention arithmetic: it only draws Q, K, V, rounds them
to bf16 and describes the workloads. Both the CUDA path and the CPU oracle read
the very same bf16 values (the oracle upcasts them to fp64).

Recipe: a CPU ``torch.Generator`` seeded per workload draws ``torch.randn`` in
fp32 for Q, then K, then V (each [B, H, N, d]); each is multiplied by sigma and
rounded to bf16 (round to nearest even). The shapes are those of the pages'
workloads: the SD2.1 512x512 self-attention (seqlen 4096, d_head 64), its UNet
block with cond/uncond batch and 5 heads, a causal LM shape, a 64x64-token 2-D
neighbourhood-attention grid, a 16384-token long sequence and a 16x16x16
volume of 3-D neighbourhood attention with two wrapped axes.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

MASKS = ("none", "causal", "clamp", "wrap")


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    sigma: float
    scale: float
    mask: str = "none"          # none | causal | clamp | wrap
    window: int = 0
    dilation: int = 1
    grid: tuple = field(default=None)  # (grid_h, grid_w) or (depth, rows, cols)
    seed: int = 0
    wrap_axes: tuple = field(default=None)  # one boolean per grid axis; None: as the mask says

    @property
    def heads(self) -> int:
        return self.B * self.H


def _w(name, B, H, N, d, sigma, mask="none", window=0, grid=None, seed=0, wrap_axes=None):
    return Workload(name, B, H, N, N, d, sigma, 1.0 / math.sqrt(d), mask, window, 1,
                    grid, seed, wrap_axes)


# The pages' workloads, in order (seed = 69000 + index).
WORKLOADS = {
    "sd21_single_head": _w("sd21_single_head", 1, 1, 4096, 64, 1.0, seed=69000),
    "sd21_unet_block": _w("sd21_unet_block", 2, 5, 4096, 64, 0.5, seed=69001),
    "lm_causal": _w("lm_causal", 4, 16, 2048, 128, 1.0, mask="causal", seed=69002),
    "na2d_clamp": _w("na2d_clamp", 1, 4, 4096, 32, 1.0, mask="clamp", window=7,
                     grid=(64, 64), seed=69003),
    "na2d_wrap": _w("na2d_wrap", 1, 4, 4096, 32, 1.0, mask="wrap", window=7,
                    grid=(64, 64), seed=69003),
    "long_seq": _w("long_seq", 1, 8, 16384, 128, 1.0, seed=69004),
    # the NATTEN issue requester's volumes: ~16 patches a side, window 5, 1-2 axes wrapped
    "na3d_wrap2": _w("na3d_wrap2", 1, 4, 4096, 32, 1.0, mask="clamp", window=5,
                     grid=(16, 16, 16), seed=69005, wrap_axes=(True, True, False)),
}


def make_qkv(B, H, Nq, Nk, d, sigma=1.0, seed=0):
    """Seeded bf16 CPU tensors q [B,H,Nq,d], k and v [B,H,Nk,d]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = (torch.randn(B, H, Nq, d, generator=g, dtype=torch.float32) * sigma).to(torch.bfloat16)
    k = (torch.randn(B, H, Nk, d, generator=g, dtype=torch.float32) * sigma).to(torch.bfloat16)
    v = (torch.randn(B, H, Nk, d, generator=g, dtype=torch.float32) * sigma).to(torch.bfloat16)
    return q, k, v


def make_workload(w: Workload):
    return make_qkv(w.B, w.H, w.Nq, w.Nk, w.d, w.sigma, w.seed)


def to_f64(t: torch.Tensor):
    """Exact upcast of a bf16 tensor to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()
