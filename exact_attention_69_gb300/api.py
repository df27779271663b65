"""Python entry points over libattn.so.

PyTorch provides device memory and streams; the computation is one launch of
the library's sm_103a kernel per call. Nothing here computes attention.

    attn_fwd(q, k, v, ...)        q,k,v [B,H,N,d] bf16 (CUDA, or CPU tensors that
                                  are staged to the GPU and back)
    na2d(q, k, v, kernel_size, mode)
                                  NATTEN's heads-last [B, X, Y, heads, d] layout,
                                  'clamp' or 'wrap' windows (NATTEN issue #142),
                                  per axis if asked
    na3d(q, k, v, kernel_size, mode)
                                  the same on volumes [B, X, Y, Z, heads, d]
    attn_bwd(q, k, v, o, lse, dout, ...), attention(q, k, v, ...)
                                  gradients; a differentiable op
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import _lib

_MASKS = {"none": _lib.ATTN_MASK_NONE, "causal": _lib.ATTN_MASK_CAUSAL,
          "causal_br": _lib.ATTN_MASK_CAUSAL_BR, "clamp": _lib.ATTN_MASK_NA2D,
          "wrap": _lib.ATTN_MASK_NA2D}


def _strides(t: torch.Tensor, layout: str):
    """Element strides (b, h, n) of a tensor viewed as [B, H, N, d]."""
    if t.stride(-1) != 1:
        raise ValueError("the last (head) dimension must be contiguous")
    if layout == "bhnd":
        sb, sh, sn, _ = t.stride()
    elif layout == "bxyzhd":  # heads-last volume [B, X, Y, Z, H, d]: n = (x * Y + y) * Z + z
        sb, sx, sy, sz, sh, _ = t.stride()
        if sy != sz * t.shape[3] or sx != sy * t.shape[2]:
            raise ValueError("X, Y and Z must be jointly contiguous in a heads-last layout")
        sn = sz
    else:  # heads-last [B, X, Y, H, d]: token n = x * Y + y
        sb, sx, sy, sh, _ = t.stride()
        if sx != sy * t.shape[2]:
            raise ValueError("X and Y must be jointly contiguous in a heads-last layout")
        sn = sy
    return (sb, sh, sn)


def _set_mask(p, mask, window, dilation, grid, wrap_axes):
    """mask_kind and the neighbourhood fields of a parameter block. A 'clamp' or
    'wrap' mask on a 3-entry grid (depth, rows, columns) is NA3D, else NA2D;
    window: k for every axis or one per grid axis; wrap_axes: None (every axis
    as the mask name says) or one boolean per grid axis."""
    if mask not in _MASKS:
        raise ValueError(f"unknown mask {mask!r}")
    p.mask_kind = _MASKS[mask]
    if mask not in ("clamp", "wrap"):
        p.window, p.dilation, p.wrap = int(window), int(dilation), 0
        return
    nax = 3 if grid is not None and len(grid) == 3 else 2
    win = tuple(int(x) for x in window) if isinstance(window, (tuple, list)) else (int(window),) * nax
    wr = (mask == "wrap",) * nax if wrap_axes is None else tuple(bool(x) for x in wrap_axes)
    if len(win) != nax or len(wr) != nax:
        raise ValueError("window and wrap_axes need one entry per grid axis")
    kh, kw = win[-2], win[-1]
    p.window, p.window_w = kh, (kw if kw != kh else 0)
    p.wrap = {(False, False): 0, (True, True): 1, (True, False): 2, (False, True): 3}[wr[-2:]]
    p.dilation = int(dilation)
    if nax == 3:
        p.mask_kind = _lib.ATTN_MASK_NA3D
        p.grid_d, p.grid_h, p.grid_w = (int(x) for x in grid)
        p.window_d = win[0] if win[0] != kh else 0
        p.wrap_d = int(wr[0])
    elif grid is not None:
        p.grid_h, p.grid_w = int(grid[0]), int(grid[1])


def _check_dev(*ts):
    for t in ts:
        if t.dtype != torch.bfloat16:
            raise TypeError("q, k, v must be bfloat16")
        if not t.is_cuda:
            raise ValueError("expected CUDA tensors")


def _launch(q, k, v, o, lse, *, B, H, Nq, Nk, d, scale, mask, window, dilation, grid,
            layout, num_ctas, timeout_ns, inject, events, stream, schedule=0, workspace=None,
            wrap_axes=None, tune_iters=0):
    p = _lib.params()
    p.q, p.k, p.v, p.o = q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr()
    p.lse = lse.data_ptr() if lse is not None else None
    p.B, p.H, p.Nq, p.Nk, p.d = B, H, Nq, Nk, d
    p.scale = float(scale)
    _set_mask(p, mask, window, dilation, grid, wrap_axes)
    for name, t in (("q_stride", q), ("k_stride", k), ("v_stride", v), ("o_stride", o)):
        getattr(p, name)[:] = _strides(t, layout)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    p.stream = stream.cuda_stream
    p.num_ctas = int(num_ctas)
    p.timeout_ns = int(timeout_ns)
    p.inject = int(inject)
    p.schedule = int(schedule)
    if workspace is not None:
        p.workspace = workspace.data_ptr()
        p.workspace_bytes = workspace.numel() * workspace.element_size()
    with torch.cuda.device(q.device):
        if tune_iters > 0:
            res = _lib.AttnTuneResult()
            _lib.check(_lib.load().attn_tune(ctypes.byref(p), int(tune_iters), ctypes.byref(res)),
                       "attn_tune")
            return res
        # torch events bracket the single launch on the same stream (events
        # recorded inside the library would be invisible to torch)
        if events is not None:
            events[0].record(stream)
        _lib.check(_lib.fwd_ex(p), "attn_fwd")
        if events is not None:
            events[1].record(stream)
    return None


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, scale: float | None = None,
             mask: str = "none", window=0, dilation: int = 1, grid=None,
             out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
             return_lse: bool = True, num_ctas: int = 0, timeout_ns: int = 0, inject: int = 0,
             events=None, stream=None, schedule: int = 0,
             workspace: torch.Tensor | None = None, wrap_axes=None):
    """Fused exact attention forward over [B, H, N, d] bf16 tensors.

    mask: 'none' | 'causal' (top-left) | 'causal_br' (bottom-right: query i sees keys
    up to i + Nk - Nq) | 'clamp' | 'wrap' (the last two: neighbourhood
    attention over grid=(rows, columns), square by default, or a volume
    grid=(depth, rows, columns), with an odd `window` or one per axis;
    wrap_axes (one boolean per axis) chooses per axis whether the window
    wraps, overriding the mask name; a (1, N) grid with window (1, k) is 1-D
    neighbourhood attention). Returns (o, lse) or o. CPU inputs are copied to the current
    CUDA device, and the results back to the CPU (the end-to-end path).
    schedule: 0 automatic, 1 whole tasks per CTA, 2 equal shares of K/V tiles
    with cut tasks merged (unmasked only). workspace: optional zero-filled
    device tensor for schedule 2 (see workspace_bytes); default: the
    library's own.
    """
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    if not q.is_cuda:
        return _host_roundtrip(q, k, v, scale=scale, mask=mask, window=window,
                               dilation=dilation, grid=grid, return_lse=return_lse,
                               wrap_axes=wrap_axes)
    _check_dev(q, k, v)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if lse is not None and (not lse.is_contiguous() or lse.dtype != torch.float32):
        raise ValueError("lse must be a contiguous float32 [B, H, Nq] tensor")
    _launch(q, k, v, out, lse, B=B, H=H, Nq=Nq, Nk=Nk, d=d, scale=scale, mask=mask,
            window=window, dilation=dilation, grid=grid, layout="bhnd", num_ctas=num_ctas,
            timeout_ns=timeout_ns, inject=inject, events=events, stream=stream,
            schedule=schedule, workspace=workspace, wrap_axes=wrap_axes)
    return (out, lse) if return_lse else out


def attn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
             lse: torch.Tensor, dout: torch.Tensor, *, scale: float | None = None,
             mask: str = "none", window=0, dilation: int = 1, grid=None, wrap_axes=None,
             stream=None, timeout_ns: int = 0):
    """Backward pass of attn_fwd: (dq, dk, dv) for the gradient dout at the output.

    q, o, dout [B, H, Nq, d]; k, v [B, H, Nk, d] contiguous bf16 CUDA tensors;
    lse the forward's float32 [B, H, Nq]. mask and the neighbourhood options as
    for attn_fwd.
    """
    ts = (q, k, v, o, dout)
    _check_dev(*ts)
    if any(not t.is_contiguous() for t in ts) or not lse.is_contiguous():
        raise ValueError("the backward pass takes contiguous tensors")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    p = _lib.bwd_params()
    p.q, p.k, p.v, p.o, p.dout = (t.data_ptr() for t in ts)
    p.lse = lse.data_ptr()
    p.dq, p.dk, p.dv = dq.data_ptr(), dk.data_ptr(), dv.data_ptr()
    p.B, p.H, p.Nq, p.Nk, p.d = B, H, Nq, Nk, d
    p.scale = float(scale)
    _set_mask(p, mask, window, dilation, grid, wrap_axes)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    p.stream = stream.cuda_stream
    p.timeout_ns = int(timeout_ns)
    with torch.cuda.device(q.device):
        _lib.check(_lib.bwd(p), "attn_bwd")
    return dq, dk, dv


class _Attention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, scale, mask, opts):
        o, lse = attn_fwd(q, k, v, scale=scale, mask=mask, **opts)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.scale, ctx.mask, ctx.opts = scale, mask, opts
        return o

    @staticmethod
    def backward(ctx, dout):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = attn_bwd(q, k, v, o, lse, dout.contiguous(), scale=ctx.scale, mask=ctx.mask,
                              **ctx.opts)
        return dq, dk, dv, None, None, None


def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, scale: float | None = None,
              mask: str = "none", window=0, dilation: int = 1, grid=None,
              wrap_axes=None) -> torch.Tensor:
    """attn_fwd as a differentiable torch op over contiguous bf16 CUDA tensors
    [B, H, N, d] (every mask): the backward pass runs attn_bwd."""
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    opts = dict(window=window, dilation=dilation, grid=grid, wrap_axes=wrap_axes)
    return _Attention.apply(q, k, v, float(scale), mask, opts)


def workspace_bytes(B: int, H: int, Nq: int, Nk: int, d: int, *, mask: str = "none",
                    num_ctas: int = 0, schedule: int = 0) -> int:
    """Bytes of workspace an attn_fwd call of this shape needs on the current device."""
    p = _lib.params()
    p.q = p.k = p.v = p.o = 256  # placeholders: only the shape is examined
    p.B, p.H, p.Nq, p.Nk, p.d = B, H, Nq, Nk, d
    p.scale = 1.0
    p.mask_kind = _MASKS[mask]
    p.num_ctas = int(num_ctas)
    p.schedule = int(schedule)
    n = _lib.load().attn_workspace_bytes(p)
    if n < 0:
        _lib.check(int(-n), "attn_workspace_bytes")
    return int(n)


def _host_roundtrip(q, k, v, *, return_lse, **kw):
    dev = torch.device("cuda", torch.cuda.current_device())
    s = torch.cuda.current_stream(dev)
    qd, kd, vd = (t.to(dev, non_blocking=True) for t in (q, k, v))
    o, lse = attn_fwd(qd, kd, vd, return_lse=True, **kw)
    o_h = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    l_h = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    o_h.copy_(o, non_blocking=True)
    l_h.copy_(lse, non_blocking=True)
    s.synchronize()
    return (o_h, l_h) if return_lse else o_h


def na2d(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, kernel_size, *,
         mode="clamp", dilation: int = 1, scale: float | None = None,
         out: torch.Tensor | None = None, return_lse: bool = False, stream=None):
    """2-D neighbourhood attention in NATTEN's heads-last layout [B, X, Y, heads, d].

    kernel_size: k, or (k_x, k_y). mode 'clamp': windows keep their full size
    and shift inward at the borders; 'wrap': windows wrap around the borders
    (circular); or a pair of those, one per axis (x, y). The output has the
    same layout; no permute or copy of the inputs is made.
    """
    modes = (mode, mode) if isinstance(mode, str) else tuple(mode)
    if len(modes) != 2 or any(m not in ("clamp", "wrap") for m in modes):
        raise ValueError("mode must be 'clamp' or 'wrap', or a pair of them")
    if q.dim() != 5:
        raise ValueError("expected [B, X, Y, heads, d] tensors")
    _check_dev(q, k, v)
    B, X, Y, H, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    lse = torch.empty((B, H, X * Y), dtype=torch.float32, device=q.device) if return_lse else None
    _launch(q, k, v, out, lse, B=B, H=H, Nq=X * Y, Nk=X * Y, d=d, scale=scale, mask="clamp",
            window=kernel_size, dilation=dilation, grid=(X, Y), layout="bxyhd", num_ctas=0,
            timeout_ns=0, inject=0, events=None, stream=stream,
            wrap_axes=(modes[0] == "wrap", modes[1] == "wrap"))
    return (out, lse) if return_lse else out


def na3d(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, kernel_size, *,
         mode="clamp", dilation: int = 1, scale: float | None = None,
         out: torch.Tensor | None = None, return_lse: bool = False, stream=None):
    """3-D neighbourhood attention in NATTEN's heads-last layout [B, X, Y, Z, heads, d].

    kernel_size: k, or (k_x, k_y, k_z). mode: 'clamp' | 'wrap', or one per axis
    (x, y, z). The output has the same layout; no permute or copy is made.
    """
    modes = (mode,) * 3 if isinstance(mode, str) else tuple(mode)
    if len(modes) != 3 or any(m not in ("clamp", "wrap") for m in modes):
        raise ValueError("mode must be 'clamp' or 'wrap', or three of them")
    if q.dim() != 6:
        raise ValueError("expected [B, X, Y, Z, heads, d] tensors")
    _check_dev(q, k, v)
    B, X, Y, Z, H, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    n = X * Y * Z
    lse = torch.empty((B, H, n), dtype=torch.float32, device=q.device) if return_lse else None
    _launch(q, k, v, out, lse, B=B, H=H, Nq=n, Nk=n, d=d, scale=scale, mask="clamp",
            window=kernel_size, dilation=dilation, grid=(X, Y, Z), layout="bxyzhd", num_ctas=0,
            timeout_ns=0, inject=0, events=None, stream=stream,
            wrap_axes=tuple(m == "wrap" for m in modes))
    return (out, lse) if return_lse else out


def tune(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, scale: float | None = None,
         mask: str = "none", window=0, dilation: int = 1, grid=None, wrap_axes=None,
         iters: int = 10, stream=None) -> dict:
    """Time the forward's schedule candidates on these inputs and return the
    fastest as {'schedule', 'num_ctas', 'us', 'n_tried'}; pass schedule and
    num_ctas to later attn_fwd calls of the same shape. Synchronous."""
    _check_dev(q, k, v)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = torch.empty_like(q, memory_format=torch.contiguous_format)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    res = _launch(q, k, v, out, lse, B=B, H=H, Nq=Nq, Nk=Nk, d=d, scale=scale, mask=mask,
                  window=window, dilation=dilation, grid=grid, layout="bhnd", num_ctas=0,
                  timeout_ns=0, inject=0, events=None, stream=stream, wrap_axes=wrap_axes,
                  tune_iters=iters)
    return {"schedule": res.schedule, "num_ctas": res.num_ctas, "us": float(res.us),
            "n_tried": res.n_tried}


def device_status():
    """Read and clear the device status word: (code, [code, role, tile, cta])."""
    return _lib.device_status()


def sm_count() -> int:
    n = _lib.load().attn_device_sm_count()
    if n < 0:
        _lib.check(-n, "attn_device_sm_count")
    return n
