"""Python interface with the signatures of the DeepSeek-V4 sparse MQA pages
(NeMo AutoModel, tilelang_sparse_mla_fwd: `sparse_mqa_fwd_interface`;
tilelang_sparse_mla_bwd: `sparse_mqa_bwd_interface`).

PyTorch only supplies device memory and the current stream; every step of the
computation runs in libsparse_mqa.so's CUDA kernels, reached through the C ABI
(include/sparse_mqa.h).  There is no CPU path: inputs must be contiguous CUDA
tensors.  The TileLang tuning knobs of the pages (block_I, num_stages,
threads) are accepted for signature compatibility and ignored.
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional

import torch

from . import _lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: int) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _shape(q: torch.Tensor, kv: torch.Tensor, attn_sink: torch.Tensor,
           topk_idxs: torch.Tensor) -> _lib.Shape:
    _need(q, "q", torch.bfloat16, 4)
    _need(kv, "kv", torch.bfloat16, 3)
    _need(attn_sink, "attn_sink", torch.float32, 1)
    _need(topk_idxs, "topk_idxs", torch.int32, 3)
    B, S, H, D = q.shape
    if kv.shape[0] != B or kv.shape[2] != D:
        raise ValueError(f"kv shape {tuple(kv.shape)} does not match q {tuple(q.shape)}")
    if attn_sink.shape[0] != H:
        raise ValueError(f"attn_sink must have H={H} entries")
    if topk_idxs.shape[0] != B or topk_idxs.shape[1] != S:
        raise ValueError(f"topk_idxs shape {tuple(topk_idxs.shape)} does not match q")
    devs = {q.device, kv.device, attn_sink.device, topk_idxs.device}
    if len(devs) != 1:
        raise ValueError("all tensors must be on the same device")
    return _lib.Shape(B, S, kv.shape[1], H, D, topk_idxs.shape[2])


def _check_device(device: torch.device, what: str) -> None:
    """Synchronizes ``device`` and raises SMQAError if a kernel's bounded
    wait ran out (the status word stays set; device_status(clear=True)
    resets it)."""
    with torch.cuda.device(device):
        st = int(_lib.load().smqa_device_status(0))
    if st != _lib.SMQA_OK:
        raise _lib.SMQAError(what, st, "a kernel's bounded wait ran out; its outputs are "
                             "undefined (device_status(clear=True) resets the status)")


def _scale(sm_scale: Optional[float], D: int) -> float:
    """None selects D^-1/2 (the pages' default); a value is used as given."""
    if sm_scale is None:
        return 1.0 / math.sqrt(D)
    s = float(sm_scale)
    if not s > 0.0 or not math.isfinite(s):
        raise ValueError("sm_scale must be a positive finite float or None")
    return s


def sparse_mqa_fwd_interface(q: torch.Tensor, kv: torch.Tensor, attn_sink: torch.Tensor,
                             topk_idxs: torch.Tensor, sm_scale: Optional[float] = None,
                             block_I: int = 64, num_stages: int = 2, threads: int = 256,
                             reference_rounding: bool = False,
                             workspace: Optional[torch.Tensor] = None,
                             check_status: bool = False
                             ) -> tuple[torch.Tensor, torch.Tensor]:
    """Top-k sparse MQA forward.

    q [B,S,H,D] bf16, kv [B,S_kv,D] bf16 (shared keys and values),
    attn_sink [H] fp32, topk_idxs [B,S,topk] int32 (entries outside
    [0,S_kv) are masked).  Returns freshly allocated O [B,S,H,D] bf16 and
    LSE [B,S,H] fp32 = log2(sum_valid exp(sm_scale q.k) + exp(sink)).
    ``workspace`` (uint8 CUDA tensor, D = 512 only) may be passed to reuse
    the exchange pool between calls; otherwise one is allocated.  With
    ``check_status`` the call synchronizes and raises SMQAError
    (SMQA_ERR_DEVICE_TIMEOUT) if a kernel's bounded wait ran out.
    """
    shp = _shape(q, kv, attn_sink, topk_idxs)
    scale = _scale(sm_scale, shp.D)
    flags = _lib.FLAG_REFERENCE_ROUNDING if reference_rounding else 0
    lib = _lib.load()
    need = int(lib.smqa_fwd_workspace_bytes(shp))
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8, 1)
    if need > 0 and (workspace is None or workspace.numel() < need):
        workspace = torch.empty((need,), dtype=torch.uint8, device=q.device)
    if need == 0:
        workspace = None
    o = torch.empty_like(q)
    lse = torch.empty((shp.B, shp.S, shp.H), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        _lib.check("smqa_fwd", lib.smqa_fwd(_ptr(q), _ptr(kv), _ptr(attn_sink), _ptr(topk_idxs),
                                            shp, scale, _ptr(o), _ptr(lse), _ptr(workspace),
                                            0 if workspace is None else workspace.numel(), flags,
                                            _stream(q.device)))
    if check_status:
        _check_device(q.device, "smqa_fwd")
    return o, lse


def fwd_workspace_bytes(shape: _lib.Shape) -> int:
    return int(_lib.load().smqa_fwd_workspace_bytes(shape))


def bwd_workspace_bytes(shape: _lib.Shape, return_dkv_accum_dtype: bool = False) -> int:
    flags = _lib.FLAG_RETURN_DKV_FP32 if return_dkv_accum_dtype else 0
    return int(_lib.load().smqa_bwd_workspace_bytes(shape, flags))


def sparse_mqa_bwd_interface(q: torch.Tensor, kv: torch.Tensor, attn_sink: torch.Tensor,
                             o: torch.Tensor, do: torch.Tensor, topk_idxs: torch.Tensor,
                             lse: torch.Tensor, sm_scale: Optional[float] = None,
                             return_dkv_accum_dtype: bool = False,
                             workspace: Optional[torch.Tensor] = None,
                             return_dsink: bool = False, deterministic: bool = False,
                             check_status: bool = False):
    """Top-k sparse MQA backward.

    Takes the forward's inputs, its output o, the gradient do [B,S,H,D] bf16
    and its log2 lse [B,S,H] fp32.  Returns freshly allocated dq [B,S,H,D]
    bf16 and dkv [B,S_kv,D] (bf16, or fp32 with return_dkv_accum_dtype), and
    with ``return_dsink`` also the gradient w.r.t. attn_sink (fp32 [H]; not
    among the pages' outputs).  ``deterministic`` accumulates dkv in 64-bit
    fixed point (binary point chosen per call from the inputs' magnitudes)
    with integer atomics, so it is bit-identical from run to run (not a
    switch of the pages).  ``workspace`` (uint8 CUDA tensor) may be passed to
    reuse scratch memory between calls; otherwise one is allocated.  With
    ``check_status`` the call synchronizes and raises SMQAError
    (SMQA_ERR_DEVICE_TIMEOUT) if a kernel's bounded wait ran out.
    """
    shp = _shape(q, kv, attn_sink, topk_idxs)
    _need(o, "o", torch.bfloat16, 4)
    _need(do, "do", torch.bfloat16, 4)
    _need(lse, "lse", torch.float32, 3)
    if o.shape != q.shape or do.shape != q.shape:
        raise ValueError("o and do must have q's shape")
    if tuple(lse.shape) != (shp.B, shp.S, shp.H):
        raise ValueError("lse must be [B,S,H]")
    scale = _scale(sm_scale, shp.D)
    flags = _lib.FLAG_RETURN_DKV_FP32 if return_dkv_accum_dtype else 0
    if deterministic:
        flags |= _lib.FLAG_DETERMINISTIC_DKV
    lib = _lib.load()
    need = int(lib.smqa_bwd_workspace_bytes(shp, flags))
    if need == 0:
        raise ValueError("unsupported shape for the backward")
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8, 1)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty((need,), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q)
    dkv = torch.empty((shp.B, shp.S_kv, shp.D),
                      dtype=torch.float32 if return_dkv_accum_dtype else torch.bfloat16,
                      device=q.device)
    dsink = torch.empty((shp.H,), dtype=torch.float32, device=q.device) if return_dsink else None
    with torch.cuda.device(q.device):
        _lib.check("smqa_bwd", lib.smqa_bwd(_ptr(q), _ptr(kv), _ptr(attn_sink), _ptr(o), _ptr(do),
                                            _ptr(topk_idxs), _ptr(lse), shp, scale, _ptr(dq),
                                            _ptr(dkv), _ptr(dsink), _ptr(workspace),
                                            workspace.numel(), flags, _stream(q.device)))
    if check_status:
        _check_device(q.device, "smqa_bwd")
    return (dq, dkv, dsink) if return_dsink else (dq, dkv)


def _need_host(t: torch.Tensor, name: str, dtype: torch.dtype, shape: tuple) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cpu":
        raise ValueError(f"{name} must be a CPU tensor (host buffer), got {t.device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _host_shape(q, kv, attn_sink, topk_idxs) -> _lib.Shape:
    for t, name in ((q, "q"), (kv, "kv"), (topk_idxs, "topk_idxs")):
        if not isinstance(t, torch.Tensor) or t.dim() != 3 + (name == "q"):
            raise ValueError(f"{name} has the wrong rank")
    B, S, H, D = q.shape
    shp = _lib.Shape(B, S, kv.shape[1], H, D, topk_idxs.shape[2])
    _need_host(q, "q", torch.bfloat16, (B, S, H, D))
    _need_host(kv, "kv", torch.bfloat16, (B, shp.S_kv, D))
    _need_host(attn_sink, "attn_sink", torch.float32, (H,))
    _need_host(topk_idxs, "topk_idxs", torch.int32, (B, S, shp.topk))
    return shp


def _host_out(out: Optional[dict], name: str, dtype: torch.dtype, shape: tuple) -> torch.Tensor:
    t = None if out is None else out.get(name)
    if t is None:
        return torch.empty(shape, dtype=dtype, pin_memory=True)
    _need_host(t, f"out[{name!r}]", dtype, shape)
    return t


def _host_workspace(workspace: Optional[torch.Tensor], need: int,
                    device: torch.device) -> torch.Tensor:
    if need == 0:
        raise ValueError("unsupported shape")
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8, 1)
        if workspace.device != device:
            raise ValueError(f"workspace must be on {device}")
        if workspace.numel() >= need:
            return workspace
    return torch.empty((need,), dtype=torch.uint8, device=device)


def fwd_host_workspace_bytes(shape: _lib.Shape) -> int:
    return int(_lib.load().smqa_fwd_host_workspace_bytes(shape))


def fwd_bwd_host_workspace_bytes(shape: _lib.Shape, return_dkv_accum_dtype: bool = False,
                                 deterministic: bool = False) -> int:
    flags = (_lib.FLAG_RETURN_DKV_FP32 if return_dkv_accum_dtype else 0) | \
        (_lib.FLAG_DETERMINISTIC_DKV if deterministic else 0)
    return int(_lib.load().smqa_fwd_bwd_host_workspace_bytes(shape, flags))


def sparse_mqa_fwd_host(q: torch.Tensor, kv: torch.Tensor, attn_sink: torch.Tensor,
                        topk_idxs: torch.Tensor, sm_scale: Optional[float] = None, *,
                        device: Optional[torch.device] = None,
                        workspace: Optional[torch.Tensor] = None,
                        out: Optional[dict] = None, reference_rounding: bool = False,
                        synchronize: bool = True) -> tuple[torch.Tensor, torch.Tensor]:
    """The forward on HOST (CPU) tensors: copies in, kernels and copies out
    run in token chunks that overlap (C ABI ``smqa_fwd_host``).

    Inputs as for sparse_mqa_fwd_interface but CPU tensors (page-locked ones
    let the copies overlap the kernels).  Returns CPU tensors O and LSE, taken
    from ``out`` ({"o", "lse"}) when given, else freshly allocated page-locked.
    ``device`` (default: the current CUDA device) runs the kernels;
    ``workspace`` (uint8 CUDA tensor there) is reused when large enough.  The
    work is queued on that device's current stream; with ``synchronize`` the
    call waits for it, otherwise the results are complete once that stream is.
    """
    shp = _host_shape(q, kv, attn_sink, topk_idxs)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else \
        torch.device(device)
    lib = _lib.load()
    ws = _host_workspace(workspace, int(lib.smqa_fwd_host_workspace_bytes(shp)), dev)
    o = _host_out(out, "o", torch.bfloat16, tuple(q.shape))
    lse = _host_out(out, "lse", torch.float32, (shp.B, shp.S, shp.H))
    flags = _lib.FLAG_REFERENCE_ROUNDING if reference_rounding else 0
    with torch.cuda.device(dev):
        _lib.check("smqa_fwd_host", lib.smqa_fwd_host(
            _ptr(q), _ptr(kv), _ptr(attn_sink), _ptr(topk_idxs), shp, _scale(sm_scale, shp.D),
            _ptr(o), _ptr(lse), _ptr(ws), ws.numel(), flags, _stream(dev)))
        if synchronize:
            torch.cuda.current_stream(dev).synchronize()
    return o, lse


def sparse_mqa_fwd_bwd_host(q: torch.Tensor, kv: torch.Tensor, attn_sink: torch.Tensor,
                            topk_idxs: torch.Tensor, do: torch.Tensor,
                            sm_scale: Optional[float] = None, *,
                            device: Optional[torch.device] = None,
                            workspace: Optional[torch.Tensor] = None,
                            out: Optional[dict] = None, return_dsink: bool = False,
                            return_dkv_accum_dtype: bool = False, deterministic: bool = False,
                            reference_rounding: bool = False, synchronize: bool = True):
    """Forward and backward on HOST (CPU) tensors with a known gradient ``do``
    of O (C ABI ``smqa_fwd_bwd_host``): copies in, kernels and copies out run
    in overlapping token chunks.

    Returns CPU tensors (o, lse, dq, dkv) and, with ``return_dsink``, dsink,
    taken from ``out`` ({"o", "lse", "dq", "dkv", "dsink"}) when given, else
    freshly allocated page-locked.  Other arguments as in
    sparse_mqa_fwd_host and sparse_mqa_bwd_interface.
    """
    shp = _host_shape(q, kv, attn_sink, topk_idxs)
    _need_host(do, "do", torch.bfloat16, tuple(q.shape))
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else \
        torch.device(device)
    flags = (_lib.FLAG_RETURN_DKV_FP32 if return_dkv_accum_dtype else 0) | \
        (_lib.FLAG_DETERMINISTIC_DKV if deterministic else 0) | \
        (_lib.FLAG_REFERENCE_ROUNDING if reference_rounding else 0)
    lib = _lib.load()
    ws = _host_workspace(workspace, int(lib.smqa_fwd_bwd_host_workspace_bytes(shp, flags)), dev)
    o = _host_out(out, "o", torch.bfloat16, tuple(q.shape))
    lse = _host_out(out, "lse", torch.float32, (shp.B, shp.S, shp.H))
    dq = _host_out(out, "dq", torch.bfloat16, tuple(q.shape))
    dkv = _host_out(out, "dkv", torch.float32 if return_dkv_accum_dtype else torch.bfloat16,
                    (shp.B, shp.S_kv, shp.D))
    dsink = _host_out(out, "dsink", torch.float32, (shp.H,)) if return_dsink else None
    with torch.cuda.device(dev):
        _lib.check("smqa_fwd_bwd_host", lib.smqa_fwd_bwd_host(
            _ptr(q), _ptr(kv), _ptr(attn_sink), _ptr(topk_idxs), _ptr(do), shp,
            _scale(sm_scale, shp.D), _ptr(o), _ptr(lse), _ptr(dq), _ptr(dkv), _ptr(dsink),
            _ptr(ws), ws.numel(), flags, _stream(dev)))
        if synchronize:
            torch.cuda.current_stream(dev).synchronize()
    return (o, lse, dq, dkv, dsink) if return_dsink else (o, lse, dq, dkv)


def device_status(clear: bool = True) -> int:
    """The device status word (0, or SMQA_ERR_DEVICE_TIMEOUT after a kernel's
    bounded wait ran out).  Synchronizes the device."""
    return int(_lib.load().smqa_device_status(1 if clear else 0))


def set_wait_limit_ns(ns: int) -> int:
    """Limit of every bounded wait in kernels launched from now on (0: the
    default, SMQA_WAIT_LIMIT_NS or 4 s); returns the previous limit."""
    return int(_lib.load().smqa_set_wait_limit_ns(int(ns)))


def indexer_bwd_interface(index_q: torch.Tensor, weights: torch.Tensor, index_k: torch.Tensor,
                          topk_indices: torch.Tensor, grad_scores: torch.Tensor) -> torch.Tensor:
    """Lightning-indexer backward for one batch element (tilelang_indexer_bwd
    page, `indexer_bwd_interface`): index_q [S,H,D] bf16, weights [S,H] fp32,
    index_k [S_kv,D] bf16, topk_indices [S,topk] int32, grad_scores [S,topk]
    fp32.  Returns a freshly allocated dq [S,H,D] bf16, the gradient of the
    scores sum_h w[t,h] ReLU(q[t,h] . k[idx[t,j]]) with respect to index_q."""
    _need(index_q, "index_q", torch.bfloat16, 3)
    _need(weights, "weights", torch.float32, 2)
    _need(index_k, "index_k", torch.bfloat16, 2)
    _need(topk_indices, "topk_indices", torch.int32, 2)
    _need(grad_scores, "grad_scores", torch.float32, 2)
    S, H, D = index_q.shape
    topk = topk_indices.shape[1]
    if tuple(weights.shape) != (S, H) or index_k.shape[1] != D or \
            tuple(topk_indices.shape) != (S, topk) or tuple(grad_scores.shape) != (S, topk):
        raise ValueError("indexer tensors do not have matching shapes")
    shp = _lib.Shape(1, S, index_k.shape[0], H, D, topk)
    dq = torch.empty_like(index_q)
    lib = _lib.load()
    with torch.cuda.device(index_q.device):
        _lib.check("smqa_indexer_bwd", lib.smqa_indexer_bwd(
            _ptr(index_q), _ptr(weights), _ptr(index_k), _ptr(topk_indices), _ptr(grad_scores),
            shp, _ptr(dq), _stream(index_q.device)))
    return dq


def batched_indexer_bwd(index_q: torch.Tensor, weights: torch.Tensor, index_k: torch.Tensor,
                        topk_indices: torch.Tensor, grad_scores: torch.Tensor) -> torch.Tensor:
    """The indexer backward in the page's batched layouts (`batched_indexer_bwd`):
    index_q [S,B,H,D] bf16, weights [S,B,H] fp32, index_k [S_kv,B,D] bf16,
    topk_indices [B,S,topk] int32, grad_scores [B,S,topk] fp32; returns dq
    [S,B,H,D] bf16.  One launch covers every batch element."""
    _need(index_q, "index_q", torch.bfloat16, 4)
    _need(weights, "weights", torch.float32, 3)
    _need(index_k, "index_k", torch.bfloat16, 3)
    _need(topk_indices, "topk_indices", torch.int32, 3)
    _need(grad_scores, "grad_scores", torch.float32, 3)
    S, B, H, D = index_q.shape
    topk = topk_indices.shape[2]
    if tuple(weights.shape) != (S, B, H) or index_k.shape[1] != B or index_k.shape[2] != D or \
            tuple(topk_indices.shape) != (B, S, topk) or tuple(grad_scores.shape) != (B, S, topk):
        raise ValueError("indexer tensors do not have matching shapes")
    shp = _lib.Shape(B, S, index_k.shape[0], H, D, topk)
    dq = torch.empty_like(index_q)
    lib = _lib.load()
    with torch.cuda.device(index_q.device):
        _lib.check("smqa_batched_indexer_bwd", lib.smqa_batched_indexer_bwd(
            _ptr(index_q), _ptr(weights), _ptr(index_k), _ptr(topk_indices), _ptr(grad_scores),
            shp, _ptr(dq), _stream(index_q.device)))
    return dq


class SparseMQAFunction(torch.autograd.Function):
    """Autograd around the forward and backward kernels: gradients flow from
    O to q, kv and attn_sink (the LSE output is not differentiable)."""

    @staticmethod
    def forward(ctx, q, kv, attn_sink, topk_idxs, sm_scale=None, check_status=False):
        o, lse = sparse_mqa_fwd_interface(q, kv, attn_sink, topk_idxs, sm_scale,
                                          check_status=check_status)
        ctx.save_for_backward(q, kv, attn_sink, topk_idxs, o, lse)
        ctx.sm_scale = sm_scale
        ctx.check_status = check_status
        ctx.mark_non_differentiable(lse)
        return o, lse

    @staticmethod
    def backward(ctx, do, dlse):
        q, kv, attn_sink, topk_idxs, o, lse = ctx.saved_tensors
        dq, dkv, dsink = sparse_mqa_bwd_interface(
            q, kv, attn_sink, o, do.to(torch.bfloat16).contiguous(), topk_idxs, lse,
            ctx.sm_scale, return_dsink=True, check_status=ctx.check_status)
        return dq, dkv, dsink.to(attn_sink.dtype), None, None, None


def sparse_mqa(q: torch.Tensor, kv: torch.Tensor, attn_sink: torch.Tensor,
               topk_idxs: torch.Tensor, sm_scale: Optional[float] = None,
               check_status: bool = False) -> tuple[torch.Tensor, torch.Tensor]:
    """Differentiable top-k sparse MQA: (O, LSE) as sparse_mqa_fwd_interface
    returns them, with gradients w.r.t. q, kv and attn_sink through O.  With
    ``check_status`` the forward and the backward each synchronize and raise
    SMQAError if a kernel's bounded wait ran out."""
    return SparseMQAFunction.apply(q, kv, attn_sink, topk_idxs, sm_scale, check_status)
