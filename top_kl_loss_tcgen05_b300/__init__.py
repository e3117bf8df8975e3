"""Offline top-K knowledge distillation on one B300 (sm_103a).

Python side of libkd (C ABI in include/kd.h). PyTorch supplies device memory
and the current stream. Every step of the computation runs in libkd's CUDA
kernels. This module only checks shapes and passes pointers.

    ids, logp = topk_cache(teacher_logits, K)                  # offline cache
    loss = FusedKL.apply(H, W, ids, logp, chunk)               # fused chunked KL
    loss.backward()                                            # dH, dW

The method: "ทำให้ Knowledge Distillation มีประสิทธิภาพ คุ้มค่า และใช้งานได้จริงใน
ระดับ Scale ใหญ่" (ai-thai.com), sections "การทำ Distillation แบบ Offline" (the
top-K cache) and "กลไก Fused Chunked KL Loss" (the fused chunked loss).
"""

from __future__ import annotations

import ctypes

import torch

from . import _native
from ._native import KDError, check, status_string  # noqa: F401

__all__ = [
    "topk_cache",
    "teacher_topk_cache",
    "fused_kl_workspace",
    "fused_kl_fwd",
    "fused_kl_bwd",
    "fused_kl_fwdbwd",
    "FusedKL",
    "read_device_status",
    "KDError",
]

_WS_ALIGN = 256


def _stream_ptr(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def workspace(nbytes: int, device) -> torch.Tensor:
    """A caller-owned workspace (uint8, 256-byte aligned) of at least nbytes."""
    buf = torch.empty(int(nbytes) + _WS_ALIGN, dtype=torch.uint8, device=device)
    off = (-buf.data_ptr()) % _WS_ALIGN
    ws = buf[off : off + int(nbytes)]
    ws.zero_()
    return ws


def read_device_status(ws: torch.Tensor) -> int:
    """Synchronise the current stream; return and clear the workspace status word."""
    return _native.lib().kd_read_device_status(ws.data_ptr(), _stream_ptr(ws.device))


# ----------------------------------------------------------------- top-K cache


def topk_cache(logits: torch.Tensor, K: int, ws: torch.Tensor | None = None):
    """Teacher logits [T, V] (bf16 or fp32, rows may be strided) ->
    (ids int32 [T, K], logp float32 [T, K]): the K largest logits per row,
    value-descending then id-ascending, and their full-vocabulary log-softmax."""
    if logits.dim() != 2:
        raise ValueError("logits must be [T, V]")
    if logits.dtype == torch.bfloat16:
        dt = _native.KD_BF16
    elif logits.dtype == torch.float32:
        dt = _native.KD_F32
    else:
        raise TypeError("logits must be bf16 or fp32")
    if not logits.is_cuda or logits.stride(1) != 1:
        raise ValueError("logits must be a CUDA tensor with unit column stride")
    T, V = logits.shape
    dev = logits.device
    ids = torch.empty(T, K, dtype=torch.int32, device=dev)
    logp = torch.empty(T, K, dtype=torch.float32, device=dev)
    L = _native.lib()
    need = L.kd_topk_workspace_size(T, V, K, dt)
    if ws is None:
        ws = workspace(need, dev)
    check(
        "kd_topk_cache",
        L.kd_topk_cache(logits.data_ptr(), dt, T, V, logits.stride(0), K, ids.data_ptr(), logp.data_ptr(),
                        ws.data_ptr(), ws.numel(), _stream_ptr(dev)),
    )
    return ids, logp


def teacher_topk_cache(H: torch.Tensor, W: torch.Tensor, K: int, chunk: int = 1024, ws: torch.Tensor | None = None):
    """Top-K cache straight from teacher hidden states H [T, d] bf16 and LM
    head W [V, d] bf16 (logits computed in fp32, one chunk at a time, never
    all at once): (ids [T, K] int32, logp [T, K] float32)."""
    _need(H, "H", torch.bfloat16)
    dev = H.device
    _need(W, "W", torch.bfloat16, dev)
    if H.dim() != 2 or W.dim() != 2 or H.shape[1] != W.shape[1]:
        raise ValueError("H [T, d] and W [V, d] required")
    T, d = H.shape
    V = W.shape[0]
    if ws is None:
        n = _native.lib().kd_teacher_topk_workspace_size(d, V, K, chunk)
        if n == 0:
            raise ValueError("invalid sizes")
        ws = workspace(n, dev)
    ids = torch.empty(T, K, dtype=torch.int32, device=dev)
    logp = torch.empty(T, K, dtype=torch.float32, device=dev)
    check(
        "kd_teacher_topk_cache",
        _native.lib().kd_teacher_topk_cache(H.data_ptr(), W.data_ptr(), T, d, V, K, chunk, ids.data_ptr(),
                                            logp.data_ptr(), ws.data_ptr(), ws.numel(), _stream_ptr(dev)),
    )
    return ids, logp


# ----------------------------------------------------------------- fused KL


def fused_kl_workspace(d: int, V: int, K: int, chunk: int, device, group: int = 0) -> torch.Tensor:
    """Workspace of the fused loss calls for this chunk and group (0 = the
    default group rule of include/kd.h)."""
    n = _native.lib().kd_fused_kl_workspace_size_ex(d, V, K, chunk, int(group))
    if n == 0:
        raise ValueError("invalid sizes")
    return workspace(n, device)


def _check_fused(H, W, ids, logp):
    _need(H, "H", torch.bfloat16)
    dev = H.device
    _need(W, "W", torch.bfloat16, dev)
    _need(ids, "ids", torch.int32, dev)
    _need(logp, "logp", torch.float32, dev)
    if H.dim() != 2 or W.dim() != 2 or H.shape[1] != W.shape[1]:
        raise ValueError("H [T, d] and W [V, d] required")
    if ids.shape != logp.shape or ids.dim() != 2 or ids.shape[0] != H.shape[0]:
        raise ValueError("ids and logp must be [T, K]")
    return H.shape[0], H.shape[1], W.shape[0], ids.shape[1]


def _options(T, dev, temperature, mask, mean_over_mask, dH_bf16, group=0):
    """kd_kl_options for the _ex calls, or None when every option is at its
    default (the plain behaviour). Returns (struct or None, mask tensor)."""
    if temperature == 1.0 and mask is None and not mean_over_mask and not dH_bf16 and not group:
        return None, None
    m = None
    if mask is not None:
        m = mask
        if m.dtype == torch.bool:
            m = m.view(torch.uint8)
        _need(m, "mask", torch.uint8, dev)
        if m.dim() != 1 or m.shape[0] != T:
            raise ValueError("mask must be [T]")
    o = _native.KLOptions(float(temperature), m.data_ptr() if m is not None else None, 1 if mean_over_mask else 0,
                          1 if dH_bf16 else 0, int(group))
    return o, m


def _optp(o):
    return ctypes.byref(o) if o is not None else None


def fused_kl_fwd(H, W, ids, logp, chunk: int, ws=None, want_rows: bool = False, temperature: float = 1.0,
                 mask=None, mean_over_mask: bool = False, group: int = 0):
    """Forward: (loss [] f32, lse [T] f32, loss_rows [T] f32 or None).

    temperature, mask, mean_over_mask and group are the kd_kl_options of
    include/kd.h (student softmax(z / tau), tempered teacher; positions with
    mask == 0 excluded; the mean over T or over the included positions;
    chunks per GEMM launch, 0 = default)."""
    T, d, V, K = _check_fused(H, W, ids, logp)
    dev = H.device
    if ws is None:
        ws = fused_kl_workspace(d, V, K, chunk, dev, group)
    o, _m = _options(T, dev, temperature, mask, mean_over_mask, False, group)
    loss = torch.empty((), dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    rows = torch.empty(T, dtype=torch.float32, device=dev) if want_rows else None
    check(
        "kd_fused_kl_fwd_ex",
        _native.lib().kd_fused_kl_fwd_ex(H.data_ptr(), W.data_ptr(), ids.data_ptr(), logp.data_ptr(), T, d, V, K,
                                         chunk, loss.data_ptr(), lse.data_ptr(), _ptr(rows), _optp(o),
                                         ws.data_ptr(), ws.numel(), _stream_ptr(dev)),
    )
    return loss, lse, rows


def _grad_outputs(T, d, V, dev, dH, dW, dH_bf16, want_dH, want_dW):
    """The dH / dW output tensors (allocated when not given), or None for a
    gradient that is not wanted (libkd then skips its GEMM)."""
    if not (want_dH or want_dW):
        raise ValueError("want_dH and want_dW are both False: nothing to compute")
    dh_dtype = torch.bfloat16 if dH_bf16 else torch.float32
    if not want_dH:
        dH = None
    elif dH is None:
        dH = torch.empty(T, d, dtype=dh_dtype, device=dev)
    if not want_dW:
        dW = None
    elif dW is None:
        dW = torch.empty(V, d, dtype=torch.float32, device=dev)
    if dH is not None:
        _need(dH, "dH", dh_dtype, dev)
    if dW is not None:
        _need(dW, "dW", torch.float32, dev)
    return dH, dW


def fused_kl_bwd(H, W, ids, logp, lse, chunk: int, grad_scale: float, grad_scale_dev=None, dH=None, dW=None,
                 accumulate_dW: bool = False, ws=None, temperature: float = 1.0, mask=None,
                 mean_over_mask: bool = False, dH_bf16: bool = False, group: int = 0, want_dH: bool = True,
                 want_dW: bool = True):
    """Backward: (dH [T, d] f32 (bf16 with dH_bf16), dW [V, d] f32) for
    dz = s (q - p); s = grad_scale * grad_scale_dev * 1/tau, times 1/N when
    mean_over_mask (then grad_scale is d objective / d loss). want_dH /
    want_dW = False skips that gradient (its GEMM does not run) and returns
    None in its place."""
    T, d, V, K = _check_fused(H, W, ids, logp)
    dev = H.device
    _need(lse, "lse", torch.float32, dev)
    if ws is None:
        ws = fused_kl_workspace(d, V, K, chunk, dev, group)
    dH, dW = _grad_outputs(T, d, V, dev, dH, dW, dH_bf16, want_dH, want_dW)
    if grad_scale_dev is not None:
        _need(grad_scale_dev, "grad_scale_dev", torch.float32, dev)
    o, _m = _options(T, dev, temperature, mask, mean_over_mask, dH_bf16, group)
    check(
        "kd_fused_kl_bwd_ex",
        _native.lib().kd_fused_kl_bwd_ex(H.data_ptr(), W.data_ptr(), ids.data_ptr(), logp.data_ptr(),
                                         lse.data_ptr(), T, d, V, K, chunk, float(grad_scale), _ptr(grad_scale_dev),
                                         _ptr(dH), _ptr(dW), 1 if accumulate_dW else 0, _optp(o),
                                         ws.data_ptr(), ws.numel(), _stream_ptr(dev)),
    )
    return dH, dW


def fused_kl_fwdbwd(H, W, ids, logp, chunk: int, grad_scale: float | None = None, grad_scale_dev=None, dH=None,
                    dW=None, accumulate_dW: bool = False, ws=None, want_rows: bool = False, temperature: float = 1.0,
                    mask=None, mean_over_mask: bool = False, dH_bf16: bool = False, group: int = 0,
                    want_dH: bool = True, want_dW: bool = True):
    """Forward and backward in one call, without recomputing the logits:
    (loss, lse, loss_rows or None, dH, dW). grad_scale defaults to the
    gradient of the loss itself: 1/T, or 1 with mean_over_mask (the library
    then applies 1/N). want_dH / want_dW as in fused_kl_bwd."""
    T, d, V, K = _check_fused(H, W, ids, logp)
    dev = H.device
    if ws is None:
        ws = fused_kl_workspace(d, V, K, chunk, dev, group)
    if grad_scale is None:
        grad_scale = 1.0 if (mean_over_mask and mask is not None) else 1.0 / T
    loss = torch.empty((), dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    rows = torch.empty(T, dtype=torch.float32, device=dev) if want_rows else None
    dH, dW = _grad_outputs(T, d, V, dev, dH, dW, dH_bf16, want_dH, want_dW)
    if grad_scale_dev is not None:
        _need(grad_scale_dev, "grad_scale_dev", torch.float32, dev)
    o, _m = _options(T, dev, temperature, mask, mean_over_mask, dH_bf16, group)
    check(
        "kd_fused_kl_fwdbwd_ex",
        _native.lib().kd_fused_kl_fwdbwd_ex(H.data_ptr(), W.data_ptr(), ids.data_ptr(), logp.data_ptr(), T, d, V, K,
                                            chunk, float(grad_scale), _ptr(grad_scale_dev), loss.data_ptr(),
                                            lse.data_ptr(), _ptr(rows), _ptr(dH), _ptr(dW),
                                            1 if accumulate_dW else 0, _optp(o), ws.data_ptr(), ws.numel(),
                                            _stream_ptr(dev)),
    )
    return loss, lse, rows, dH, dW


class FusedKL(torch.autograd.Function):
    """loss = mean KL(p_teacher,topK || softmax(W h_t)), fused and chunked.

    FusedKL.apply(H, W, ids, logp, chunk, temperature=1.0, mask=None,
    mean_over_mask=False, group=0). Forward saves only lse [T] (4 bytes per
    position). Backward recomputes each chunk's logits. The upstream gradient
    goes to the kernels as a device scalar, so backward does not synchronise.
    dH comes out of the kernels in H's dtype when H is bf16. Only the
    gradients autograd asks for are computed: with a frozen LM head
    (W.requires_grad False) the dW GEMM does not run.
    """

    @staticmethod
    def forward(ctx, H, W, ids, logp, chunk: int, temperature: float = 1.0, mask=None, mean_over_mask: bool = False,
                group: int = 0):
        ws = fused_kl_workspace(H.shape[1], W.shape[0], ids.shape[1], chunk, H.device, group)
        loss, lse, _ = fused_kl_fwd(H, W, ids, logp, chunk, ws=ws, temperature=temperature, mask=mask,
                                    mean_over_mask=mean_over_mask, group=group)
        ctx.save_for_backward(H, W, ids, logp, lse)
        ctx.chunk, ctx.ws, ctx.group = chunk, ws, group
        ctx.temperature, ctx.mask, ctx.mean_over_mask = temperature, mask, mean_over_mask
        return loss

    @staticmethod
    def backward(ctx, g):
        H, W, ids, logp, lse = ctx.saved_tensors
        want_dH, want_dW = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        if not (want_dH or want_dW):
            return None, None, None, None, None, None, None, None, None
        g = g.detach().to(torch.float32).contiguous()
        over_mask = bool(ctx.mean_over_mask) and ctx.mask is not None
        dH, dW = fused_kl_bwd(H, W, ids, logp, lse, ctx.chunk, 1.0 if over_mask else 1.0 / H.shape[0],
                              grad_scale_dev=g, ws=ctx.ws, temperature=ctx.temperature, mask=ctx.mask,
                              mean_over_mask=ctx.mean_over_mask, dH_bf16=H.dtype == torch.bfloat16,
                              group=ctx.group, want_dH=want_dH, want_dW=want_dW)
        return dH, dW, None, None, None, None, None, None, None
