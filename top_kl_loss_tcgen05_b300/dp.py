"""Position-sharded data parallelism for the fused chunked KL loss.

The loss is a mean over positions of per-position terms, and the method
already computes it one chunk of positions at a time ("ทำให้ Knowledge
Distillation มีประสิทธิภาพ..." (ai-thai.com), section "กลไก Fused Chunked KL
Loss"). Across GPUs the natural split is the same one: each rank holds a
contiguous shard of the T positions (its rows of H and of the teacher cache)
and a full replica of the LM head W. Then, with T_global positions in all:

  * every rank runs the loss on its shard with the gradient scale
    1 / T_global (times the upstream gradient), so its dz, dH and dW are
    exactly its share of the gradient of the global mean;
  * the global loss is the sum over ranks of the shards' loss sums, divided
    by T_global: one scalar all-reduce;
  * dH stays local (it is the gradient of the rank's own H rows);
  * dW is the sum over ranks of the shards' dW: one all-reduce of [V, d]
    fp32, the ordinary data-parallel gradient sync.

Nothing else crosses ranks. The collectives are plain torch.distributed
calls (NCCL between GPUs); every other step runs in libkd's kernels on each
rank's own GPU. The per-shard call is an argument, so the reduction logic
can be checked with any implementation of the loss on the shard.
"""

from __future__ import annotations

from typing import Callable, NamedTuple

import torch
import torch.distributed as dist

from . import fused_kl_bwd, fused_kl_fwd, fused_kl_fwdbwd

__all__ = ["shard_range", "ShardResult", "libkd_shard_call", "dp_fused_kl_step", "DPFusedKL"]


def shard_range(T_global: int, world: int, rank: int) -> tuple[int, int]:
    """[t0, t1) of rank `rank`: contiguous shards whose sizes differ by at
    most one position, in rank order."""
    if world < 1 or not 0 <= rank < world or T_global < 0:
        raise ValueError("bad shard request")
    base, extra = divmod(T_global, world)
    t0 = rank * base + min(rank, extra)
    return t0, t0 + base + (1 if rank < extra else 0)


class ShardResult(NamedTuple):
    loss_sum: torch.Tensor  # scalar: sum over the shard's positions of L_t
    dH: torch.Tensor        # [T_shard, d]: gradient of the rank's H rows
    dW: torch.Tensor        # [V, d] fp32: the shard's contribution to dW


ShardCall = Callable[..., ShardResult]


def libkd_shard_call(H, W, ids, logp, chunk: int, grad_scale: float, grad_scale_dev=None, group: int = 0):
    """The loss on one shard through libkd's single call (kd_fused_kl_fwdbwd):
    loss sum over the shard and the gradients for dz scaled by grad_scale
    (times *grad_scale_dev)."""
    T = H.shape[0]
    loss, _, _, dH, dW = fused_kl_fwdbwd(H, W, ids, logp, chunk, grad_scale=grad_scale,
                                         grad_scale_dev=grad_scale_dev, group=group)
    return ShardResult(loss * T, dH, dW)


def _empty_shard(H, W) -> ShardResult:
    """What a rank without positions contributes: no loss, no dH rows and a
    zero dW (in the precision the loss would return it: fp32 for bf16, fp16
    or fp32 weights). The loss itself is not called, since it refuses T = 0;
    the rank still joins every collective."""
    dW_dtype = torch.promote_types(W.dtype, torch.float32)
    return ShardResult(torch.zeros((), dtype=torch.float64, device=W.device),
                       torch.zeros((0, H.shape[1]), dtype=dW_dtype, device=H.device),
                       torch.zeros(W.shape, dtype=dW_dtype, device=W.device))


def _distributed() -> bool:
    """True when a default process group exists: the collectives then run
    (a one-rank group included)."""
    return dist.is_available() and dist.is_initialized()


def dp_fused_kl_step(H, W, ids, logp, chunk: int, T_global: int, shard_call: ShardCall = libkd_shard_call,
                     process_group=None, grad_scale: float = 1.0):
    """One forward + backward of the global-mean loss, position-sharded.

    H, ids, logp hold this rank's positions (any shard sizes, summing to
    T_global over the ranks); W is the full LM head on every rank.
    shard_call(H, W, ids, logp, chunk, s) must return a ShardResult for dz
    scaled by s. It is called with s = grad_scale / T_global.
    Returns (loss, dH, dW): the global mean loss (the same on every rank),
    this rank's dH rows, and the summed dW (the same on every rank). With no
    process group initialised there are no collectives: the result is the
    shard's share of the global loss and gradient."""
    if T_global <= 0:
        raise ValueError("T_global must be positive")
    if H.shape[0] == 0:  # more ranks than positions: this one has none
        r = _empty_shard(H, W)
    else:
        r = shard_call(H, W, ids, logp, chunk, grad_scale / T_global)
    loss_sum = r.loss_sum.detach().reshape(1).to(torch.float64)
    dW = r.dW
    if _distributed():
        dist.all_reduce(loss_sum, op=dist.ReduceOp.SUM, group=process_group)
        dist.all_reduce(dW, op=dist.ReduceOp.SUM, group=process_group)
    return (loss_sum / T_global).to(torch.float32).reshape(()), r.dH, dW


class DPFusedKL(torch.autograd.Function):
    """The global-mean fused KL loss over position shards, for autograd.

    DPFusedKL.apply(H_shard, W, ids_shard, logp_shard, chunk, T_global,
    process_group=None). Forward: libkd's forward on the shard, then one
    scalar all-reduce of the loss sum. Backward: libkd's recompute backward
    on the shard with the gradient scale 1 / T_global and the upstream
    gradient as a device scalar, then an all-reduce of dW; dH stays local.
    Only the gradients autograd asks for are computed (a frozen LM head
    skips the dW GEMM and its all-reduce, on every rank alike). Saves only
    the shard's lse (4 bytes per position). A rank whose shard is empty
    contributes zeros and still joins both all-reduces."""

    @staticmethod
    def forward(ctx, H, W, ids, logp, chunk: int, T_global: int, process_group=None):
        if H.shape[0] == 0:
            lse = torch.zeros(0, dtype=torch.float32, device=H.device)
            loss_sum = torch.zeros(1, dtype=torch.float64, device=H.device)
        else:
            loss, lse, _ = fused_kl_fwd(H, W, ids, logp, chunk)
            loss_sum = (loss.to(torch.float64) * H.shape[0]).reshape(1)
        if _distributed():
            dist.all_reduce(loss_sum, op=dist.ReduceOp.SUM, group=process_group)
        ctx.save_for_backward(H, W, ids, logp, lse)
        ctx.chunk, ctx.T_global, ctx.pg = chunk, T_global, process_group
        return (loss_sum / T_global).to(torch.float32).reshape(())

    @staticmethod
    def backward(ctx, g):
        H, W, ids, logp, lse = ctx.saved_tensors
        want_dH, want_dW = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        if not (want_dH or want_dW):
            return None, None, None, None, None, None, None
        if H.shape[0] == 0:
            dH = torch.zeros_like(H) if want_dH else None
            dW = torch.zeros(W.shape, dtype=torch.float32, device=W.device) if want_dW else None
        else:
            g = g.detach().to(torch.float32).contiguous()
            dH, dW = fused_kl_bwd(H, W, ids, logp, lse, ctx.chunk, 1.0 / ctx.T_global, grad_scale_dev=g,
                                  dH_bf16=H.dtype == torch.bfloat16, want_dH=want_dH, want_dW=want_dW)
        if want_dW and _distributed():
            dist.all_reduce(dW, op=dist.ReduceOp.SUM, group=ctx.pg)
        return dH, dW, None, None, None, None, None
