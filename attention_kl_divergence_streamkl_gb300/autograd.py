"""Autograd entry point: the attention KL divergence as a differentiable loss.

``attention_kl(q1, k1, q2, k2)`` returns KL(P1 || P2) per query row (or its mean
or sum) with P_t = softmax(scale Q_t K_t^T).  The forward is streamkl_fwd; the
backward calls the recompute backward of the StreamKL technical summary
(gist.science/ja/paper/2606.20005, section 手法 2) in whichever settings the
inputs need: setting 1 (P1 held fixed) for gradients of Q2/K2, setting 2 (P2
held fixed) for gradients of Q1/K1, both when both sides require grad (in one
call, which rebuilds each logit tile pair once for both settings where that is
faster).  Only
the reduction of the per-row values to a scalar happens in PyTorch.
"""
from __future__ import annotations

import torch

from . import _lib


class _AttentionKL(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q1, k1, q2, k2, scale, causal, reduction, bwd_mode):
        kl, lse1, lse2 = _lib.fwd(q1, k1, q2, k2, scale, causal)
        ctx.save_for_backward(q1, k1, q2, k2, kl, lse1, lse2)
        ctx.scale, ctx.causal, ctx.reduction, ctx.bwd_mode = scale, causal, reduction, bwd_mode
        if reduction == "none":
            return kl
        return kl.sum() if reduction == "sum" else kl.mean()

    @staticmethod
    def backward(ctx, grad_out):
        q1, k1, q2, k2, kl, lse1, lse2 = ctx.saved_tensors
        if ctx.reduction == "none":
            g = grad_out.contiguous().float()
        else:
            w = 1.0 if ctx.reduction == "sum" else 1.0 / kl.numel()
            g = (grad_out.float() * w).expand_as(kl).contiguous()
        need1 = ctx.needs_input_grad[0] or ctx.needs_input_grad[1]
        need2 = ctx.needs_input_grad[2] or ctx.needs_input_grad[3]
        dq1 = dk1 = dq2 = dk2 = None
        if need1 and need2 and ctx.bwd_mode in (_lib.BWD_AUTO, _lib.BWD_FUSED, _lib.BWD_SEPARATE):
            # the mutual case in one call (the library picks one recompute for both settings, or a pass each)
            return (*_lib.bwd_mutual(q1, k1, q2, k2, lse1, lse2, kl, g, ctx.scale, ctx.causal, ctx.bwd_mode),
                    None, None, None, None)
        if need2:
            dq2, dk2 = _lib.bwd_s1(q1, k1, q2, k2, lse1, lse2, g, ctx.scale, ctx.causal, ctx.bwd_mode)
        if need1:
            dq1, dk1 = _lib.bwd_s2(q1, k1, q2, k2, lse1, lse2, kl, g, ctx.scale, ctx.causal, ctx.bwd_mode)
        return dq1, dk1, dq2, dk2, None, None, None, None


def attention_kl(q1, k1, q2, k2, scale=None, causal=False, reduction="mean", bwd_mode=_lib.BWD_AUTO):
    """KL(softmax(scale Q1 K1^T) || softmax(scale Q2 K2^T)) per row, reduced by `reduction`.

    q_t: [B, H, N_Q, D] and k_t: [B, H, N_K, D] bf16 CUDA tensors; reduction is
    "mean" (over all B*H*N_Q rows), "sum" or "none" (fp32 [B, H, N_Q]).
    """
    if reduction not in ("mean", "sum", "none"):
        raise ValueError("reduction must be 'mean', 'sum' or 'none'")
    return _AttentionKL.apply(q1, k1, q2, k2, scale, causal, reduction, bwd_mode)
