"""The attention-KL path split over several GPUs, one process per GPU.

Two exact partitions (torch.distributed moves the data; every arithmetic step
runs in libstreamkl's kernels):

* **heads** -- every (batch, head) is an independent problem, so each rank
  takes a contiguous block of heads and runs the ordinary forward and
  backward on it.  The only exchange is the loss: an all-reduce of the
  per-rank sums of g_i KL_i.  Gradients stay with the rank that owns the head.
* **keys** (context parallelism) -- each rank holds a contiguous range of the
  keys of every head and all query rows.  The forward reduces the rank's keys
  to the five running scalars per row (m1, m2, l1, l2, acc) and all-gathers
  them; every rank then merges the gathered sets exactly, the merge of the
  Split-K variant (StreamKL technical summary, gist.science/ja/paper/2606.20005,
  section 手法 3), and holds the whole KL, LSE1, LSE2.  The backward recomputes
  P_t = exp(S_t - LSE_t) (section 手法 2) from those merged values over the
  rank's keys: its dK rows are complete (every query row is local) and its
  contribution to dQ is all-reduced.

``ops`` is the set of kernels the sharded calls use (fwd, bwd_s1, bwd_s2,
fwd_partials, merge_partials, bwd_keyshard, dq_from_partial, with the
signatures of this package's functions); it defaults to libstreamkl's.
"""
from __future__ import annotations

import types

import torch
import torch.distributed as dist

from . import _lib

DEFAULT_OPS = types.SimpleNamespace(fwd=_lib.fwd, bwd_s1=_lib.bwd_s1, bwd_s2=_lib.bwd_s2,
                                    fwd_partials=_lib.fwd_partials, merge_partials=_lib.merge_partials,
                                    bwd_keyshard=_lib.bwd_keyshard, dq_from_partial=_lib.dq_from_partial)


def split_range(n: int, parts: int, rank: int, align: int = 1) -> tuple[int, int]:
    """[lo, hi) of part `rank` when n items are cut into `parts` contiguous ranges.

    Cut points are multiples of `align` (the last range takes the remainder),
    spread so that the ranges differ by at most one aligned block; a range may
    be empty when there are fewer blocks than parts.
    """
    if parts < 1 or not 0 <= rank < parts or n < 0 or align < 1:
        raise ValueError("bad split")
    blocks = -(-n // align)
    cut = lambda r: min(n, ((blocks * r) // parts) * align)  # noqa: E731
    return cut(rank), cut(rank + 1)


def _world(group) -> tuple[int, int]:
    if not (dist.is_available() and dist.is_initialized()):
        return 1, 0
    return dist.get_world_size(group), dist.get_rank(group)


# ------------------------------------------------------------------------------ heads

def head_range(H: int, group=None) -> tuple[int, int]:
    """The heads [h0, h1) this rank owns."""
    world, rank = _world(group)
    return split_range(H, world, rank)


def heads_forward(q1, k1, q2, k2, scale=None, causal=False, g=None, group=None, ops=DEFAULT_OPS):
    """Forward on this rank's heads ([B, h1 - h0, N, D] slices) and the job's loss.

    Returns (kl, lse1, lse2, loss): the local per-row values and the sum over
    every rank of sum_i g_i KL_i (g = 1 per row when None), all-reduced.
    """
    B, Hl, NQ, _ = q1.shape
    if Hl == 0:  # more ranks than heads: this rank owns none, but still joins the all-reduce
        kl, lse1, lse2 = (torch.zeros((B, 0, NQ), dtype=torch.float32, device=q1.device) for _ in range(3))
    else:
        kl, lse1, lse2 = ops.fwd(q1, k1, q2, k2, scale, causal)
    w = torch.ones_like(kl) if g is None else g
    loss = (w.double() * kl.double()).sum().reshape(1)
    if _world(group)[0] > 1:
        dist.all_reduce(loss, op=dist.ReduceOp.SUM, group=group)
    return kl, lse1, lse2, loss[0]


def heads_backward(setting, q1, k1, q2, k2, lse1, lse2, kl, g, scale=None, causal=False, ops=DEFAULT_OPS,
                   bwd_mode=_lib.BWD_AUTO):
    """Backward on this rank's heads: no exchange (each head's gradient is local)."""
    if q1.shape[1] == 0:  # a rank that owns no heads
        q, k = (q2, k2) if setting == 1 else (q1, k1)
        return torch.empty_like(q), torch.empty_like(k)
    if setting == 1:
        return ops.bwd_s1(q1, k1, q2, k2, lse1, lse2, g, scale, causal, bwd_mode)
    return ops.bwd_s2(q1, k1, q2, k2, lse1, lse2, kl, g, scale, causal, bwd_mode)


# ------------------------------------------------------------------------------ keys

def key_range(nk_total: int, group=None, align: int = 128) -> tuple[int, int]:
    """The keys [k0, k1) this rank owns (cut at multiples of the 128-key tile)."""
    world, rank = _world(group)
    return split_range(nk_total, world, rank, align)


def _all_gather(t: torch.Tensor, group) -> torch.Tensor:
    world, _ = _world(group)
    if world == 1:
        return t.unsqueeze(0)
    out = [torch.empty_like(t) for _ in range(world)]
    dist.all_gather(out, t.contiguous(), group=group)
    return torch.stack(out)


def keys_forward(q1, k1, q2, k2, key_offset: int, nk_total: int, scale=None, causal=False, group=None,
                 ops=DEFAULT_OPS):
    """KL, LSE1, LSE2 [B, H, N_Q] of the whole sequence from this rank's key shard.

    q_t hold every query row; k_t hold keys [key_offset, key_offset + k_t.shape[2])
    of nk_total.  Every rank returns the same merged values.  A rank may own no
    keys (k_t with zero rows): it contributes an empty partial set.
    """
    B, H, NQ, D = q1.shape
    if k1.shape[2] > 0:
        part = ops.fwd_partials(q1, k1, q2, k2, key_offset, nk_total, scale, causal)
    else:  # an empty shard: m = -inf, l = acc = 0 for every row
        part = torch.zeros((B, H, NQ, 5), dtype=torch.float32, device=q1.device)
        part[..., :2] = float("-inf")
    parts = _all_gather(part, group)
    return ops.merge_partials(parts, D, scale)


def keys_backward(setting, q1, k1, q2, k2, key_offset: int, nk_total: int, lse1, lse2, kl, g, scale=None,
                  causal=False, group=None, ops=DEFAULT_OPS):
    """(dQ, dK of this rank's keys) of the whole sequence, bf16.

    lse1, lse2, kl are keys_forward's merged values; g is dLoss/dKL_i for every
    row.  Each rank's unscaled dQ contribution is summed over the group
    (all-reduce), then scaled and rounded to bf16 by the library.
    """
    B, H, NQ, D = q1.shape
    if k1.shape[2] > 0:
        dq_part, dk = ops.bwd_keyshard(setting, q1, k1, q2, k2, key_offset, nk_total, lse1, lse2, kl, g, scale,
                                       causal)
    else:
        dq_part = torch.zeros((B, H, NQ, D), dtype=torch.float32, device=q1.device)
        dk = torch.empty_like(k1)
    if _world(group)[0] > 1:
        dist.all_reduce(dq_part, op=dist.ReduceOp.SUM, group=group)
    return ops.dq_from_partial(dq_part, q1 if setting == 2 else q2, scale), dk


class _KeyShardedKL(torch.autograd.Function):
    """KL per row of the whole sequence from this rank's key shard, differentiable (see keys_attention_kl)."""

    @staticmethod
    def forward(ctx, q1, k1, q2, k2, key_offset, nk_total, scale, causal, group, ops):
        kl, lse1, lse2 = keys_forward(q1, k1, q2, k2, key_offset, nk_total, scale, causal, group, ops)
        ctx.save_for_backward(q1, k1, q2, k2, kl, lse1, lse2)
        ctx.args = (key_offset, nk_total, scale, causal, group, ops)
        return kl

    @staticmethod
    def backward(ctx, grad_kl):
        q1, k1, q2, k2, kl, lse1, lse2 = ctx.saved_tensors
        key_offset, nk_total, scale, causal, group, ops = ctx.args
        g = grad_kl.contiguous().to(kl.dtype)
        dq1 = dk1 = dq2 = dk2 = None
        if ctx.needs_input_grad[2] or ctx.needs_input_grad[3]:
            dq2, dk2 = keys_backward(1, q1, k1, q2, k2, key_offset, nk_total, lse1, lse2, kl, g, scale, causal,
                                     group, ops)
        if ctx.needs_input_grad[0] or ctx.needs_input_grad[1]:
            dq1, dk1 = keys_backward(2, q1, k1, q2, k2, key_offset, nk_total, lse1, lse2, kl, g, scale, causal,
                                     group, ops)
        return dq1, dk1, dq2, dk2, None, None, None, None, None, None


def keys_attention_kl(q1, k1, q2, k2, key_offset: int, nk_total: int, scale=None, causal=False, group=None,
                      ops=DEFAULT_OPS):
    """Differentiable per-row KL [B, H, N_Q] of the whole sequence, computed from this rank's key shard.

    Every rank holds every query row (q_t replicated) and its own keys; every
    rank gets the same KL.  In the backward, the gradient of q_t is the whole
    dQ (the shards' contributions all-reduced, so replicated queries need no
    further reduction) and the gradient of k_t covers this rank's keys.  The
    upstream gradient must be the same on every rank, as it is for a loss
    computed from the returned KL on each rank.  Heads need no such function:
    with the heads split over ranks, attention_kl on each rank's heads gives
    that rank's gradients, and the job's loss is the all-reduced sum.
    """
    return _KeyShardedKL.apply(q1, k1, q2, k2, key_offset, nk_total, scale, causal, group, ops)


def mean_rows_grad(B: int, H: int, NQ: int, device=None, dtype=torch.float32) -> torch.Tensor:
    """g for a loss that is the mean of KL over all B * H * N_Q rows of the job."""
    return torch.full((B, H, NQ), 1.0 / max(B * H * NQ, 1), dtype=dtype, device=device)


def local_heads(t: torch.Tensor, group=None) -> torch.Tensor:
    """This rank's heads of a [B, H, N, D] (or [B, H, N]) tensor, as a view."""
    h0, h1 = head_range(t.shape[1], group)
    return t[:, h0:h1]


def local_keys(t: torch.Tensor, group=None, align: int = 128) -> tuple[torch.Tensor, int]:
    """(this rank's rows of a [B, H, N_K, D] key tensor as a view, the first row's index)."""
    k0, k1 = key_range(t.shape[2], group, align)
    return t[:, :, k0:k1], k0


__all__ = ["split_range", "head_range", "heads_forward", "heads_backward", "key_range", "keys_forward",
           "keys_backward", "keys_attention_kl", "mean_rows_grad", "local_heads", "local_keys", "DEFAULT_OPS"]
