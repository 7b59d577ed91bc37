"""A CPU stand-in for the kernels that shard.py calls, for gloo tests of the
partition and exchange logic on machines without a GPU.  Test infrastructure:
it computes each call's documented result with the fp64 oracle's functions
(logits, masks, softmax statistics, dlogits) on torch tensors; nothing here is
used by the library itself.

Partial sets follow the library's contract for key shards: per row
(m1, m2, l1, l2, acc) over the shard's keys, m_t = max_j c s_t,j with
c = scale log2(e) and s the raw dot product, l_t = sum_j 2^(c s_t,j - m_t),
acc = sum_j 2^(c s_1,j - m1) (s_1,j - s_2,j); (-inf, -inf, 0, 0, 0) for a row
that sees none of the shard's keys.
"""
from __future__ import annotations

import math
import types

import numpy as np
import torch

from oracle import oracle as O

LOG2E = 1.0 / math.log(2.0)


def _np(t):
    return t.detach().double().cpu().numpy()


def _scale(scale, D):
    return scale if scale else 1.0 / math.sqrt(D)


def fwd(q1, k1, q2, k2, scale=None, causal=False):
    kl, l1, l2 = O.forward(_np(q1), _np(k1), _np(q2), _np(k2), _scale(scale, q1.shape[3]), causal)
    return tuple(torch.from_numpy(x) for x in (kl, l1, l2))


def _bwd(setting, q1, k1, q2, k2, g, scale, causal):
    dq, dk = O.backward(setting, _np(q1), _np(k1), _np(q2), _np(k2), _scale(scale, q1.shape[3]), causal, _np(g))
    return torch.from_numpy(dq), torch.from_numpy(dk)


def bwd_s1(q1, k1, q2, k2, lse1, lse2, g, scale=None, causal=False, bwd_mode=0):
    return _bwd(1, q1, k1, q2, k2, g, scale, causal)


def bwd_s2(q1, k1, q2, k2, lse1, lse2, kl, g, scale=None, causal=False, bwd_mode=0):
    return _bwd(2, q1, k1, q2, k2, g, scale, causal)


def _shard_keep(nq, nk, key_offset, nk_total, causal):
    return O.causal_mask(np.arange(nq), nq, nk_total, causal)[:, key_offset:key_offset + nk]


def fwd_partials(q1, k1, q2, k2, key_offset, nk_total, scale=None, causal=False):
    B, H, NQ, D = q1.shape
    c = _scale(scale, D) * LOG2E
    keep = _shard_keep(NQ, k1.shape[2], key_offset, nk_total, causal)
    out = np.zeros((B, H, NQ, 5))
    for b in range(B):
        for h in range(H):
            s1 = O.logits(_np(q1[b, h]), _np(k1[b, h]), 1.0)
            s2 = O.logits(_np(q2[b, h]), _np(k2[b, h]), 1.0)
            for i in range(NQ):
                kk = keep[i]
                if not kk.any():
                    out[b, h, i] = (-np.inf, -np.inf, 0.0, 0.0, 0.0)
                    continue
                x1, x2 = c * s1[i, kk], c * s2[i, kk]
                m1, m2 = x1.max(), x2.max()
                w1 = np.exp2(x1 - m1)
                out[b, h, i] = (m1, m2, w1.sum(), np.exp2(x2 - m2).sum(), float(w1 @ (s1[i, kk] - s2[i, kk])))
    return torch.from_numpy(out)


def merge_partials(parts, D, scale=None):
    p = _np(parts)  # [S, B, H, NQ, 5]
    M1, M2 = p[..., 0].max(axis=0), p[..., 1].max(axis=0)
    w1, w2 = np.exp2(p[..., 0] - M1), np.exp2(p[..., 1] - M2)
    l1, l2 = (p[..., 2] * w1).sum(axis=0), (p[..., 3] * w2).sum(axis=0)
    acc = (p[..., 4] * w1).sum(axis=0)
    lse1, lse2 = (M1 + np.log2(l1)) / LOG2E, (M2 + np.log2(l2)) / LOG2E
    kl = _scale(scale, D) * acc / l1 + lse2 - lse1
    return tuple(torch.from_numpy(x) for x in (kl, lse1, lse2))


def bwd_keyshard(setting, q1, k1, q2, k2, key_offset, nk_total, lse1, lse2, kl, g, scale=None, causal=False):
    B, H, NQ, D = q1.shape
    nk = k1.shape[2]
    sc = _scale(scale, D)
    keep = _shard_keep(NQ, nk, key_offset, nk_total, causal)
    dq = np.zeros((B, H, NQ, D))
    dk = np.zeros((B, H, nk, D))
    for b in range(B):
        for h in range(H):
            S1 = O.logits(_np(q1[b, h]), _np(k1[b, h]), sc)
            S2 = O.logits(_np(q2[b, h]), _np(k2[b, h]), sc)
            P1 = np.where(keep, np.exp(S1 - _np(lse1[b, h])[:, None]), 0.0)
            P2 = np.where(keep, np.exp(S2 - _np(lse2[b, h])[:, None]), 0.0)
            dS = O.dlogits(setting, P1, P2, _np(kl[b, h]), _np(g[b, h]))
            qo, ko = (q2, k2) if setting == 1 else (q1, k1)
            dq[b, h] = dS @ _np(ko[b, h])            # unscaled: dQ = scale * sum over shards
            dk[b, h] = sc * (dS.T @ _np(qo[b, h]))
    return torch.from_numpy(dq), torch.from_numpy(dk)


def dq_from_partial(dq_partial, q_like, scale=None):
    return _scale(scale, dq_partial.shape[3]) * dq_partial.double()


OPS = types.SimpleNamespace(fwd=fwd, bwd_s1=bwd_s1, bwd_s2=bwd_s2, fwd_partials=fwd_partials,
                            merge_partials=merge_partials, bwd_keyshard=bwd_keyshard, dq_from_partial=dq_from_partial)
