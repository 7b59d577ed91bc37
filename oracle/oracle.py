"""fp64 CPU oracle for the attention KL divergence and its two gradients.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it.  It shares no code with
the CUDA path and imports nothing from the product package: callers hand it
plain float arrays (the bf16 inputs upcast to float64).

What it computes is the plain, materialised definition (the method being
replaced, described under "problem statement" of the StreamKL technical
summary, gist.science/ja/paper/2606.20005, section 問題提起): both attention
distributions are formed in full for a block of query rows, and the KL reduction
is taken element by element.  The online one-pass formulation of the pages
reaches the same numbers up to rounding order, so this is the reference the
kernels are compared against.

Notation (per batch b, head h):

    S_t = scale * Q_t K_t^T                       t in {1, 2}
    M_ij = [j <= i + N_K - N_Q]  (causal)  or 1    bottom-right aligned mask
    P_t = row-softmax of S_t over the unmasked keys
    LSE_t,i = log sum_j M_ij exp(S_t,ij)
    KL_i = sum_j P1_ij (log P1_ij - log P2_ij)    KL(P1 || P2), 0 log 0 := 0

P1 (teacher) is the first pair; the training objective is L = sum_i g_i KL_i.
Gradients, the two settings of the recompute backward (technical summary,
section 手法 2 "recompute strategy"):

* setting 1 (P1 held fixed, Q2/K2 optimised):   dS2 = g_i (P2 - P1)
* setting 2 (P2 held fixed, Q1/K1 optimised):   dS1 = g_i P1 (log P1 - log P2 - KL_i)

and for the optimised pair t:  dQ_t = scale dS_t K_t,  dK_t = scale dS_t^T Q_t.
Both dS formulas are the chain rule applied to the definition above; the tests
pin them with central finite differences and with torch autograd in fp64.

Parity pins (see tests/test_oracle_pins.py): finite differences, a library
routine (torch CPU fp64 kl_div + autograd), closed forms (identical pairs,
uniform keys, zero student queries, single-key causal row, two-key Bernoulli
case), invariants (KL >= 0, logit-shift invariance, dS row sums, the trace
identity), and the pages' own online identity KL = acc/l1 + LSE2 - LSE1.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "logits", "causal_mask", "row_softmax", "kl_from_probs", "head_forward", "dlogits",
    "head_backward_rows", "head_backward", "forward", "backward", "rows_forward", "rows_backward_dq",
    "materialised_distribution_bytes",
]

ROW_BLOCK = 256


def logits(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """S = scale * q k^T in float64 (q: [n, D], k: [m, D])."""
    return scale * (np.asarray(q, np.float64) @ np.asarray(k, np.float64).T)


def causal_mask(rows: np.ndarray, nq: int, nk: int, causal: bool) -> np.ndarray:
    """Boolean keep-mask [len(rows), nk]: key j is seen by row i iff j <= i + nk - nq.

    The pages only say "causal"; every causal workload has N_Q = N_K, where this
    is the usual j <= i.  For N_Q != N_K the bottom-right alignment is the
    reading taken (a query row is the last N_Q positions of the key sequence).
    """
    rows = np.asarray(rows, dtype=np.int64)
    if not causal:
        return np.ones((rows.size, nk), dtype=bool)
    j = np.arange(nk, dtype=np.int64)[None, :]
    return j <= (rows[:, None] + (nk - nq))


def row_softmax(S: np.ndarray, M: np.ndarray):
    """P = softmax over the kept keys of each row, and LSE = log sum exp (kept keys)."""
    Sm = np.where(M, S, -np.inf)
    m = Sm.max(axis=1, keepdims=True)
    E = np.where(M, np.exp(Sm - m), 0.0)
    l = E.sum(axis=1, keepdims=True)
    P = E / l
    lse = m[:, 0] + np.log(l[:, 0])
    return P, lse


def kl_from_probs(P1: np.ndarray, P2: np.ndarray) -> np.ndarray:
    """KL_i = sum_j P1_ij (log P1_ij - log P2_ij), terms with P1_ij = 0 count 0."""
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.where(P1 > 0, P1 * (np.log(P1) - np.log(P2)), 0.0)
    return t.sum(axis=1)


def _block_rows(nq: int, block: int):
    for r0 in range(0, nq, block):
        yield np.arange(r0, min(nq, r0 + block), dtype=np.int64)


def _key_limit(rows: np.ndarray, nq: int, nk: int, causal: bool) -> int:
    """Keys past the last row's causal frontier have P = 0 exactly; leave them out."""
    if not causal:
        return nk
    return int(min(nk, rows.max() + (nk - nq) + 1))


def _rows_state(q1, k1, q2, k2, scale, causal, rows):
    """P1, P2, KL, LSE1, LSE2 for the given query rows of one head."""
    nq, nk = q1.shape[0], k1.shape[0]
    kmax = _key_limit(rows, nq, nk, causal)
    M = causal_mask(rows, nq, nk, causal)[:, :kmax]
    S1 = logits(q1[rows], k1[:kmax], scale)
    S2 = logits(q2[rows], k2[:kmax], scale)
    P1, lse1 = row_softmax(S1, M)
    P2, lse2 = row_softmax(S2, M)
    kl = kl_from_probs(P1, P2)
    return P1, P2, kl, lse1, lse2, kmax


def head_forward(q1, k1, q2, k2, scale: float, causal: bool, block: int = ROW_BLOCK):
    """KL, LSE1, LSE2 [N_Q] of one head (q_t: [N_Q, D], k_t: [N_K, D])."""
    nq = q1.shape[0]
    kl = np.empty(nq)
    lse1 = np.empty(nq)
    lse2 = np.empty(nq)
    for rows in _block_rows(nq, block):
        _, _, kl[rows], lse1[rows], lse2[rows], _ = _rows_state(q1, k1, q2, k2, scale, causal, rows)
    return kl, lse1, lse2


def dlogits(setting: int, P1: np.ndarray, P2: np.ndarray, kl: np.ndarray, g: np.ndarray) -> np.ndarray:
    """dL/dS for the optimised side: setting 1 -> dS2, setting 2 -> dS1."""
    g = np.asarray(g, np.float64)[:, None]
    if setting == 1:
        return g * (P2 - P1)
    if setting == 2:
        with np.errstate(divide="ignore", invalid="ignore"):
            logratio = np.where(P1 > 0, np.log(P1) - np.log(P2), 0.0)
        return g * P1 * (logratio - np.asarray(kl, np.float64)[:, None])
    raise ValueError("setting must be 1 or 2")


def head_backward_rows(setting: int, q1, k1, q2, k2, scale: float, causal: bool, g, rows):
    """dQ_t of the given query rows and their contribution to dK_t (one head).

    dK_t = scale sum_i dS_i^T q_i is a sum over query rows, so the full dK_t is
    the sum of these contributions over any partition of the rows.
    """
    rows = np.asarray(rows, dtype=np.int64)
    q_opt, k_opt = (q2, k2) if setting == 1 else (q1, k1)
    dk = np.zeros((k1.shape[0], q1.shape[1]))
    P1, P2, kl, _, _, kmax = _rows_state(q1, k1, q2, k2, scale, causal, rows)
    dS = dlogits(setting, P1, P2, kl, np.asarray(g, np.float64)[rows])
    dq = scale * (dS @ np.asarray(k_opt[:kmax], np.float64))
    dk[:kmax] = scale * (dS.T @ np.asarray(q_opt[rows], np.float64))
    return dq, dk


def head_backward(setting: int, q1, k1, q2, k2, scale: float, causal: bool, g,
                  block: int = ROW_BLOCK):
    """(dQ_t, dK_t) of one head for the optimised pair t (2 in setting 1, 1 in setting 2)."""
    nq, nk, d = q1.shape[0], k1.shape[0], q1.shape[1]
    dq = np.zeros((nq, d))
    dk = np.zeros((nk, d))
    for rows in _block_rows(nq, block):
        dq_r, dk_r = head_backward_rows(setting, q1, k1, q2, k2, scale, causal, g, rows)
        dq[rows] = dq_r
        dk += dk_r
    return dq, dk


def forward(Q1, K1, Q2, K2, scale: float, causal: bool, block: int = ROW_BLOCK):
    """KL, LSE1, LSE2 [B, H, N_Q] for inputs [B, H, N, D]."""
    B, H, nq, _ = Q1.shape
    out = [np.empty((B, H, nq)) for _ in range(3)]
    for b in range(B):
        for h in range(H):
            r = head_forward(Q1[b, h], K1[b, h], Q2[b, h], K2[b, h], scale, causal, block)
            for o, v in zip(out, r):
                o[b, h] = v
    return tuple(out)


def backward(setting: int, Q1, K1, Q2, K2, scale: float, causal: bool, g, block: int = ROW_BLOCK):
    """(dQ_t, dK_t) [B, H, N, D] of the optimised pair for inputs [B, H, N, D]."""
    B, H, nq, d = Q1.shape
    nk = K1.shape[2]
    dq = np.empty((B, H, nq, d))
    dk = np.empty((B, H, nk, d))
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h] = head_backward(setting, Q1[b, h], K1[b, h], Q2[b, h], K2[b, h],
                                               scale, causal, g[b, h], block)
    return dq, dk


def rows_forward(q1, k1, q2, k2, scale: float, causal: bool, rows, block: int = ROW_BLOCK):
    """KL, LSE1, LSE2 of selected query rows (any order) of one head; O(N_K D) per row."""
    rows = np.asarray(rows, dtype=np.int64)
    out = [np.empty(rows.size) for _ in range(3)]
    for b0 in range(0, rows.size, block):
        sel = rows[b0:b0 + block]
        _, _, kl, l1, l2, _ = _rows_state(q1, k1, q2, k2, scale, causal, sel)
        out[0][b0:b0 + sel.size], out[1][b0:b0 + sel.size], out[2][b0:b0 + sel.size] = kl, l1, l2
    return tuple(out)


def rows_backward_dq(setting: int, q1, k1, q2, k2, scale: float, causal: bool, g_rows, rows,
                     block: int = ROW_BLOCK):
    """dQ rows [len(rows), D] of the optimised pair for selected query rows of one head.

    A query row's gradient depends only on its own row of S1 and S2, so it is
    exact to evaluate rows apart from the rest.
    """
    rows = np.asarray(rows, dtype=np.int64)
    g_rows = np.asarray(g_rows, np.float64)
    k_opt = k2 if setting == 1 else k1
    out = np.empty((rows.size, q1.shape[1]))
    for b0 in range(0, rows.size, block):
        sel = rows[b0:b0 + block]
        P1, P2, kl, _, _, kmax = _rows_state(q1, k1, q2, k2, scale, causal, sel)
        dS = dlogits(setting, P1, P2, kl, g_rows[b0:b0 + sel.size])
        out[b0:b0 + sel.size] = scale * (dS @ np.asarray(k_opt[:kmax], np.float64))
    return out


def materialised_distribution_bytes(n_q: int, n_k: int, heads: int, bytes_per_elem: int,
                                    n_distributions: int = 2) -> int:
    """HBM bytes that materialising P1 and P2 in full takes (the replaced method)."""
    return n_distributions * heads * n_q * n_k * bytes_per_elem
