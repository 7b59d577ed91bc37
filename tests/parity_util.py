"""Helpers for the GPU parity tests: inputs to the device, oracle on chosen
heads or rows, and the tolerances every comparison uses.

Tolerances (per query row, against the fp64 oracle on the same bf16 inputs):
    |dKL|  <= 1e-3 + 5e-3 |KL|
    |dLSE| <= 1e-3
    gradients: ||G - G*||_F / ||G*||_F <= 1e-2 over the checked rows
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

from attention_kl_divergence_streamkl_gb300 import synth
from oracle import oracle as O

KL_ABS, KL_REL, LSE_ABS, GRAD_REL = 1e-3, 5e-3, 1e-3, 1e-2


def to_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev_inputs(inp):
    return [to_dev(inp[k]) for k in ("q1", "k1", "q2", "k2")]


def f64(bits):
    return synth.bf16_bits_to_f64(bits)


def head_f64(inp, b, h):
    return [f64(inp[k][b, h]) for k in ("q1", "k1", "q2", "k2")]


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_rows(kl, l1, l2, rkl, rl1, rl2, what=""):
    kl, l1, l2 = (np.asarray(x, np.float64) for x in (kl, l1, l2))
    bad = np.abs(kl - rkl) > KL_ABS + KL_REL * np.abs(rkl)
    assert not (bad.any() or np.isnan(kl).any()), \
        f"{what} KL: {int(bad.sum())} rows out of tolerance, max err {np.nanmax(np.abs(kl - rkl)):.3e}"
    e1, e2 = np.abs(l1 - rl1), np.abs(l2 - rl2)
    assert np.all(e1 <= LSE_ABS) and np.all(e2 <= LSE_ABS), \
        f"{what} LSE max err {np.nanmax(e1):.3e} / {np.nanmax(e2):.3e}"


def rel_fro(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


# Where the exact gradient vanishes (a row with one visible key has P1 = P2 = 1),
# a relative error is undefined; there the error is measured against an RMS
# floor of 1e-4 per element instead.
GRAD_FLOOR_RMS = 1e-4


def assert_grad(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    denom = max(np.linalg.norm(ref), GRAD_FLOOR_RMS * np.sqrt(max(ref.size, 1)))
    e = float(np.linalg.norm(got - ref) / denom)
    assert e <= GRAD_REL, f"{what}: relative Frobenius error {e:.3e}"


def oracle_head(inp, w, b, h, setting=None, g=None):
    """fwd (and bwd if setting) of one head with the full oracle."""
    q1, k1, q2, k2 = head_f64(inp, b, h)
    fw = O.head_forward(q1, k1, q2, k2, w.softmax_scale, w.causal)
    if setting is None:
        return fw, None
    gg = inp["g"][b, h] if g is None else g
    return fw, O.head_backward(setting, q1, k1, q2, k2, w.softmax_scale, w.causal, gg)


def oracle_head_dk_parallel(inp, w, b, h, setting, threads=8, chunk=1024):
    """dK of one head, the oracle's row blocks spread over threads (sums of fp64 partials)."""
    q1, k1, q2, k2 = head_f64(inp, b, h)
    g = np.asarray(inp["g"][b, h], np.float64)
    nq = q1.shape[0]

    def part(r0):
        rows = np.arange(r0, min(nq, r0 + chunk))
        return O.head_backward_rows(setting, q1, k1, q2, k2, w.softmax_scale, w.causal, g, rows)

    with ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(part, range(0, nq, chunk)))
    dk = np.zeros_like(k1)
    for _, dkp in parts:
        dk += dkp
    return dk


def oracle_rows(inp, w, rows, setting=None):
    """KL, LSE1, LSE2 (and dQ rows of the optimised pair) for sampled (b, h, i) rows."""
    n = len(rows)
    kl, l1, l2 = np.empty(n), np.empty(n), np.empty(n)
    dq = np.empty((n, w.D)) if setting else None
    heads = {}
    for idx, (b, h, i) in enumerate(rows):
        heads.setdefault((int(b), int(h)), []).append((idx, int(i)))
    for (b, h), items in heads.items():
        q1, k1, q2, k2 = head_f64(inp, b, h)
        idxs = np.array([x[0] for x in items])
        rr = np.array([x[1] for x in items])
        a, c, d = O.rows_forward(q1, k1, q2, k2, w.softmax_scale, w.causal, rr)
        kl[idxs], l1[idxs], l2[idxs] = a, c, d
        if setting:
            g = np.asarray(inp["g"][b, h], np.float64)[rr]
            dq[idxs] = O.rows_backward_dq(setting, q1, k1, q2, k2, w.softmax_scale, w.causal, g, rr)
    return kl, l1, l2, dq


def dk_invariants(dk, k_opt, dq, q_opt):
    """sum_j dK_j = 0 per (b, h, d) and sum_i <dQ_i, Q_i> = sum_j <dK_j, K_j> per (b, h).

    Both sides are sums with heavy cancellation, so each residual is measured
    against the magnitude of its terms (sum of |dK_j| per column, and the sum of
    |<dQ_i, Q_i>| + |<dK_j, K_j>|), which is what bf16 output rounding scales with.
    """
    dk = dk.double()
    col = dk.sum(dim=2)  # [B, H, D]
    scale_ = dk.abs().sum(dim=2).clamp_min(1e-30)
    r_sum = float((col.abs() / scale_).max())
    tq = (dq.double() * q_opt.double()).sum(dim=3)  # [B, H, N_Q]
    tk = (dk * k_opt.double()).sum(dim=3)  # [B, H, N_K]
    lhs, rhs = tq.sum(dim=2), tk.sum(dim=2)
    mag = (tq.abs().sum(dim=2) + tk.abs().sum(dim=2)).clamp_min(1e-30)
    r_tr = float(((lhs - rhs).abs() / mag).max())
    return r_sum, r_tr
