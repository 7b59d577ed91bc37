"""Helpers for the GPU parity tests: inputs to the device, oracle on chosen
heads or rows, and the tolerances every comparison uses.

Tolerances (per query row, against the fp64 oracle on the same bf16 inputs):
    |dKL|  <= 1e-3 + 5e-3 |KL|
    |dLSE| <= 1e-3
    gradients: ||G - G*||_F / ||G*||_F <= 1e-2 over the checked rows
"""
from __future__ import annotations

import math
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


# A row whose exact gradient is zero (a causal row that sees one key has
# P1 = P2 = 1; a row with g_i = 0) has no relative error.  Such rows are held to
# an absolute bound instead: ZERO_ROW_REL times the largest row norm of the
# reference (a real gradient row is of that order, g * scale * |K|), or the
# caller's bound when the whole reference is zero.  Every other row is inside
# the relative Frobenius error, which has no floor.
ZERO_ROW_REL = 1e-3


def grad_error(got, ref):
    """Relative Frobenius error ||got - ref|| / ||ref|| (inf when ref is zero)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rn = float(np.linalg.norm(ref))
    if rn == 0.0:
        return math.inf
    return float(np.linalg.norm(got - ref)) / rn


def assert_grad(got, ref, what="", zero_tol=None):
    """Gradient parity: relative Frobenius error <= GRAD_REL, exact-zero rows within a bound.

    zero_tol: absolute bound on the norm of a row whose reference is exactly
    zero; required when the whole reference is zero, else ZERO_ROW_REL x the
    largest reference row norm.
    """
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    if ref.size == 0:
        return
    rows_r = ref.reshape(-1, ref.shape[-1])
    rows_g = got.reshape(-1, got.shape[-1])
    row_norm = np.linalg.norm(rows_r, axis=1)
    zero = row_norm == 0.0
    if not zero.all():
        e = grad_error(got, ref)
        assert e <= GRAD_REL, f"{what}: relative Frobenius error {e:.3e}"
        if zero_tol is None:
            zero_tol = ZERO_ROW_REL * float(row_norm.max())
    assert zero_tol is not None, f"{what}: the reference is zero; give an absolute bound"
    if zero.any():
        worst = float(np.linalg.norm(rows_g[zero], axis=1).max())
        assert worst <= zero_tol, f"{what}: a row whose exact gradient is 0 has norm {worst:.3e} > {zero_tol:.3e}"


def zero_grad_tol(g, scale, other):
    """Absolute row bound for a gradient that is exactly zero: 1e-4 |g| scale max_j |other_j|.

    A dQ row is scale * sum_j dS_ij k_j with |dS_ij| <= 2|g_i|, so 1e-4 of that
    size is far above fp32 rounding of P1 - P2 = 0 and far below any real row.
    """
    g = np.abs(np.asarray(g, np.float64))
    other = np.asarray(other, np.float64)
    return 1e-4 * float(g.max(initial=0.0)) * scale * float(np.linalg.norm(other, axis=-1).max(initial=0.0))


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


TRACE_TOL = 1e-2


def dk_invariants(dk, k_opt, dq, q_opt):
    """Two identities every exact gradient pair obeys, measured on whole heads.

    * sum_j dK_j = 0 per (b, h, d), because every dS row sums to zero in both
      settings.  Residual |sum_j dK_jd| / sum_j |dK_jd|; a column that is all
      zero scores inf, so a zero dK fails.
    * the trace identity sum_i <dQ_i, Q_i> = sum_j <dK_j, K_j> per (b, h)
      (both sides equal sum_ij dS_ij S_ij, for any dS, so the kernels' own bf16
      dS obeys it too).  Its residual is divided by the error the arithmetic
      allows: TRACE_TOL x the root-sum-square of the element products dQ*Q and
      dK*K (bf16 rounding of the outputs moves each side by about 2^-9/sqrt(3)
      of that), plus delta x the sum of their magnitudes, delta = 2^-23 per
      128-wide step of the longer fp32 accumulation (one ulp per step: the
      accumulator's rounding need not be unbiased, so this part adds up
      linearly).  A residual below 1 passes.

    Returns (r_sum, r_tr, power): the worst residuals over heads, and the
    smallest |sum_i <dQ_i, Q_i>| / allowed error over heads -- what a dK of
    zero would score on the trace identity.  In setting 1 the sum has no
    cancellation (power in the thousands), so the identity pins dK's scale on
    every head; in setting 2 it cancels (power can drop below 1) and the
    identity only bounds dK's errors.
    """
    dk = dk.double()
    col = dk.sum(dim=2)  # [B, H, D]
    mag = dk.abs().sum(dim=2)
    r_col = torch.where(mag > 0, col.abs() / mag.clamp_min(1e-300), torch.full_like(mag, math.inf))
    r_sum = float(r_col.max())
    tq = dq.double() * q_opt.double()  # [B, H, N_Q, D]
    tk = dk * k_opt.double()
    lhs, rhs = tq.sum(dim=(2, 3)), tk.sum(dim=(2, 3))
    rss = ((tq * tq).sum(dim=(2, 3)) + (tk * tk).sum(dim=(2, 3))).sqrt()
    steps = max(-(-dq.shape[2] // 128), -(-dk.shape[2] // 128))
    delta = steps * 2.0 ** -23
    allowed = TRACE_TOL * rss + delta * (tq.abs().sum(dim=(2, 3)) + tk.abs().sum(dim=(2, 3)))
    ok = allowed > 0
    r_tr = float(torch.where(ok, (lhs - rhs).abs() / allowed.clamp_min(1e-300), torch.full_like(rss, math.inf)).max())
    power = float(torch.where(ok, lhs.abs() / allowed.clamp_min(1e-300), torch.zeros_like(rss)).min())
    return r_sum, r_tr, power


def assert_dk_invariants(dk, k_opt, dq, q_opt, setting, what=""):
    r_sum, r_tr, power = dk_invariants(dk, k_opt, dq, q_opt)
    print(f"{what}: dK identities r_sum {r_sum:.3e} r_tr {r_tr:.3e} power {power:.3e}")
    assert r_sum < TRACE_TOL, f"{what}: sum_j dK_j residual {r_sum:.3e}"
    assert r_tr < 1.0, f"{what}: trace identity residual {r_tr:.3e} of the allowed error"
    if setting == 1:
        assert power > 10.0, f"{what}: trace identity cannot see dK's scale (power {power:.3e})"
    return r_sum, r_tr, power


def map_heads(fn, heads, threads=8):
    """fn(b, h) over heads, in threads (numpy releases the GIL in its kernels)."""
    with ThreadPoolExecutor(threads) as ex:
        return list(ex.map(lambda bh: fn(*bh), heads))


def oracle_forward_heads(inp, w, heads, threads=8):
    """KL, LSE1, LSE2 [len(heads), N_Q] of the given heads with the full oracle."""
    def one(b, h):
        q1, k1, q2, k2 = head_f64(inp, b, h)
        return O.head_forward(q1, k1, q2, k2, w.softmax_scale, w.causal)
    outs = map_heads(one, heads, threads)
    return tuple(np.stack([o[t] for o in outs]) for t in range(3))


def oracle_last_keys_dk(inp, w, b, h, setting, keys, chunk=32):
    """dK rows of the last `keys` keys of one head (causal, N_Q = N_K).

    Under the causal mask key j is seen only by the rows i >= j, so the dK of
    the last R keys is the sum over the last R query rows alone: an exact slice
    of the full gradient at O(R N_K D) cost.
    """
    assert w.causal and w.NQ == w.NK and keys <= w.NK
    q1, k1, q2, k2 = head_f64(inp, b, h)
    g = np.asarray(inp["g"][b, h], np.float64)
    dk = np.zeros((keys, w.D))
    for r0 in range(w.NQ - keys, w.NQ, chunk):
        rows = np.arange(r0, min(w.NQ, r0 + chunk))
        _, dkp = O.head_backward_rows(setting, q1, k1, q2, k2, w.softmax_scale, w.causal, g, rows)
        dk += dkp[w.NK - keys:]
    return dk
