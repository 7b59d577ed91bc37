"""Pins of the fp64 oracle against facts outside itself (CPU only)."""
import json
import math
import os

import numpy as np
import pytest

from oracle import oracle as O
from tests import pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    fails = check()
    assert not fails, "\n".join(fails)


def test_pages_materialisation_figure():
    with open(os.path.join(GOLDEN, "pages_figures.json")) as f:
        fig = json.load(f)
    b = O.materialised_distribution_bytes(fig["context"], fig["context"], fig["heads"],
                                          fig["bytes_per_elem"], fig["distributions"])
    assert b == 2 * 32 * 65536 * 65536 * 2
    # "about 512 GB": exactly 512 GiB
    assert abs(b / 2**30 - fig["stated_about_gb"]) < 1e-9
    assert b > fig["stated_exceeds_gb"] * 1e9


# --------------------------------------------------------------------------
# the pages' online recurrence (five running scalars) and the Split-K merge,
# emulated in fp64, reach the oracle's definition exactly up to rounding
# --------------------------------------------------------------------------

def _online(S1, S2, keep, tile, lazy=0.0):
    """Five-scalar online update of one row over key tiles (derived update rules).

    lazy > 0 keeps the reference max until a tile exceeds it by more than
    ``lazy`` (the rescale is skipped, exact because l1 and acc share m1).
    """
    m1 = m2 = -math.inf
    l1 = l2 = acc = 0.0
    for t0 in range(0, S1.size, tile):
        s1, s2, k = S1[t0:t0 + tile], S2[t0:t0 + tile], keep[t0:t0 + tile]
        if not k.any():
            continue
        s1, s2 = s1[k], s2[k]
        n1, n2 = max(m1, s1.max()), max(m2, s2.max())
        if lazy > 0 and m1 > -math.inf and n1 <= m1 + lazy:
            n1 = m1
        if lazy > 0 and m2 > -math.inf and n2 <= m2 + lazy:
            n2 = m2
        a1 = 0.0 if m1 == -math.inf else math.exp(m1 - n1)
        a2 = 0.0 if m2 == -math.inf else math.exp(m2 - n2)
        e1 = np.exp(s1 - n1)
        l1 = a1 * l1 + e1.sum()
        acc = a1 * acc + float(e1 @ (s1 - s2))
        l2 = a2 * l2 + np.exp(s2 - n2).sum()
        m1, m2 = n1, n2
    return m1, m2, l1, l2, acc


def _finish(m1, m2, l1, l2, acc):
    lse1, lse2 = m1 + math.log(l1), m2 + math.log(l2)
    return acc / l1 + lse2 - lse1, lse1, lse2


def _merge(parts):
    parts = [p for p in parts if p[0] > -math.inf]
    M1 = max(p[0] for p in parts)
    M2 = max(p[1] for p in parts)
    l1 = sum(p[2] * math.exp(p[0] - M1) for p in parts)
    acc = sum(p[4] * math.exp(p[0] - M1) for p in parts)
    l2 = sum(p[3] * math.exp(p[1] - M2) for p in parts)
    return M1, M2, l1, l2, acc


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("lazy", [0.0, 8.0])
def test_online_recurrence_and_splitk_merge(causal, lazy):
    rng = np.random.default_rng(11)
    nq, nk, d, scale = 9, 37, 6, 1.3
    q1, k1, q2, k2 = (rng.standard_normal((n, d)) for n in (nq, nk, nq, nk))
    kl, l1, l2 = O.head_forward(q1, k1, q2, k2, scale, causal)
    S1, S2 = scale * q1 @ k1.T, scale * q2 @ k2.T
    M = O.causal_mask(np.arange(nq), nq, nk, causal)
    for i in range(nq):
        got = _finish(*_online(S1[i], S2[i], M[i], tile=8, lazy=lazy))
        assert np.allclose(got, (kl[i], l1[i], l2[i]), rtol=0, atol=1e-12)
        # Split-K: three key ranges, merged
        bounds = [0, 5, 22, nk]
        parts = [_online(S1[i, a:b], S2[i, a:b], M[i, a:b], tile=4, lazy=lazy)
                 for a, b in zip(bounds[:-1], bounds[1:])]
        got = _finish(*_merge(parts))
        assert np.allclose(got, (kl[i], l1[i], l2[i]), rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# planted mistakes: each plausible error in the oracle fails some pin
# --------------------------------------------------------------------------

def _run_all():
    fails = []
    for c in pins.ALL_CHECKS:
        try:
            fails += c()
        except Exception as e:  # a mistake may also break shapes
            fails.append(f"{c.__name__} raised {type(e).__name__}: {e}")
    return fails


def _mut_reverse_kl(mp):
    orig = O.kl_from_probs
    mp.setattr(O, "kl_from_probs", lambda P1, P2: orig(P2, P1))


def _mut_flip_ds2(mp):
    orig = O.dlogits
    mp.setattr(O, "dlogits", lambda s, P1, P2, kl, g: -orig(s, P1, P2, kl, g) if s == 1 else orig(s, P1, P2, kl, g))


def _mut_drop_kl_term(mp):
    orig = O.dlogits
    mp.setattr(O, "dlogits", lambda s, P1, P2, kl, g: orig(s, P1, P2, 0 * np.asarray(kl), g))


def _mut_drop_scale_dq(mp):
    orig = O.head_backward

    def bad(setting, q1, k1, q2, k2, scale, causal, g, block=O.ROW_BLOCK):
        dq, dk = orig(setting, q1, k1, q2, k2, scale, causal, g, block)
        return dq / scale, dk
    mp.setattr(O, "head_backward", bad)


def _mut_mask_off_by_one(mp):
    def bad(rows, nq, nk, causal):
        rows = np.asarray(rows, dtype=np.int64)
        if not causal:
            return np.ones((rows.size, nk), dtype=bool)
        return np.arange(nk)[None, :] < rows[:, None] + (nk - nq)
    mp.setattr(O, "causal_mask", bad)


def _mut_lse_without_max(mp):
    orig = O.row_softmax

    def bad(S, M):
        P, lse = orig(S, M)
        m = np.where(M, S, -np.inf).max(axis=1)
        return P, lse - m
    mp.setattr(O, "row_softmax", bad)


def _mut_g_on_keys(mp):
    orig = O.dlogits
    mp.setattr(O, "dlogits", lambda s, P1, P2, kl, g: orig(s, P1, P2, kl, np.ones_like(g)) * np.asarray(g)[:, None] ** 2)


def _mut_transposed_dk(mp):
    orig = O.head_backward

    def bad(setting, q1, k1, q2, k2, scale, causal, g, block=O.ROW_BLOCK):
        dq, dk = orig(setting, q1, k1, q2, k2, scale, causal, g, block)
        return dq, dk[::-1].copy()
    mp.setattr(O, "head_backward", bad)


def _mut_wrapper_g_of_next_head(mp):
    orig = O.head_backward

    def bad(setting, Q1, K1, Q2, K2, scale, causal, g, block=O.ROW_BLOCK):
        B, H, nq, d = Q1.shape
        dq, dk = np.empty((B, H, nq, d)), np.empty((B, H, K1.shape[2], d))
        for b in range(B):
            for h in range(H):
                dq[b, h], dk[b, h] = orig(setting, Q1[b, h], K1[b, h], Q2[b, h], K2[b, h], scale, causal,
                                          g[b, (h + 1) % H], block)
        return dq, dk
    mp.setattr(O, "backward", bad)


def _mut_wrapper_batch_heads_swapped(mp):
    orig = O.forward

    def bad(Q1, K1, Q2, K2, scale, causal, block=O.ROW_BLOCK):
        return tuple(x[::-1].copy() for x in orig(Q1, K1, Q2, K2, scale, causal, block))
    mp.setattr(O, "forward", bad)


@pytest.mark.parametrize("mutation", [_mut_reverse_kl, _mut_flip_ds2, _mut_drop_kl_term, _mut_drop_scale_dq,
                                      _mut_mask_off_by_one, _mut_lse_without_max, _mut_g_on_keys,
                                      _mut_transposed_dk, _mut_wrapper_g_of_next_head,
                                      _mut_wrapper_batch_heads_swapped], ids=lambda f: f.__name__[5:])
def test_planted_mistake_is_caught(monkeypatch, mutation):
    mutation(monkeypatch)
    assert _run_all(), "a planted mistake passed every pin"


def test_row_subsets_agree_with_full_head():
    """The sampled-row entry points give the full-head values for any row order."""
    rng = np.random.default_rng(5)
    for nq, nk, causal in ((40, 40, True), (23, 61, True), (31, 17, False)):
        q1, k1, q2, k2 = (rng.standard_normal((n, 8)) for n in (nq, nk, nq, nk))
        g = rng.uniform(0.5, 1.5, nq)
        kl, l1, l2 = O.head_forward(q1, k1, q2, k2, 0.4, causal)
        rows = rng.permutation(nq)[: nq // 2]
        a, b, c = O.rows_forward(q1, k1, q2, k2, 0.4, causal, rows, block=5)
        assert np.allclose(a, kl[rows], atol=1e-13) and np.allclose(b, l1[rows]) and np.allclose(c, l2[rows])
        for setting in (1, 2):
            dq, _ = O.head_backward(setting, q1, k1, q2, k2, 0.4, causal, g)
            got = O.rows_backward_dq(setting, q1, k1, q2, k2, 0.4, causal, g[rows], rows, block=4)
            assert np.allclose(got, dq[rows], atol=1e-13)
