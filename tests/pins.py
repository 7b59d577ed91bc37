"""Checks that pin the fp64 oracle to facts outside itself.

Each ``check_*`` returns a list of failure strings (empty = pinned).  They call
the oracle through its module object at call time, so a test can plant a
mistake in the oracle (monkeypatch) and confirm that some check catches it.
"""
from __future__ import annotations

import math

import numpy as np

from oracle import oracle as O


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _bad(err, tol) -> bool:
    """True unless err <= tol (a NaN error counts as a failure)."""
    return not (np.max(np.abs(np.asarray(err, np.float64))) <= tol)


def _loss(q1, k1, q2, k2, scale, causal, g):
    kl, _, _ = O.head_forward(q1, k1, q2, k2, scale, causal, block=3)
    return float(np.dot(g, kl))


def check_finite_differences(seed=0, cases=((5, 7, False), (5, 7, True), (6, 6, True), (1, 4, False)),
                             d=4, scale=0.7, h=1e-6, tol=1e-6):
    """Central finite differences of L = sum_i g_i KL_i, both settings (brute force)."""
    fails = []
    rng = np.random.default_rng(seed)
    for nq, nk, causal in cases:
        q1, k1, q2, k2 = _rand(rng, nq, d), _rand(rng, nk, d), _rand(rng, nq, d), _rand(rng, nk, d)
        g = rng.uniform(0.5, 1.5, nq)
        for setting in (1, 2):
            dq, dk = O.head_backward(setting, q1, k1, q2, k2, scale, causal, g, block=2)
            t = 2 if setting == 1 else 1
            args = {"q1": q1, "k1": k1, "q2": q2, "k2": k2}
            num = {}
            for name in (f"q{t}", f"k{t}"):
                base = args[name]
                grad = np.zeros_like(base)
                for idx in np.ndindex(base.shape):
                    a = dict(args)
                    p = base.copy(); p[idx] += h; a[name] = p
                    lp = _loss(a["q1"], a["k1"], a["q2"], a["k2"], scale, causal, g)
                    p = base.copy(); p[idx] -= h; a[name] = p
                    lm = _loss(a["q1"], a["k1"], a["q2"], a["k2"], scale, causal, g)
                    grad[idx] = (lp - lm) / (2 * h)
                num[name] = grad
            for name, got in ((f"q{t}", dq), (f"k{t}", dk)):
                ref = num[name]
                err = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
                if not err < tol:
                    fails.append(f"fd setting {setting} d{name} nq={nq} nk={nk} causal={causal}: rel err {err:.3e}")
    return fails


def check_torch_library(seed=1, cases=((40, 40, False), (40, 40, True), (24, 56, True), (33, 17, False)),
                        d=16, scale=0.3, tol=1e-10):
    """torch CPU float64 log_softmax / kl_div / autograd on small shapes (library routine)."""
    import torch
    fails = []
    rng = np.random.default_rng(seed)
    for nq, nk, causal in cases:
        arr = [_rand(rng, nq, d), _rand(rng, nk, d), _rand(rng, nq, d), _rand(rng, nk, d)]
        g = rng.uniform(0.1, 2.0, nq)
        kl, l1, l2 = O.head_forward(*arr, scale, causal, block=7)
        for setting in (1, 2):
            t = [torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in arr]
            tq1, tk1, tq2, tk2 = t
            S1 = scale * tq1 @ tk1.T
            S2 = scale * tq2 @ tk2.T
            total = 0
            kls, lses1, lses2 = [], [], []
            for i in range(nq):
                n = min(nk, i + nk - nq + 1) if causal else nk
                lp1 = torch.log_softmax(S1[i, :n], dim=0)
                lp2 = torch.log_softmax(S2[i, :n], dim=0)
                # kl_div(input, target, log_target) = sum exp(target) (target - input)
                kli = torch.nn.functional.kl_div(lp2, lp1, reduction="sum", log_target=True)
                kls.append(kli.item())
                lses1.append(torch.logsumexp(S1[i, :n], 0).item())
                lses2.append(torch.logsumexp(S2[i, :n], 0).item())
                total = total + float(g[i]) * kli
            total.backward()
            for name, got, ref in (("KL", kl, kls), ("LSE1", l1, lses1), ("LSE2", l2, lses2)):
                e = np.max(np.abs(np.asarray(got) - np.asarray(ref)))
                if not e < tol:
                    fails.append(f"torch {name} nq={nq} nk={nk} causal={causal}: max err {e:.3e}")
            dq, dk = O.head_backward(setting, *arr, scale, causal, g, block=5)
            tq, tk = (tq2, tk2) if setting == 1 else (tq1, tk1)
            for name, got, ref in (("dQ", dq, tq.grad.numpy()), ("dK", dk, tk.grad.numpy())):
                e = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
                if not e < tol:
                    fails.append(f"torch setting {setting} {name} nq={nq} nk={nk} causal={causal}: rel {e:.3e}")
    return fails


def check_closed_forms(seed=2, d=8, scale=0.5):
    """Closed forms: identical pairs, uniform keys, zero student queries, one-key row, two keys."""
    from scipy.special import softmax as sp_softmax
    from scipy.stats import entropy as sp_entropy
    fails = []
    rng = np.random.default_rng(seed)
    for nq, nk, causal in ((9, 9, True), (9, 13, False), (6, 11, True)):
        q1, k1 = _rand(rng, nq, d), _rand(rng, nk, d)
        g = rng.uniform(0.5, 1.5, nq)
        n_i = np.array([min(nk, i + nk - nq + 1) if causal else nk for i in range(nq)])
        # (i) identical pairs: KL = 0 and both gradients vanish, exactly
        kl, l1, l2 = O.head_forward(q1, k1, q1, k1, scale, causal)
        if not (np.all(kl == 0) and np.all(l1 == l2)):
            fails.append(f"identical pairs: KL {np.max(np.abs(kl)):.3e}")
        for setting in (1, 2):
            dq, dk = O.head_backward(setting, q1, k1, q1, k1, scale, causal, g)
            if not (np.all(dq == 0) and np.all(dk == 0)):
                fails.append(f"identical pairs setting {setting}: nonzero grads")
        # (ii) K_t = 0: uniform rows, LSE_t = log n_i
        kl, l1, l2 = O.head_forward(q1, np.zeros((nk, d)), q1, np.zeros((nk, d)), scale, causal)
        if _bad(l1 - np.log(n_i), 1e-13) or _bad(l2 - np.log(n_i), 1e-13):
            fails.append("zero keys: LSE != log n")
        # (iii) Q2 = 0: P2 uniform, KL_i = log n_i - H(P1_i)
        kl, l1, l2 = O.head_forward(q1, k1, np.zeros((nq, d)), k1, scale, causal)
        S1 = scale * q1 @ k1.T
        ref = np.array([math.log(n_i[i]) - sp_entropy(sp_softmax(S1[i, :n_i[i]])) for i in range(nq)])
        if _bad(kl - ref, 1e-12):
            fails.append(f"zero student queries: KL err {np.max(np.abs(kl - ref)):.3e}")
        if _bad(l2 - np.log(n_i), 1e-13):
            fails.append("zero student queries: LSE2 != log n")
    # (iv) causal first row (N_Q = N_K) sees one key: KL_0 = 0, LSE_t,0 = S_t,00
    q1, k1, q2, k2 = (_rand(rng, 5, d) for _ in range(4))
    kl, l1, l2 = O.head_forward(q1, k1, q2, k2, scale, True)
    if _bad(kl[0], 1e-15) or _bad(l1[0] - scale * q1[0] @ k1[0], 1e-13) or _bad(l2[0] - scale * q2[0] @ k2[0], 1e-13):
        fails.append("single-key causal row")
    # (v) two keys: Bernoulli KL
    q1, k1, q2, k2 = _rand(rng, 7, d), _rand(rng, 2, d), _rand(rng, 7, d), _rand(rng, 2, d)
    kl, _, _ = O.head_forward(q1, k1, q2, k2, scale, False)
    for i in range(7):
        a = scale * (q1[i] @ k1[0] - q1[i] @ k1[1])
        b = scale * (q2[i] @ k2[0] - q2[i] @ k2[1])
        p, q = 1 / (1 + math.exp(-a)), 1 / (1 + math.exp(-b))
        ref = p * math.log(p / q) + (1 - p) * math.log((1 - p) / (1 - q))
        if _bad(kl[i] - ref, 1e-13):
            fails.append(f"bernoulli row {i}: {kl[i]} vs {ref}")
    return fails


def check_invariants(seed=3, d=8, scale=0.6):
    """KL >= 0, logit-shift invariance, dS row sums (sum_j dK_j = 0), trace identity."""
    fails = []
    rng = np.random.default_rng(seed)
    for nq, nk, causal in ((12, 12, True), (10, 15, False), (7, 19, True)):
        q1, k1, q2, k2 = _rand(rng, nq, d), _rand(rng, nk, d), _rand(rng, nq, d), _rand(rng, nk, d)
        g = rng.uniform(0.5, 1.5, nq)
        kl, l1, l2 = O.head_forward(q1, k1, q2, k2, scale, causal)
        if not np.all(kl >= -1e-14):
            fails.append("KL < 0")
        c1, c2 = _rand(rng, d), _rand(rng, d)
        kls, l1s, l2s = O.head_forward(q1, k1 + c1, q2, k2 + c2, scale, causal)
        if _bad(kls - kl, 1e-12):
            fails.append("KL changed under a per-row logit shift")
        if _bad(l1s - (l1 + scale * q1 @ c1), 1e-12) or _bad(l2s - (l2 + scale * q2 @ c2), 1e-12):
            fails.append("LSE did not shift with the logits")
        for setting in (1, 2):
            dq, dk = O.head_backward(setting, q1, k1, q2, k2, scale, causal, g)
            qo, ko = (q2, k2) if setting == 1 else (q1, k1)
            if _bad(dk.sum(axis=0), 1e-12):
                fails.append(f"setting {setting}: sum_j dK_j != 0")
            lhs, rhs = float(np.sum(dq * qo)), float(np.sum(dk * ko))
            if _bad(lhs - rhs, 1e-12 * max(1.0, abs(lhs))):
                fails.append(f"setting {setting}: trace identity {lhs} vs {rhs}")
    return fails


def check_online_identity(seed=4, d=8, scale=0.8):
    """The pages' reformulation KL = acc/l1 + LSE2 - LSE1 with acc/l1 = E_P1[S1 - S2]."""
    from scipy.special import logsumexp as sp_lse, softmax as sp_softmax
    fails = []
    rng = np.random.default_rng(seed)
    for nq, nk, causal in ((11, 11, True), (8, 21, False)):
        q1, k1, q2, k2 = _rand(rng, nq, d), _rand(rng, nk, d), _rand(rng, nq, d), _rand(rng, nk, d)
        kl, l1, l2 = O.head_forward(q1, k1, q2, k2, scale, causal)
        S1, S2 = scale * q1 @ k1.T, scale * q2 @ k2.T
        for i in range(nq):
            n = min(nk, i + nk - nq + 1) if causal else nk
            w = sp_softmax(S1[i, :n])
            ref = float(w @ (S1[i, :n] - S2[i, :n])) + sp_lse(S2[i, :n]) - sp_lse(S1[i, :n])
            if _bad(kl[i] - ref, 1e-12):
                fails.append(f"online identity row {i}: {kl[i]} vs {ref}")
    return fails


ALL_CHECKS = (check_finite_differences, check_torch_library, check_closed_forms, check_invariants,
              check_online_identity)


def check_batched_wrappers(seed=5, B=2, H=3, d=8, scale=0.45, tol=1e-10):
    """The [B, H] entry points forward / backward against torch CPU float64 on the whole batch at once.

    torch's log_softmax, kl_div and autograd run over [B, H, N_Q, N_K] logits,
    so a head or batch index taken from the wrong place in the oracle's loops
    (inputs, g, or where a result is stored) shows up as a mismatch.  Masked
    logits are set to -1e4, whose exp underflows to exactly 0 in float64, so
    masked keys carry no weight and no NaN enters the gradient.
    """
    import torch
    fails = []
    rng = np.random.default_rng(seed)
    for nq, nk, causal in ((6, 6, True), (5, 9, False), (4, 10, True)):
        arr = [_rand(rng, B, H, nq, d), _rand(rng, B, H, nk, d), _rand(rng, B, H, nq, d), _rand(rng, B, H, nk, d)]
        g = rng.uniform(0.2, 2.0, (B, H, nq)) * (1.0 + np.arange(B * H).reshape(B, H, 1))
        kl, l1, l2 = O.forward(*arr, scale, causal, block=4)
        keep = torch.ones(nq, nk, dtype=torch.bool)
        if causal:
            keep = torch.arange(nk)[None, :] <= torch.arange(nq)[:, None] + (nk - nq)
        for setting in (1, 2):
            t = [torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in arr]
            S1 = (scale * t[0] @ t[1].transpose(-1, -2)).masked_fill(~keep, -1e4)
            S2 = (scale * t[2] @ t[3].transpose(-1, -2)).masked_fill(~keep, -1e4)
            lp1, lp2 = torch.log_softmax(S1, dim=-1), torch.log_softmax(S2, dim=-1)
            rows_kl = torch.nn.functional.kl_div(lp2, lp1, reduction="none", log_target=True).sum(dim=-1)
            (torch.tensor(g) * rows_kl).sum().backward()
            for name, got, ref in (("KL", kl, rows_kl), ("LSE1", l1, torch.logsumexp(S1, -1)),
                                   ("LSE2", l2, torch.logsumexp(S2, -1))):
                e = np.max(np.abs(np.asarray(got) - ref.detach().numpy()))
                if not e < tol:
                    fails.append(f"batched {name} nq={nq} nk={nk} causal={causal}: max err {e:.3e}")
            dq, dk = O.backward(setting, *arr, scale, causal, g, block=3)
            tq, tk = (t[2], t[3]) if setting == 1 else (t[0], t[1])
            for name, got, ref in (("dQ", dq, tq.grad.numpy()), ("dK", dk, tk.grad.numpy())):
                e = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
                if not e < tol:
                    fails.append(f"batched setting {setting} {name} nq={nq} nk={nk} causal={causal}: rel {e:.3e}")
    return fails


ALL_CHECKS = ALL_CHECKS + (check_batched_wrappers,)
