"""Seeded synthetic inputs for the attention-KL workloads.

This module holds input generation only: no step of the KL method lives here.
Both the fp64 CPU oracle (through the tests) and the CUDA path (through the
tests, ``bench.py`` and ``smoke()``) take their inputs from it.

Recipe (one reading of the workloads, stated once here):

* every tensor is ``[B, H, N, D]`` bf16, stored as raw bf16 bit patterns
  (``numpy.uint16``) so that both sides see the very same values;
* the teacher pair ``(Q1, K1)`` is standard normal, rounded to bf16 by
  round-to-nearest-even;
* the student pair is ``Q2 = bf16(f32(Q1) + sigma * Z)``, ``K2`` alike, with an
  independent standard-normal ``Z`` and ``sigma`` 0.3 (the 128-row case) or 0.5
  (every other workload);
* each ``(tensor, b, h)`` slice has its own Philox stream seeded by
  ``SeedSequence([seed, tensor_id, b, h])``, so a single head can be rebuilt
  without generating the rest (the sampled-row checks on long contexts rely on
  it) and the result does not depend on the thread count or the machine.

The upstream gradient ``g`` is the constant ``1/N_Q`` per query row (the mean
of the per-row KL values), the plainest reading for every workload.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np

# tensor ids inside the seed sequence
_Q1, _K1, _ZQ, _ZK = 0, 1, 2, 3


@dataclass(frozen=True)
class Workload:
    """One synthetic problem: shapes, mask, noise level and seed."""

    name: str
    B: int
    H: int
    NQ: int
    NK: int
    D: int
    causal: bool
    sigma: float
    seed: int
    scale: float = field(default=0.0)  # 0 means 1/sqrt(D)

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale > 0 else 1.0 / float(np.sqrt(self.D))

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    def unmasked_pairs(self) -> int:
        """Number of (query, key) pairs that carry weight, over all heads."""
        return self.B * self.H * count_pairs(self.NQ, self.NK, self.causal)


def count_pairs(nq: int, nk: int, causal: bool) -> int:
    """Unmasked (i, j) pairs of one head; causal keeps j <= i + nk - nq."""
    if not causal:
        return nq * nk
    # row i keeps keys 0 .. i + nk - nq (inclusive), clipped to nk
    return int(np.minimum(nk, np.arange(nq, dtype=np.int64) + (nk - nq) + 1).sum())


# The five workloads (shapes, masks and seeds of the method's evaluation).
WORKLOADS = {
    "kl_b1h1_n128_d64": Workload("kl_b1h1_n128_d64", 1, 1, 128, 128, 64, False, 0.3, 0),
    "kl_b2h32_n4096_d128": Workload("kl_b2h32_n4096_d128", 2, 32, 4096, 4096, 128, False, 0.5, 2),
    "kl_b2h32_n4096_d128_causal": Workload("kl_b2h32_n4096_d128_causal", 2, 32, 4096, 4096, 128, True, 0.5, 2),
    "kl_b1h32_n65536_d128_causal": Workload("kl_b1h32_n65536_d128_causal", 1, 32, 65536, 65536, 128, True, 0.5, 3),
    "decode_b8h32_nq1_nk131072_d128": Workload("decode_b8h32_nq1_nk131072_d128", 8, 32, 1, 131072, 128, False, 0.5, 4),
    "decode_b8h32_nq4_nk131072_d128": Workload("decode_b8h32_nq4_nk131072_d128", 8, 32, 4, 131072, 128, False, 0.5, 4),
    "decode_b8h32_nq16_nk131072_d128": Workload("decode_b8h32_nq16_nk131072_d128", 8, 32, 16, 131072, 128, False, 0.5, 4),
    "kl_b1h8_n524288_d128_causal": Workload("kl_b1h8_n524288_d128_causal", 1, 8, 524288, 524288, 128, True, 0.5, 5),
}


# ----------------------------------------------------------------------------
# bf16 helpers (bit patterns in uint16)
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round to nearest, ties to even); finite inputs."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(b).astype(np.float64)


# ----------------------------------------------------------------------------
# generation
# ----------------------------------------------------------------------------

def _normal(seed: int, tensor: int, b: int, h: int, n: int, d: int) -> np.ndarray:
    gen = np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, tensor, b, h])))
    out = np.empty((n, d), dtype=np.float32)
    gen.standard_normal(out=out, dtype=np.float32)
    return out


def head_slice(w: Workload, which: str, b: int, h: int) -> np.ndarray:
    """bf16 bits ``[N, D]`` of one head of ``which`` in {"q1","k1","q2","k2"}."""
    is_q = which[0] == "q"
    n = w.NQ if is_q else w.NK
    teacher = f32_to_bf16_bits(_normal(w.seed, _Q1 if is_q else _K1, b, h, n, w.D))
    if which[1] == "1":
        return teacher
    z = _normal(w.seed, _ZQ if is_q else _ZK, b, h, n, w.D)
    student = bf16_bits_to_f32(teacher) + np.float32(w.sigma) * z
    return f32_to_bf16_bits(student)


def head_rows(w: Workload, which: str, b: int, h: int, n: int) -> np.ndarray:
    """The first ``n`` rows of ``head_slice(w, which, b, h)`` without drawing the rest.

    Each Philox stream fills its ``[N, D]`` array row by row, so a shorter draw
    is a prefix of the full one.
    """
    is_q = which[0] == "q"
    full = w.NQ if is_q else w.NK
    return head_slice(w.with_(**({"NQ": min(n, full)} if is_q else {"NK": min(n, full)})), which, b, h)


def _threads() -> int:
    try:
        return max(1, min(32, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, min(32, os.cpu_count() or 1))


def make_inputs(w: Workload, threads: int | None = None) -> dict[str, np.ndarray]:
    """All four tensors as bf16 bits ``[B, H, N, D]`` plus ``g`` fp32 ``[B, H, N_Q]``."""
    out = {
        "q1": np.empty((w.B, w.H, w.NQ, w.D), np.uint16),
        "k1": np.empty((w.B, w.H, w.NK, w.D), np.uint16),
        "q2": np.empty((w.B, w.H, w.NQ, w.D), np.uint16),
        "k2": np.empty((w.B, w.H, w.NK, w.D), np.uint16),
    }

    def fill(job):
        b, h, is_q = job
        n = w.NQ if is_q else w.NK
        t1, z = (_Q1, _ZQ) if is_q else (_K1, _ZK)
        teacher = f32_to_bf16_bits(_normal(w.seed, t1, b, h, n, w.D))
        student = f32_to_bf16_bits(bf16_bits_to_f32(teacher) + np.float32(w.sigma) *
                                   _normal(w.seed, z, b, h, n, w.D))
        key = "q" if is_q else "k"
        out[key + "1"][b, h] = teacher
        out[key + "2"][b, h] = student

    jobs = [(b, h, q) for b in range(w.B) for h in range(w.H) for q in (True, False)]
    nt = threads or _threads()
    if nt == 1 or len(jobs) == 1:
        for j in jobs:
            fill(j)
    else:
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(fill, jobs))
    out["g"] = upstream_grad(w)
    return out


def upstream_grad(w: Workload) -> np.ndarray:
    """Per-row dLoss/dKL_i for a mean over query rows: the constant 1/N_Q."""
    return np.full((w.B, w.H, w.NQ), 1.0 / max(w.NQ, 1), dtype=np.float32)


def sample_rows(w: Workload, count: int, seed: int) -> np.ndarray:
    """``count`` distinct (b, h, i) triples, always holding the tile edges.

    Rows 0, 1, 127, 128 and N_Q-1 (those that exist) are always present, on
    seeded heads; the rest are drawn uniformly without replacement.
    """
    rng = np.random.default_rng(seed)
    forced = sorted({i for i in (0, 1, 127, 128, w.NQ - 1) if 0 <= i < w.NQ})
    picks = set()
    for i in forced:
        picks.add((int(rng.integers(w.B)), int(rng.integers(w.H)), i))
    total = w.B * w.H * w.NQ
    count = min(count, total)
    while len(picks) < count:
        flat = rng.integers(total, size=2 * count)
        for f in flat:
            b, rem = divmod(int(f), w.H * w.NQ)
            h, i = divmod(rem, w.NQ)
            picks.add((b, h, i))
            if len(picks) >= count:
                break
    return np.array(sorted(picks), dtype=np.int64).reshape(-1, 3)
