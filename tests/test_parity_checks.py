"""The GPU tests' gradient checks must fail a wrong gradient at the sizes the
workloads really have (CPU only).

With g = 1/N_Q a gradient element is tiny at long contexts (about 1e-6 at 4K
queries, 1e-7 at 64K, 1e-8 at 512K), so any absolute floor in a relative
check would pass an all-zero gradient there.  These tests take dQ rows of the
real workloads from the oracle (their first rows, causal, with the workload's
g) and feed the checks a zero gradient, a 5 % scale error and bf16-sized noise.
"""
import numpy as np
import pytest
import torch

from attention_kl_divergence_streamkl_gb300 import synth
from oracle import oracle as O
from tests import parity_util as U

PREFIX = 1024  # causal rows i < PREFIX see only the first PREFIX keys


def _dq_rows(name, setting):
    w = synth.WORKLOADS[name]
    n = min(PREFIX, w.NQ)
    q1, k1, q2, k2 = (synth.bf16_bits_to_f64(synth.head_rows(w, k, 0, 0, n)) for k in ("q1", "k1", "q2", "k2"))
    rows = np.arange(n - 64, n)
    g = np.full(rows.size, 1.0 / w.NQ)
    return O.rows_backward_dq(setting, q1, k1, q2, k2, w.softmax_scale, True, g, rows)


@pytest.mark.parametrize("name", ["kl_b2h32_n4096_d128_causal", "kl_b1h32_n65536_d128_causal",
                                  "kl_b1h8_n524288_d128_causal"])
@pytest.mark.parametrize("setting", [1, 2])
def test_assert_grad_has_no_floor(name, setting):
    ref = _dq_rows(name, setting)
    assert 0 < np.sqrt(np.mean(ref ** 2)) < 1e-4  # the magnitudes a floor would swallow
    rng = np.random.default_rng(0)
    U.assert_grad(ref + ref * rng.uniform(-2 ** -8, 2 ** -8, ref.shape), ref, "bf16-sized noise")
    for bad, what in ((0 * ref, "zero"), (1.05 * ref, "5% scale"), (ref[::-1], "rows swapped")):
        with pytest.raises(AssertionError):
            U.assert_grad(bad, ref, what)


def test_assert_grad_zero_rows():
    ref = np.zeros((3, 8))
    ref[1] = 1e-7
    U.assert_grad(ref, ref)
    got = ref.copy()
    got[0] = 1e-11  # within 1e-3 of the largest row
    U.assert_grad(got, ref)
    got[0] = 5e-10  # 0.5 % of the Frobenius norm, but 5e-3 of the largest row
    assert U.grad_error(got, ref) < U.GRAD_REL
    with pytest.raises(AssertionError):
        U.assert_grad(got, ref)
    with pytest.raises(AssertionError):  # an all-zero reference needs a bound from the caller
        U.assert_grad(np.zeros((2, 4)), np.zeros((2, 4)))
    U.assert_grad(np.full((2, 4), 1e-12), np.zeros((2, 4)), zero_tol=1e-10)


def _head_grads(setting, nq=512, d=32, seed=7):
    w = synth.Workload("inv", 1, 2, nq, nq, d, True, 0.5, seed)
    inp = synth.make_inputs(w)
    Q1, K1, Q2, K2 = (synth.bf16_bits_to_f64(inp[k]) for k in ("q1", "k1", "q2", "k2"))
    dq, dk = O.backward(setting, Q1, K1, Q2, K2, w.softmax_scale, True, inp["g"])
    qo, ko = (Q2, K2) if setting == 1 else (Q1, K1)
    return [torch.from_numpy(x) for x in (dk, ko, dq, qo)]


@pytest.mark.parametrize("setting", [1, 2])
def test_dk_invariants_reject_zero_and_scaled_dk(setting):
    dk, ko, dq, qo = _head_grads(setting)
    r_sum, r_tr, power = U.assert_dk_invariants(dk, ko, dq, qo, setting)
    assert r_sum < 1e-10 and r_tr < 1e-10
    with pytest.raises(AssertionError):
        U.assert_dk_invariants(0 * dk, ko, dq, qo, setting)
    if setting == 1:  # the trace identity sees dK's scale on every head
        for f in (1e-3, 0.9):
            with pytest.raises(AssertionError):
                U.assert_dk_invariants(f * dk, ko, dq, qo, setting)
