"""The autograd entry point: gradients route to setting 1 / setting 2 and match the oracle."""
import numpy as np
import pytest
import torch

import attention_kl_divergence_streamkl_gb300 as skl
from attention_kl_divergence_streamkl_gb300 import build, synth
from oracle import oracle as O
from tests import parity_util as U

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
@pytest.mark.parametrize("causal", [False, True])
def test_attention_kl_autograd_matches_oracle(reduction, causal):
    build.build()
    w = synth.Workload("ag", 1, 3, 200, 200, 128, causal, 0.5, 31)
    inp = synth.make_inputs(w)
    q1, k1, q2, k2 = (t.requires_grad_() for t in U.dev_inputs(inp))
    out = skl.attention_kl(q1, k1, q2, k2, w.softmax_scale, causal, reduction)
    rng = np.random.default_rng(5)
    if reduction == "none":
        gout = torch.from_numpy(rng.uniform(0.5, 1.5, (w.B, w.H, w.NQ)).astype(np.float32)).cuda()
        out.backward(gout)
        g = gout.double().cpu().numpy()
    else:
        out.backward(torch.tensor(2.0, device="cuda"))
        n = w.B * w.H * w.NQ
        g = np.full((w.B, w.H, w.NQ), 2.0 / (n if reduction == "mean" else 1.0))
    F = [U.f64(inp[k]) for k in ("q1", "k1", "q2", "k2")]
    kl, _, _ = O.forward(*F, w.softmax_scale, causal)
    ref = {"mean": kl.mean(), "sum": kl.sum()}.get(reduction)
    if ref is None:
        got = U.np64(out)
        assert np.all(np.abs(got - kl) <= U.KL_ABS + U.KL_REL * np.abs(kl))
    else:
        assert abs(float(out) - ref) <= 1e-3 + 5e-3 * abs(ref)
    dq2, dk2 = O.backward(1, *F, w.softmax_scale, causal, g)
    dq1, dk1 = O.backward(2, *F, w.softmax_scale, causal, g)
    for got, ref_, name in ((q1.grad, dq1, "dQ1"), (k1.grad, dk1, "dK1"), (q2.grad, dq2, "dQ2"), (k2.grad, dk2, "dK2")):
        U.assert_grad(U.np64(got), ref_, name)


def test_only_the_side_that_requires_grad_is_computed():
    build.build()
    w = synth.Workload("ag2", 1, 2, 130, 150, 64, True, 0.5, 32)
    inp = synth.make_inputs(w)
    q1, k1, q2, k2 = U.dev_inputs(inp)
    q2.requires_grad_()
    k2.requires_grad_()
    skl.attention_kl(q1, k1, q2, k2, w.softmax_scale, True).backward()
    assert q1.grad is None and k1.grad is None
    F = [U.f64(inp[k]) for k in ("q1", "k1", "q2", "k2")]
    g = np.full((w.B, w.H, w.NQ), 1.0 / (w.B * w.H * w.NQ))
    dq2, dk2 = O.backward(1, *F, w.softmax_scale, True, g)
    U.assert_grad(U.np64(q2.grad), dq2, "dQ2")
    U.assert_grad(U.np64(k2.grad), dk2, "dK2")
