"""GPU parity of the mutual-case backward (streamkl_bwd_mutual): dQ1, dK1 and
dQ2, dK2 of one loss, with the mutual kernels (one recompute of each logit tile
pair for both settings) or a fused pass per setting.

Each output is checked against the fp64 oracle's setting-2 (dQ1, dK1) and
setting-1 (dQ2, dK2) gradients.  The mutual kernels are also checked against
the separate single-setting kernels: they form the same dS bits and accumulate
them in the same order with the same MMA shapes, so their outputs are
bit-identical.
"""
import ctypes

import numpy as np
import pytest
import torch

import attention_kl_divergence_streamkl_gb300 as skl
from attention_kl_divergence_streamkl_gb300 import _lib as K
from attention_kl_divergence_streamkl_gb300 import build, synth
from oracle import oracle as O
from tests import parity_util as U

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    skl.lib()
    yield
    assert skl.check_device_status() == K.OK, "a device-side wait timed out during this module"


def _forward(inp, w):
    ins = U.dev_inputs(inp)
    kl, l1, l2 = skl.fwd(*ins, w.softmax_scale, w.causal)
    g = torch.from_numpy(inp["g"]).cuda()
    return ins, kl, l1, l2, g


def _separate(ins, kl, l1, l2, g, w):
    dq2, dk2 = skl.bwd_s1(*ins, l1, l2, g, w.softmax_scale, w.causal, skl.BWD_SEPARATE)
    dq1, dk1 = skl.bwd_s2(*ins, l1, l2, kl, g, w.softmax_scale, w.causal, skl.BWD_SEPARATE)
    return dq1, dk1, dq2, dk2


NAMES = ("dQ1", "dK1", "dQ2", "dK2")

SMALL = [
    # B, H, NQ, NK, D, causal
    (1, 1, 128, 128, 64, False),
    (2, 3, 300, 300, 128, True),
    (2, 2, 300, 300, 128, False),
    (1, 2, 77, 333, 128, True),
    (1, 2, 77, 333, 64, False),
    (1, 2, 5, 200, 64, True),
    (1, 1, 130, 70, 128, False),
    (2, 1, 1, 1, 128, False),
    (1, 1, 257, 1000, 64, True),
    (1, 2, 700, 700, 128, True),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "b{}h{}q{}k{}d{}{}".format(*c[:5], "c" if c[5] else ""))
def test_small_shapes_full_oracle_and_separate(case):
    B, H, NQ, NK, D, causal = case
    w = synth.Workload("mutual", B, H, NQ, NK, D, causal, 0.5, 200 + NQ + NK + D)
    inp = synth.make_inputs(w)
    ins, kl, l1, l2, g = _forward(inp, w)
    got = skl.bwd_mutual(*ins, l1, l2, kl, g, w.softmax_scale, causal, skl.BWD_SEPARATE)
    sep = _separate(ins, kl, l1, l2, g, w)
    for name, a, b in zip(NAMES, got, sep):
        assert torch.equal(a, b), f"{name}: mutual differs from the separate kernels"
    Q1, K1, Q2, K2 = (U.f64(inp[k]) for k in ("q1", "k1", "q2", "k2"))
    r2 = O.backward(2, Q1, K1, Q2, K2, w.softmax_scale, causal, inp["g"])
    r1 = O.backward(1, Q1, K1, Q2, K2, w.softmax_scale, causal, inp["g"])
    gsum = np.abs(inp["g"]).sum(axis=-1)
    tols = (U.zero_grad_tol(inp["g"], w.softmax_scale, K1), U.zero_grad_tol(gsum, w.softmax_scale, Q1),
            U.zero_grad_tol(inp["g"], w.softmax_scale, K2), U.zero_grad_tol(gsum, w.softmax_scale, Q2))
    for name, t, ref, zt in zip(NAMES, got, (r2[0], r2[1], r1[0], r1[1]), tols):
        U.assert_grad(U.np64(t), ref, f"mutual {name}", zero_tol=zt)


@pytest.mark.parametrize("name", ["kl_b2h32_n4096_d128", "kl_b2h32_n4096_d128_causal"])
def test_b2h32_n4096_every_head_bitwise_and_two_heads_oracle(name):
    w = W[name]
    inp = synth.make_inputs(w)
    ins, kl, l1, l2, g = _forward(inp, w)
    got = skl.bwd_mutual(*ins, l1, l2, kl, g, w.softmax_scale, w.causal, skl.BWD_SEPARATE)
    sep = _separate(ins, kl, l1, l2, g, w)
    for nm, a, b in zip(NAMES, got, sep):
        assert torch.equal(a, b), f"{nm}: mutual differs from the separate kernels"
    rng = np.random.default_rng(4000 + w.seed)
    heads = [(int(rng.integers(w.B)), int(rng.integers(w.H))) for _ in range(2)]
    for b, h in heads:
        _, (rdq2, rdk2) = U.oracle_head(inp, w, b, h, setting=1)
        _, (rdq1, rdk1) = U.oracle_head(inp, w, b, h, setting=2)
        for nm, t, ref in zip(NAMES, got, (rdq1, rdk1, rdq2, rdk2)):
            U.assert_grad(U.np64(t[b, h]), ref, f"{name} head {b},{h} {nm}")


def test_n65536_causal_two_heads_bitwise_sampled_rows_and_last_keys():
    """Two heads of the long causal workload: mutual = separate on every element;
    dQ1, dQ2 on 64 sampled rows and dK1, dK2 of the last 128 keys against the oracle."""
    full = W["kl_b1h32_n65536_d128_causal"]
    w = synth.Workload("mutual_64k", 1, 2, full.NQ, full.NK, full.D, True, full.sigma, full.seed)
    inp = synth.make_inputs(w)
    ins, kl, l1, l2, g = _forward(inp, w)
    got = skl.bwd_mutual(*ins, l1, l2, kl, g, w.softmax_scale, True, skl.BWD_SEPARATE)
    sep = _separate(ins, kl, l1, l2, g, w)
    for nm, a, b in zip(NAMES, got, sep):
        assert torch.equal(a, b), f"{nm}: mutual differs from the separate kernels"
    rows = synth.sample_rows(w, 64, 5000 + w.seed)
    b, h, i = rows[:, 0], rows[:, 1], rows[:, 2]
    for setting, dq in ((2, got[0]), (1, got[2])):
        _, _, _, rdq = U.oracle_rows(inp, w, rows, setting=setting)
        U.assert_grad(U.np64(dq)[b, h, i], rdq, f"setting {setting} dQ sampled rows")
    R = 128
    for setting, dk in ((2, got[1]), (1, got[3])):
        refs = U.map_heads(lambda bb, hh: U.oracle_last_keys_dk(inp, w, bb, hh, setting, R), [(0, 0), (0, 1)],
                           threads=2)
        for hh, rdk in enumerate(refs):
            U.assert_grad(U.np64(dk[0, hh, -R:]), rdk, f"setting {setting} dK last {R} keys head {hh}")


def test_strided_inputs_write_strided_gradients():
    """[B, N, H, D] storage viewed as [B, H, N, D]: the gradients take their inputs' strides and equal
    the contiguous run bit for bit."""
    w = synth.Workload("mutual_strided", 2, 3, 260, 390, 128, True, 0.5, 77)
    inp = synth.make_inputs(w)
    ins, kl, l1, l2, g = _forward(inp, w)
    strided = [t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3) for t in ins]
    a = skl.bwd_mutual(*strided, l1, l2, kl, g, w.softmax_scale, True, skl.BWD_SEPARATE)
    b = skl.bwd_mutual(*ins, l1, l2, kl, g, w.softmax_scale, True, skl.BWD_SEPARATE)
    for t, src in zip(a, (strided[0], strided[1], strided[2], strided[3])):
        assert K._bhn_strides(t) == K._bhn_strides(src)
    for nm, x, y in zip(NAMES, a, b):
        assert torch.equal(x, y), nm


def test_no_query_rows_and_bad_pointers():
    w = synth.Workload("mutual_empty", 1, 2, 0, 200, 64, False, 0.5, 8)
    inp = synth.make_inputs(w)
    ins = U.dev_inputs(inp)
    rows = torch.zeros((1, 2, 0), device="cuda")
    for mode in (skl.BWD_SEPARATE, skl.BWD_FUSED, skl.BWD_AUTO):
        dq1, dk1, dq2, dk2 = skl.bwd_mutual(*ins, rows, rows, rows, rows, None, False, mode)
        assert dq1.numel() == 0 and dq2.numel() == 0
        assert float(dk1.float().abs().max()) == 0.0 and float(dk2.float().abs().max()) == 0.0
    # a NULL output is refused before any launch
    w = synth.Workload("mutual_bad", 1, 1, 64, 64, 64, False, 0.5, 9)
    inp = synth.make_inputs(w)
    ins, kl, l1, l2, g = _forward(inp, w)
    s = K.make_shape(1, 1, 64, 64, 64, None, False)
    out = [torch.empty_like(t) for t in ins]
    ptrs = [K._ptr(t) for t in out]
    for k in range(4):
        bad = list(ptrs)
        bad[k] = None
        st = K.lib().streamkl_bwd_mutual(*(K._ptr(t) for t in ins), s, K._ptr(l1), K._ptr(l2), K._ptr(kl), K._ptr(g),
                                         *bad, K.BWD_SEPARATE, None, 0, K._stream(ins[0].device))
        assert st == K.ERR_INVALID
    st = K.lib().streamkl_bwd_mutual(*(K._ptr(t) for t in ins), s, K._ptr(l1), K._ptr(l2), None, K._ptr(g),
                                     *ptrs, K.BWD_SEPARATE, None, 0, K._stream(ins[0].device))
    assert st == K.ERR_INVALID


@pytest.mark.parametrize("case", [(2, 3, 300, 300, 128, True), (1, 2, 77, 333, 64, False), (1, 4, 128, 40000, 128, False)],
                         ids=lambda c: "b{}h{}q{}k{}d{}{}".format(*c[:5], "c" if c[5] else ""))
def test_fused_and_auto_modes_against_oracle(case):
    """A fused pass per setting (and whatever AUTO picks) gives the oracle's four gradients; its dQ equals the
    single-setting fused call bit for bit (dQ is summed in a fixed order; dK by atomics is not)."""
    B, H, NQ, NK, D, causal = case
    w = synth.Workload("mutual_modes", B, H, NQ, NK, D, causal, 0.5, 300 + NQ + NK + D)
    inp = synth.make_inputs(w)
    ins, kl, l1, l2, g = _forward(inp, w)
    Q1, K1, Q2, K2 = (U.f64(inp[k]) for k in ("q1", "k1", "q2", "k2"))
    heads = [(b, h) for b in range(B) for h in range(H)][:2]
    for mode in (skl.BWD_FUSED, skl.BWD_AUTO):
        got = skl.bwd_mutual(*ins, l1, l2, kl, g, w.softmax_scale, causal, mode)
        if mode == skl.BWD_FUSED:
            dq2, _ = skl.bwd_s1(*ins, l1, l2, g, w.softmax_scale, causal, skl.BWD_FUSED)
            dq1, _ = skl.bwd_s2(*ins, l1, l2, kl, g, w.softmax_scale, causal, skl.BWD_FUSED)
            assert torch.equal(got[0], dq1) and torch.equal(got[2], dq2)
        for b, h in heads:
            q1, k1, q2, k2 = U.head_f64(inp, b, h)
            gg = inp["g"][b, h]
            rdq2, rdk2 = O.head_backward(1, q1, k1, q2, k2, w.softmax_scale, causal, gg)
            rdq1, rdk1 = O.head_backward(2, q1, k1, q2, k2, w.softmax_scale, causal, gg)
            for nm, t, ref in zip(NAMES, got, (rdq1, rdk1, rdq2, rdk2)):
                U.assert_grad(U.np64(t[b, h]), ref, f"mode {mode} head {b},{h} {nm}")


def test_auto_follows_the_mutual_rule():
    props = torch.cuda.get_device_properties(0)
    l2, sms = props.L2_cache_size, props.multi_processor_count
    assert skl.bwd_mutual_select(1, 32, 128, 65536, 128, l2, sms) == skl.BWD_SEPARATE
    assert skl.bwd_mutual_select(1, 32, 65536, 65536, 128, l2, sms, True) == skl.BWD_FUSED


@pytest.mark.parametrize("causal", [False, True])
def test_autograd_mutual_matches_the_oracle(causal):
    """attention_kl with all four inputs requiring grad: the four gradients of the mean KL against the oracle,
    through AUTO and through an explicit mutual-kernel request (then equal to the separate kernels' bits)."""
    w = synth.Workload("mutual_autograd", 2, 2, 200, 300 if not causal else 200, 64, causal, 0.5, 31)
    inp = synth.make_inputs(w)
    Q1, K1, Q2, K2 = (U.f64(inp[k]) for k in ("q1", "k1", "q2", "k2"))
    gm = np.full((w.B, w.H, w.NQ), 1.0 / (w.B * w.H * w.NQ))
    r2 = O.backward(2, Q1, K1, Q2, K2, w.softmax_scale, causal, gm)
    r1 = O.backward(1, Q1, K1, Q2, K2, w.softmax_scale, causal, gm)
    for mode in (skl.BWD_AUTO, skl.BWD_SEPARATE):
        ins = [t.clone().requires_grad_() for t in U.dev_inputs(inp)]
        loss = skl.attention_kl(*ins, w.softmax_scale, causal, reduction="mean", bwd_mode=mode)
        loss.backward()
        for nm, t, ref in zip(NAMES, ins, (r2[0], r2[1], r1[0], r1[1])):
            U.assert_grad(U.np64(t.grad), ref, f"autograd mode {mode} {nm}")
        if mode == skl.BWD_SEPARATE:
            kl, l1, l2 = skl.fwd(*(t.detach() for t in ins), w.softmax_scale, causal)
            gg = torch.full_like(kl, 1.0 / kl.numel())
            ref = _separate([t.detach() for t in ins], kl, l1, l2, gg, w)
            for nm, t, r in zip(NAMES, ins, ref):
                assert torch.equal(t.grad, r), nm
