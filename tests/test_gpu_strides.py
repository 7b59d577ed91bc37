"""GPU parity for inputs read in place through strides: [B, N, H, D] tensors
permuted to [B, H, N, D], and Q/K slices of a packed [B, N, 3, H, D] tensor.

Every strided run is compared with the fp64 oracle and with the same call on
contiguous copies of the inputs.  The kernels see the same tiles either way, so
everything they compute in a fixed order (KL, LSE, dQ, the separate path's dK)
is bit-identical; the fused path's dK, summed by atomics in no fixed order, is
held to the oracle's tolerance.  Gradients are written with the strides of the
input they belong to, and nothing outside those rows is touched.
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


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    skl.lib()
    yield
    assert skl.check_device_status() == K.OK, "a device-side wait timed out during this module"


def bnhd(t):
    """The same values stored as [B, N, H, D], viewed as [B, H, N, D]."""
    return t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)


def packed(ts):
    """Views of slot i of one packed [B, N, len(ts), H, D] tensor holding ts[i]."""
    B, H, N, D = ts[0].shape
    buf = torch.zeros(B, N, len(ts), H, D, dtype=ts[0].dtype, device=ts[0].device)
    for i, t in enumerate(ts):
        buf[:, :, i] = t.permute(0, 2, 1, 3)
    return [buf[:, :, i].permute(0, 2, 1, 3) for i in range(len(ts))]


def layout(kind, q1, k1, q2, k2):
    if kind == "bnhd":
        return [bnhd(t) for t in (q1, k1, q2, k2)]
    if kind == "q_bnhd_k_contig":
        return [bnhd(q1), k1, bnhd(q2), k2]
    if kind == "packed":  # Q1, Q2 from one packed tensor, K1, K2 from another
        (a1, a2), (b1, b2) = packed([q1, q2]), packed([k1, k2])
        return [a1, b1, a2, b2]
    raise ValueError(kind)


CASES = [
    # B, H, NQ, NK, D, causal
    (2, 3, 300, 300, 128, True),
    (1, 2, 77, 333, 64, False),
    (2, 2, 260, 390, 128, True),
]


def _bwd(setting, ins, kl, l1, l2, g, w, mode):
    q1, k1, q2, k2 = ins
    if setting == 1:
        return skl.bwd_s1(q1, k1, q2, k2, l1, l2, g, w.softmax_scale, w.causal, mode)
    return skl.bwd_s2(q1, k1, q2, k2, l1, l2, kl, g, w.softmax_scale, w.causal, mode)


@pytest.mark.parametrize("kind", ["bnhd", "q_bnhd_k_contig", "packed"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}h{}q{}k{}d{}{}".format(*c[:5], "c" if c[5] else ""))
def test_strided_inputs_match_contiguous_and_oracle(case, kind):
    B, H, NQ, NK, D, causal = case
    w = synth.Workload("strided", B, H, NQ, NK, D, causal, 0.5, 7 + NQ + NK + D)
    inp = synth.make_inputs(w)
    contig = U.dev_inputs(inp)
    strided = layout(kind, *contig)
    for t, c in zip(strided, contig):
        assert torch.equal(t, c)
    assert K._bhn_strides(strided[0]) != K._bhn_strides(contig[0])
    g = torch.from_numpy(inp["g"]).cuda()

    ref_rows = skl.fwd(*contig, w.softmax_scale, causal)
    rows = skl.fwd(*strided, w.softmax_scale, causal)
    for a, b in zip(rows, ref_rows):
        assert torch.equal(a, b)
    Q1, K1, Q2, K2 = (U.f64(inp[k]) for k in ("q1", "k1", "q2", "k2"))
    rkl, rl1, rl2 = O.forward(Q1, K1, Q2, K2, w.softmax_scale, causal)
    U.assert_rows(*(U.np64(x) for x in rows), rkl, rl1, rl2, f"{kind} fwd")
    kl, l1, l2 = rows

    for setting in (1, 2):
        rdq, rdk = O.backward(setting, Q1, K1, Q2, K2, w.softmax_scale, causal, inp["g"])
        q_src, k_src = (strided[2], strided[3]) if setting == 1 else (strided[0], strided[1])
        for mode in (skl.BWD_FUSED, skl.BWD_SEPARATE):
            dq, dk = _bwd(setting, strided, kl, l1, l2, g, w, mode)
            cq, ck = _bwd(setting, contig, kl, l1, l2, g, w, mode)
            assert K._bhn_strides(dq) == K._bhn_strides(q_src) and K._bhn_strides(dk) == K._bhn_strides(k_src)
            assert torch.equal(dq, cq), f"{kind} setting {setting} mode {mode}: dQ differs from the contiguous run"
            if mode == skl.BWD_SEPARATE:
                assert torch.equal(dk, ck), f"{kind} setting {setting}: dK differs from the contiguous run"
            U.assert_grad(U.np64(dq), rdq, f"{kind} setting {setting} mode {mode} dQ")
            U.assert_grad(U.np64(dk), rdk, f"{kind} setting {setting} mode {mode} dK")


@pytest.mark.parametrize("nq", [1, 4, 16])
def test_strided_splitk(nq):
    w = synth.Workload("strided_decode", 2, 4, nq, 3000, 128, False, 0.5, 31 + nq)
    inp = synth.make_inputs(w)
    contig = U.dev_inputs(inp)
    strided = layout("bnhd", *contig)
    a = skl.fwd_splitk(*strided, w.softmax_scale, False, 5)
    b = skl.fwd_splitk(*contig, w.softmax_scale, False, 5)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    Q1, K1, Q2, K2 = (U.f64(inp[k]) for k in ("q1", "k1", "q2", "k2"))
    U.assert_rows(*(U.np64(x) for x in a), *O.forward(Q1, K1, Q2, K2, w.softmax_scale, False), "strided splitk")


@pytest.mark.parametrize("mode", [K.BWD_FUSED, K.BWD_SEPARATE])
def test_gradients_land_in_a_packed_gradient_buffer(mode):
    """Inputs are slots of packed [B, N, 3, H, D] tensors; dQ2 and dK2 are written
    straight into slots 0 and 1 of a packed gradient buffer of the same layout,
    and slot 2 keeps its sentinel."""
    B, H, N, D = 2, 3, 200, 128
    w = synth.Workload("packed_grad", B, H, N, N, D, True, 0.5, 99)
    inp = synth.make_inputs(w)
    contig = U.dev_inputs(inp)
    pad = torch.zeros_like(contig[0])
    q1, k1, _ = packed([contig[0], contig[1], pad])
    q2, k2, _ = packed([contig[2], contig[3], pad])
    kl, l1, l2 = skl.fwd(q1, k1, q2, k2, w.softmax_scale, True)
    g = torch.from_numpy(inp["g"]).cuda()
    sentinel = torch.tensor(-7.0, dtype=torch.bfloat16).item()
    grad = torch.full((B, N, 3, H, D), sentinel, dtype=torch.bfloat16, device="cuda")
    dq_v, dk_v = grad[:, :, 0].permute(0, 2, 1, 3), grad[:, :, 1].permute(0, 2, 1, 3)
    qs, ks = K._bhn_strides(q2), K._bhn_strides(k2)
    assert qs == K._bhn_strides(dq_v) and ks == K._bhn_strides(dk_v)
    s = K.make_shape(B, H, N, N, D, w.softmax_scale, True, qs, ks)
    nbytes = ctypes.c_size_t(0)
    assert K.lib().streamkl_bwd_workspace(s, mode, ctypes.byref(nbytes)) == K.OK
    ws = torch.empty(max(16, nbytes.value), dtype=torch.uint8, device="cuda")
    st = K.lib().streamkl_bwd_s1(K._ptr(q1), K._ptr(k1), K._ptr(q2), K._ptr(k2), s, K._ptr(l1), K._ptr(l2),
                                 K._ptr(g), K._ptr(dq_v), K._ptr(dk_v), mode, K._ptr(ws), nbytes.value,
                                 K._stream(q1.device))
    assert st == K.OK
    torch.cuda.synchronize()
    assert bool((grad[:, :, 2] == sentinel).all())
    ref_q, ref_k = skl.bwd_s1(*contig, l1, l2, g, w.softmax_scale, True, mode)
    assert torch.equal(dq_v, ref_q)
    if mode == K.BWD_SEPARATE:
        assert torch.equal(dk_v, ref_k)
    else:
        U.assert_grad(U.np64(dk_v), U.np64(ref_k), "packed fused dK")
    Q1, K1, Q2, K2 = (U.f64(inp[k]) for k in ("q1", "k1", "q2", "k2"))
    rdq, rdk = O.backward(1, Q1, K1, Q2, K2, w.softmax_scale, True, inp["g"])
    U.assert_grad(U.np64(dq_v), rdq, "packed dQ2")
    U.assert_grad(U.np64(dk_v), rdk, "packed dK2")


def test_unaligned_view_is_copied_not_refused():
    """A view whose strides the tensor maps cannot take is made contiguous by the binding."""
    w = synth.Workload("odd", 1, 2, 100, 100, 64, False, 0.5, 5)
    inp = synth.make_inputs(w)
    contig = U.dev_inputs(inp)
    big = torch.zeros(1, 2, 100, 64 + 4, dtype=torch.bfloat16, device="cuda")  # row stride 68: not a multiple of 8
    big[..., :64] = contig[0]
    q1 = big[..., :64]
    assert K._bhn_strides(q1) is None
    a = skl.fwd(q1, *contig[1:], w.softmax_scale, False)
    b = skl.fwd(*contig, w.softmax_scale, False)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("mode", [K.BWD_FUSED, K.BWD_SEPARATE])
def test_no_query_rows_zero_only_the_strided_dk_rows(mode):
    """With N_Q = 0 the loss is an empty sum, so dK is zero: it is written with
    K's strides into slot 1 of a packed gradient buffer, and slots 0 and 2 keep
    their sentinel."""
    B, H, NK, D = 2, 3, 200, 128
    w = synth.Workload("packed_empty", B, H, 0, NK, D, True, 0.5, 98)
    inp = synth.make_inputs(w)
    q1, k1, q2, k2 = U.dev_inputs(inp)
    pad = torch.zeros_like(k1)
    _, k1p, _ = packed([pad, k1, pad])
    _, k2p, _ = packed([pad, k2, pad])
    sentinel = torch.tensor(-7.0, dtype=torch.bfloat16).item()
    grad = torch.full((B, NK, 3, H, D), sentinel, dtype=torch.bfloat16, device="cuda")
    dk_v = grad[:, :, 1].permute(0, 2, 1, 3)
    ks = K._bhn_strides(k2p)
    assert ks == K._bhn_strides(dk_v)
    s = K.make_shape(B, H, 0, NK, D, w.softmax_scale, True, (0, 0, 0), ks)
    nbytes = ctypes.c_size_t(0)
    assert K.lib().streamkl_bwd_workspace(s, mode, ctypes.byref(nbytes)) == K.OK
    ws = torch.empty(max(16, nbytes.value), dtype=torch.uint8, device="cuda")
    rows = torch.zeros((B, H, 16), device="cuda")  # 16-byte aligned stand-ins for the empty row vectors
    dq = torch.empty((B, H, 0, D), dtype=torch.bfloat16, device="cuda")
    st = K.lib().streamkl_bwd_s1(K._ptr(q1), K._ptr(k1p), K._ptr(q2), K._ptr(k2p), s, K._ptr(rows), K._ptr(rows),
                                 K._ptr(rows), K._ptr(dq), K._ptr(dk_v), mode, K._ptr(ws), nbytes.value,
                                 K._stream(k1.device))
    assert st == K.OK
    torch.cuda.synchronize()
    assert bool((dk_v == 0).all())
    assert bool((grad[:, :, 0] == sentinel).all()) and bool((grad[:, :, 2] == sentinel).all())
