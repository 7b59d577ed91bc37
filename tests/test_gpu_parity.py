"""GPU parity: libstreamkl (through the C-ABI) against the fp64 CPU oracle.

Small multi-tile shapes with ragged tails are compared element by element
with the full oracle; each full-size workload runs in the launch configuration
the benchmark uses and is compared on seeded sampled rows or heads, plus
properties that hold at any size (sum_j dK_j = 0, the trace identity, Split-K =
non-split, fused = separate).
"""
import numpy as np
import pytest
import torch

import attention_kl_divergence_streamkl_gb300 as skl
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
    assert skl.check_device_status() == skl._lib.OK, "a device-side wait timed out during this module"


def _run_fwd(inp, w, splitk=False, num_splits=0):
    q1, k1, q2, k2 = U.dev_inputs(inp)
    if splitk:
        return skl.fwd_splitk(q1, k1, q2, k2, w.softmax_scale, w.causal, num_splits)
    return skl.fwd(q1, k1, q2, k2, w.softmax_scale, w.causal)


def _run_bwd(inp, w, setting, mode, kl, l1, l2):
    q1, k1, q2, k2 = U.dev_inputs(inp)
    g = torch.from_numpy(inp["g"]).cuda()
    if setting == 1:
        return skl.bwd_s1(q1, k1, q2, k2, l1, l2, g, w.softmax_scale, w.causal, mode)
    return skl.bwd_s2(q1, k1, q2, k2, l1, l2, kl, g, w.softmax_scale, w.causal, mode)


# ------------------------------------------------------------------ small shapes

SMALL = [
    # B, H, NQ, NK, D, causal
    (1, 1, 128, 128, 64, False),
    (2, 3, 300, 300, 128, True),
    (2, 3, 300, 300, 128, False),
    (1, 2, 77, 333, 128, True),
    (1, 2, 77, 333, 64, False),
    (1, 2, 5, 200, 64, True),
    (1, 1, 130, 70, 128, False),
    (2, 1, 1, 1, 128, False),
    (1, 1, 257, 257, 64, True),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "b{}h{}q{}k{}d{}{}".format(*c[:5], "c" if c[5] else ""))
def test_small_shapes_full_oracle(case):
    B, H, NQ, NK, D, causal = case
    w = synth.Workload("small", B, H, NQ, NK, D, causal, 0.5, 100 + NQ + NK + D)
    inp = synth.make_inputs(w)
    kl, l1, l2 = _run_fwd(inp, w)
    torch.cuda.synchronize()
    Q1, K1, Q2, K2 = (U.f64(inp[k]) for k in ("q1", "k1", "q2", "k2"))
    rkl, rl1, rl2 = O.forward(Q1, K1, Q2, K2, w.softmax_scale, causal)
    U.assert_rows(U.np64(kl), U.np64(l1), U.np64(l2), rkl, rl1, rl2, "fwd")
    if NQ <= 16:
        skl_ = _run_fwd(inp, w, splitk=True, num_splits=3)
        U.assert_rows(*(U.np64(x) for x in skl_), rkl, rl1, rl2, "splitk")
    for setting in (1, 2):
        rdq, rdk = O.backward(setting, Q1, K1, Q2, K2, w.softmax_scale, causal, inp["g"])
        Qo, Ko = (Q2, K2) if setting == 1 else (Q1, K1)
        zq = U.zero_grad_tol(inp["g"], w.softmax_scale, Ko)
        zk = U.zero_grad_tol(np.abs(inp["g"]).sum(axis=-1), w.softmax_scale, Qo)
        for mode in (skl.BWD_FUSED, skl.BWD_SEPARATE):
            dq, dk = _run_bwd(inp, w, setting, mode, kl, l1, l2)
            U.assert_grad(U.np64(dq), rdq, f"setting {setting} mode {mode} dQ", zero_tol=zq)
            U.assert_grad(U.np64(dk), rdk, f"setting {setting} mode {mode} dK", zero_tol=zk)


def test_128_row_workload_fwd_and_setting1():
    """The 128-row, D = 64 workload (sigma 0.3, seed 0): KL/LSE and dQ2, dK2 on every element."""
    w = W["kl_b1h1_n128_d64"]
    inp = synth.make_inputs(w)
    kl, l1, l2 = _run_fwd(inp, w)
    (rkl, rl1, rl2), (rdq, rdk) = U.oracle_head(inp, w, 0, 0, setting=1)
    U.assert_rows(U.np64(kl)[0, 0], U.np64(l1)[0, 0], U.np64(l2)[0, 0], rkl, rl1, rl2)
    for mode in (skl.BWD_AUTO, skl.BWD_FUSED, skl.BWD_SEPARATE):
        dq, dk = _run_bwd(inp, w, 1, mode, kl, l1, l2)
        U.assert_grad(U.np64(dq)[0, 0], rdq, "dQ2")
        U.assert_grad(U.np64(dk)[0, 0], rdk, "dK2")


# ------------------------------------------------------------------ full-size workloads

@pytest.mark.parametrize("name", ["kl_b2h32_n4096_d128", "kl_b2h32_n4096_d128_causal"])
def test_b2h32_n4096(name):
    """KL/LSE of every row of every head against the full oracle; both settings and both backward paths
    against the full oracle on 8 seeded heads; fused = separate and the dK identities on every head."""
    w = W[name]
    inp = synth.make_inputs(w)
    kl, l1, l2 = _run_fwd(inp, w)
    torch.cuda.synchronize()
    every = [(b, h) for b in range(w.B) for h in range(w.H)]
    rkl, rl1, rl2 = U.oracle_forward_heads(inp, w, every)
    U.assert_rows(U.np64(kl).reshape(-1, w.NQ), U.np64(l1).reshape(-1, w.NQ), U.np64(l2).reshape(-1, w.NQ),
                  rkl, rl1, rl2, "every row")
    rng = np.random.default_rng(1000 + w.seed)
    picks = rng.choice(len(every), size=8, replace=False)
    heads = [every[int(x)] for x in sorted(picks)]
    q1, k1, q2, k2 = U.dev_inputs(inp)
    for setting in (1, 2):
        outs = {m: _run_bwd(inp, w, setting, m, kl, l1, l2) for m in (skl.BWD_FUSED, skl.BWD_SEPARATE)}
        torch.cuda.synchronize()
        refs = U.map_heads(lambda b, h: U.oracle_head(inp, w, b, h, setting=setting)[1], heads)
        for (b, h), (rdq, rdk) in zip(heads, refs):
            for m, (dq, dk) in outs.items():
                U.assert_grad(U.np64(dq[b, h]), rdq, f"setting {setting} mode {m} dQ head {b},{h}")
                U.assert_grad(U.np64(dk[b, h]), rdk, f"setting {setting} mode {m} dK head {b},{h}")
        # fused = separate on every head (separate is deterministic and checked above)
        for which in (0, 1):
            f, s_ = outs[skl.BWD_FUSED][which].double(), outs[skl.BWD_SEPARATE][which].double()
            per_head = ((f - s_).norm(dim=(2, 3)) / s_.norm(dim=(2, 3))).max().item()
            assert per_head < 1e-2, ("dQ" if which == 0 else "dK", per_head)
        qo, ko = (q2, k2) if setting == 1 else (q1, k1)
        for m, (dq, dk) in outs.items():
            U.assert_dk_invariants(dk, ko, dq, qo, setting, f"setting {setting} mode {m}")


def test_b1h32_n65536_causal_setting1():
    """The long causal workload: 256 sampled rows (KL, LSE, dQ2); dK2 of the last 256 keys of 4 seeded heads
    against the oracle (only the last 256 query rows see them); the dK2 identities on every head."""
    w = W["kl_b1h32_n65536_d128_causal"]
    inp = synth.make_inputs(w)
    kl, l1, l2 = _run_fwd(inp, w)
    dq, dk = _run_bwd(inp, w, 1, skl.BWD_AUTO, kl, l1, l2)
    torch.cuda.synchronize()
    rows = synth.sample_rows(w, 256, 1000 + w.seed)
    rkl, rl1, rl2, rdq = U.oracle_rows(inp, w, rows, setting=1)
    b, h, i = rows[:, 0], rows[:, 1], rows[:, 2]
    U.assert_rows(U.np64(kl)[b, h, i], U.np64(l1)[b, h, i], U.np64(l2)[b, h, i], rkl, rl1, rl2)
    U.assert_grad(U.np64(dq)[b, h, i], rdq, "dQ2 sampled rows")
    R = 256
    rng = np.random.default_rng(3000 + w.seed)
    heads = [(0, int(x)) for x in sorted(rng.choice(w.H, size=4, replace=False))]
    refs = U.map_heads(lambda bb, hh: U.oracle_last_keys_dk(inp, w, bb, hh, 1, R), heads, threads=4)
    for (bb, hh), rdk in zip(heads, refs):
        U.assert_grad(U.np64(dk[bb, hh, -R:]), rdk, f"dK2 last {R} keys head {bb},{hh}")
    q1, k1, q2, k2 = U.dev_inputs(inp)
    U.assert_dk_invariants(dk, k2, dq, q2, 1, "dK2")


@pytest.mark.slow
def test_b1h32_n65536_causal_one_full_head_dk():
    """dK2 of one seeded head of the long causal workload against the full oracle."""
    w = W["kl_b1h32_n65536_d128_causal"]
    rng = np.random.default_rng(2000 + w.seed)
    b, h = 0, int(rng.integers(w.H))
    inp = synth.make_inputs(w)
    kl, l1, l2 = _run_fwd(inp, w)
    _, dk = _run_bwd(inp, w, 1, skl.BWD_AUTO, kl, l1, l2)
    dk_h = U.np64(dk[b, h])
    del kl, l1, l2, dk
    rdk = U.oracle_head_dk_parallel(inp, w, b, h, setting=1)
    U.assert_grad(dk_h, rdk, f"dK2 head {b},{h}")


@pytest.mark.parametrize("nq", [1, 4, 16])
def test_decode_splitk(nq):
    """Split-K decode: every row (N_Q 1, 4) or 256 sampled rows (16); split = non-split."""
    w = W[f"decode_b8h32_nq{nq}_nk131072_d128"]
    inp = synth.make_inputs(w)
    kl, l1, l2 = _run_fwd(inp, w, splitk=True)
    nkl, nl1, nl2 = _run_fwd(inp, w, splitk=False)
    torch.cuda.synchronize()
    if nq <= 4:
        rows = np.array([(b, h, i) for b in range(w.B) for h in range(w.H) for i in range(nq)])
    else:
        rows = synth.sample_rows(w, 256, 1000 + w.seed)
    rkl, rl1, rl2, _ = U.oracle_rows(inp, w, rows)
    b, h, i = rows[:, 0], rows[:, 1], rows[:, 2]
    U.assert_rows(U.np64(kl)[b, h, i], U.np64(l1)[b, h, i], U.np64(l2)[b, h, i], rkl, rl1, rl2, "splitk")
    U.assert_rows(U.np64(nkl)[b, h, i], U.np64(nl1)[b, h, i], U.np64(nl2)[b, h, i], rkl, rl1, rl2, "non-split")
    assert float((kl - nkl).abs().max()) < 1e-3
    assert float((l1 - nl1).abs().max()) < 1e-3


def test_b1h8_n524288_causal_setting2():
    """The 512K causal workload: fwd + setting 2, on the fused path over key ranges (what AUTO takes: one head's
    dK rows, 256 MiB, exceed L2) and on the separate path.  128 sampled rows (KL, LSE, dQ1); dK1 of the last 128
    keys of every head against the oracle (only the last 128 query rows see them; they lie in the last key
    range); sum_j dK_j = 0 and the trace identity on every head."""
    w = W["kl_b1h8_n524288_d128_causal"]
    inp = synth.make_inputs(w)
    kl, l1, l2 = _run_fwd(inp, w)
    props = torch.cuda.get_device_properties(0)
    assert skl.bwd_select(w.B, w.H, w.NQ, w.NK, w.D, props.L2_cache_size, props.multi_processor_count,
                          w.causal) == skl.BWD_FUSED
    ranges, _ = skl.bwd_fused_plan(w.B, w.H, w.NQ, w.NK, w.D, props.L2_cache_size, props.multi_processor_count,
                                   w.causal)
    assert ranges > 1
    rows = synth.sample_rows(w, 128, 1000 + w.seed)
    rkl, rl1, rl2, rdq = U.oracle_rows(inp, w, rows, setting=2)
    b, h, i = rows[:, 0], rows[:, 1], rows[:, 2]
    U.assert_rows(U.np64(kl)[b, h, i], U.np64(l1)[b, h, i], U.np64(l2)[b, h, i], rkl, rl1, rl2)
    R = 128
    heads = [(0, hh) for hh in range(w.H)]
    rdk = U.map_heads(lambda bb, hh: U.oracle_last_keys_dk(inp, w, bb, hh, 2, R), heads, threads=4)
    q1, k1, q2, k2 = U.dev_inputs(inp)
    for mode in (skl.BWD_AUTO, skl.BWD_SEPARATE):
        dq, dk = _run_bwd(inp, w, 2, mode, kl, l1, l2)
        torch.cuda.synchronize()
        U.assert_grad(U.np64(dq)[b, h, i], rdq, f"mode {mode}: dQ1 sampled rows")
        for (bb, hh), ref in zip(heads, rdk):
            U.assert_grad(U.np64(dk[bb, hh, -R:]), ref, f"mode {mode}: dK1 last {R} keys head {bb},{hh}")
        U.assert_dk_invariants(dk, k1, dq, q1, 2, f"mode {mode}")
        del dq, dk


def test_auto_takes_separate_kernels_for_short_queries_and_long_keys():
    """One query tile per head and keys whose live dK rows exceed L2: AUTO picks the separate kernels (the
    measured rule); both settings against the oracle on four seeded heads."""
    w = synth.Workload("auto_sep", 1, 32, 128, 65536, 128, False, 0.5, 31)
    props = torch.cuda.get_device_properties(0)
    assert skl.bwd_select(w.B, w.H, w.NQ, w.NK, w.D, props.L2_cache_size, props.multi_processor_count,
                          w.causal) == skl.BWD_SEPARATE
    assert skl.bwd_workspace_bytes(w.B, w.H, w.NQ, w.NK, w.D, skl.BWD_AUTO, w.causal) == 0
    inp = synth.make_inputs(w)
    kl, l1, l2 = _run_fwd(inp, w)
    rng = np.random.default_rng(4000 + w.seed)
    heads = [(0, int(x)) for x in sorted(rng.choice(w.H, size=4, replace=False))]
    for setting in (1, 2):
        dq, dk = _run_bwd(inp, w, setting, skl.BWD_AUTO, kl, l1, l2)
        torch.cuda.synchronize()
        refs = U.map_heads(lambda b, h: U.oracle_head(inp, w, b, h, setting=setting), heads, threads=4)
        for (b, h), ((rkl, rl1, rl2), (rdq, rdk)) in zip(heads, refs):
            U.assert_rows(U.np64(kl[b, h]), U.np64(l1[b, h]), U.np64(l2[b, h]), rkl, rl1, rl2, f"head {b},{h}")
            U.assert_grad(U.np64(dq[b, h]), rdq, f"setting {setting} dQ head {b},{h}")
            U.assert_grad(U.np64(dk[b, h]), rdk, f"setting {setting} dK head {b},{h}")


# ------------------------------------------------------------------ edge cases

@pytest.mark.parametrize("causal", [False, True])
def test_logits_growing_past_the_first_tile(causal):
    """Keys after the first tile scaled by 30: the row maxima jump by far more than 2^64 (log2 units) after the
    first tile, so the forward's tiles that reuse the running maxima must detect it and redo the tile against
    its own maximum."""
    w = synth.Workload("growth", 1, 2, 256, 512, 64, causal, 0.5, 21)
    inp = synth.make_inputs(w)
    for k in ("k1", "k2"):
        f = U.f64(inp[k])
        f[:, :, 128:] *= 30.0
        inp[k] = synth.f32_to_bf16_bits(f.astype(np.float32))
    Q1, K1, Q2, K2 = (U.f64(inp[k]) for k in ("q1", "k1", "q2", "k2"))
    rkl, rl1, rl2 = O.forward(Q1, K1, Q2, K2, w.softmax_scale, causal)
    assert (rl1[:, :, 200:] * np.log2(np.e) - 64).max() > 0  # the late rows' maxima are far above the first tile's
    kl, l1, l2 = _run_fwd(inp, w)
    U.assert_rows(U.np64(kl), U.np64(l1), U.np64(l2), rkl, rl1, rl2, "growth fwd")


@pytest.mark.parametrize("causal", [False, True])
def test_upstream_gradient_of_mixed_sign(causal):
    """g of either sign and zero rows: the fused path folds a positive g into its exponents and multiplies by
    any other g; both settings and both paths against the oracle."""
    w = synth.Workload("gsign", 2, 2, 300, 300, 128, causal, 0.5, 23)
    inp = synth.make_inputs(w)
    g = (np.random.default_rng(5).standard_normal((2, 2, 300)) / 300).astype(np.float32)
    g[:, :, ::7] = 0.0
    inp["g"] = g
    kl, l1, l2 = _run_fwd(inp, w)
    Q1, K1, Q2, K2 = (U.f64(inp[k]) for k in ("q1", "k1", "q2", "k2"))
    for setting in (1, 2):
        rdq, rdk = O.backward(setting, Q1, K1, Q2, K2, w.softmax_scale, causal, g)
        for mode in (skl.BWD_FUSED, skl.BWD_SEPARATE):
            dq, dk = _run_bwd(inp, w, setting, mode, kl, l1, l2)
            U.assert_grad(U.np64(dq), rdq, f"setting {setting} mode {mode} dQ")
            U.assert_grad(U.np64(dk), rdk, f"setting {setting} mode {mode} dK")


def test_identical_pairs_give_exact_zero():
    w = synth.Workload("same", 1, 2, 200, 200, 128, True, 0.5, 7)
    inp = synth.make_inputs(w)
    inp["q2"], inp["k2"] = inp["q1"], inp["k1"]
    kl, l1, l2 = _run_fwd(inp, w)
    assert float(kl.abs().max()) == 0.0
    assert torch.equal(l1, l2)
    for setting in (1, 2):
        for mode in (skl.BWD_FUSED, skl.BWD_SEPARATE):
            dq, dk = _run_bwd(inp, w, setting, mode, kl, l1, l2)
            assert float(dq.float().abs().max()) == 0.0 and float(dk.float().abs().max()) == 0.0


def test_empty_query_rows():
    w = synth.Workload("empty", 1, 2, 0, 64, 64, False, 0.5, 8)
    inp = synth.make_inputs(w)
    kl, l1, l2 = _run_fwd(inp, w)
    assert kl.numel() == 0
    q1, k1, q2, k2 = U.dev_inputs(inp)
    g = torch.zeros((1, 2, 0), device="cuda")
    dq, dk = skl.bwd_s1(q1, k1, q2, k2, l1, l2, g, None, False, skl.BWD_SEPARATE)
    assert dq.numel() == 0 and float(dk.float().abs().max()) == 0.0


def test_host_buffers_round_trip():
    """CPU tensors in, CPU tensors out: same numbers as the device call."""
    w = synth.Workload("host", 1, 2, 96, 160, 128, True, 0.5, 9)
    inp = synth.make_inputs(w)
    d = _run_fwd(inp, w)
    hq = [torch.from_numpy(inp[k].view(np.int16)).view(torch.bfloat16).pin_memory() for k in ("q1", "k1", "q2", "k2")]
    h = skl.fwd(*hq, w.softmax_scale, w.causal)
    assert all(x.device.type == "cpu" for x in h)
    for a, b in zip(d, h):
        assert torch.equal(a.cpu(), b)


def test_workspace_too_small_is_refused():
    w = synth.Workload("ws", 1, 1, 8, 640, 128, False, 0.5, 10)
    inp = synth.make_inputs(w)
    q1, k1, q2, k2 = U.dev_inputs(inp)
    import ctypes
    s = skl.make_shape(1, 1, 8, 640, 128)
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    out = [torch.empty(8, device="cuda") for _ in range(3)]
    st = skl.lib().streamkl_fwd_splitk(*(ctypes.c_void_p(t.data_ptr()) for t in (q1, k1, q2, k2)), s, 4,
                                       ctypes.c_void_p(ws.data_ptr()), 16,
                                       *(ctypes.c_void_p(t.data_ptr()) for t in out), None)
    assert st == skl._lib.ERR_WORKSPACE


def test_fused_workspace_too_small_is_refused():
    w = synth.Workload("ws", 1, 2, 100, 300, 64, True, 0.5, 11)
    inp = synth.make_inputs(w)
    q1, k1, q2, k2 = U.dev_inputs(inp)
    import ctypes
    s = skl.make_shape(1, 2, 100, 300, 64, w.softmax_scale, True)
    need = skl.bwd_workspace_bytes(1, 2, 100, 300, 64, skl.BWD_FUSED, True)
    assert need == 2 * 300 * 64 * 4
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    rows = [torch.zeros((1, 2, 100), device="cuda") for _ in range(3)]
    dq, dk = torch.empty_like(q2), torch.empty_like(k2)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = skl.lib().streamkl_bwd_s1(*(ptr(t) for t in (q1, k1, q2, k2)), s, *(ptr(t) for t in rows), ptr(dq), ptr(dk),
                                   skl.BWD_FUSED, ptr(ws), need - 1, None)
    assert st == skl._lib.ERR_WORKSPACE


def test_device_wait_timeout_is_reported_and_context_survives():
    assert skl.check_device_status() == skl._lib.OK
    assert skl.debug_wait_timeout(2000) == skl._lib.OK
    assert skl.check_device_status() == skl._lib.ERR_TIMEOUT
    assert skl.check_device_status() == skl._lib.OK  # cleared by the read
    # the context still works
    w = synth.Workload("after", 1, 1, 64, 64, 64, False, 0.5, 11)
    inp = synth.make_inputs(w)
    kl, l1, l2 = _run_fwd(inp, w)
    (rkl, rl1, rl2), _ = U.oracle_head(inp, w, 0, 0)
    U.assert_rows(U.np64(kl)[0, 0], U.np64(l1)[0, 0], U.np64(l2)[0, 0], rkl, rl1, rl2)
