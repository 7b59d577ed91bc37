"""Key shards on one GPU: the kernels behind shard.py's context-parallel path.

The keys are cut into contiguous shards (tile-aligned and not), each shard's
five-scalar partials come from streamkl_fwd_partials, and
streamkl_merge_partials merges them (in place of an all-gather): KL and LSE
must equal the one-pass forward's and the oracle's.  The backward runs
streamkl_bwd_keyshard per shard with the merged LSE/KL; the shards' unscaled dQ
contributions are summed (in place of an all-reduce) and converted by
streamkl_dq_from_partial; dQ and the concatenated dK are compared with the
oracle in both settings.
"""
import numpy as np
import pytest
import torch

import attention_kl_divergence_streamkl_gb300 as skl
from attention_kl_divergence_streamkl_gb300 import build, synth
from oracle import oracle as O
from tests import parity_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    skl.lib()
    yield
    assert skl.check_device_status() == skl._lib.OK, "a device-side wait timed out during this module"


CASES = [
    # B, H, NQ, NK, D, causal, cut points inside (0, NK)
    (1, 2, 300, 300, 128, True, (128, 256)),
    (1, 2, 300, 300, 128, True, (100, 171)),
    (2, 2, 257, 700, 64, False, (256, 512)),
    (1, 3, 200, 530, 128, True, (200, 385)),
    (2, 2, 5, 900, 128, True, (128, 333, 640)),
    (1, 2, 130, 130, 64, True, (129,)),
]


def _ids(c):
    return "b{}h{}q{}k{}d{}{}_cuts{}".format(*c[:5], "c" if c[5] else "", "-".join(map(str, c[6])))


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_key_shards_match_oracle(case):
    B, H, NQ, NK, D, causal, cuts = case
    w = synth.Workload("keyshard", B, H, NQ, NK, D, causal, 0.5, 500 + NQ + NK)
    inp = synth.make_inputs(w)
    q1, k1, q2, k2 = U.dev_inputs(inp)
    g = torch.from_numpy(inp["g"]).cuda()
    sc = w.softmax_scale
    bounds = [0, *cuts, NK]
    shards = list(zip(bounds[:-1], bounds[1:]))
    parts = torch.stack([skl.fwd_partials(q1, k1[:, :, a:b], q2, k2[:, :, a:b], a, NK, sc, causal)
                         for a, b in shards])
    kl, l1, l2 = skl.merge_partials(parts, D, sc)
    fkl, fl1, fl2 = skl.fwd(q1, k1, q2, k2, sc, causal)
    torch.cuda.synchronize()
    # same arithmetic in another order: equal to the one-pass forward well inside the oracle tolerance
    assert float((kl - fkl).abs().max()) < 2e-4 and float((l1 - fl1).abs().max()) < 2e-5
    Q1, K1, Q2, K2 = (U.f64(inp[k]) for k in ("q1", "k1", "q2", "k2"))
    rkl, rl1, rl2 = O.forward(Q1, K1, Q2, K2, sc, causal)
    U.assert_rows(U.np64(kl), U.np64(l1), U.np64(l2), rkl, rl1, rl2, "merged shards")
    for setting in (1, 2):
        rdq, rdk = O.backward(setting, Q1, K1, Q2, K2, sc, causal, inp["g"])
        dq_sum = None
        dks = []
        for a, b in shards:
            dqp, dk = skl.bwd_keyshard(setting, q1, k1[:, :, a:b], q2, k2[:, :, a:b], a, NK, l1, l2, kl, g, sc,
                                       causal)
            dq_sum = dqp if dq_sum is None else dq_sum + dqp
            dks.append(dk)
        dq = skl.dq_from_partial(dq_sum, q2 if setting == 1 else q1, sc)
        dk = torch.cat(dks, dim=2)
        torch.cuda.synchronize()
        U.assert_grad(U.np64(dq), rdq, f"setting {setting} dQ from shards")
        U.assert_grad(U.np64(dk), rdk, f"setting {setting} dK from shards")


def test_shard_seen_by_no_row_of_a_tile():
    """A causal shard far past some query tiles' frontier: those rows' partials are empty and merge as nothing."""
    w = synth.Workload("keyshard_far", 1, 1, 256, 256, 64, True, 0.5, 77)
    inp = synth.make_inputs(w)
    q1, k1, q2, k2 = U.dev_inputs(inp)
    part = skl.fwd_partials(q1, k1[:, :, 200:], q2, k2[:, :, 200:], 200, 256, w.softmax_scale, True)
    torch.cuda.synchronize()
    p = U.np64(part)[0, 0]
    assert np.all(np.isneginf(p[:200, :2])) and np.all(p[:200, 2:] == 0)
    assert np.all(np.isfinite(p[200:])) and np.all(p[200:, 2] > 0)


def test_invalid_shard_arguments_are_refused():
    w = synth.Workload("keyshard_bad", 1, 1, 64, 128, 64, True, 0.5, 78)
    inp = synth.make_inputs(w)
    q1, k1, q2, k2 = U.dev_inputs(inp)
    with pytest.raises(skl.StreamKLError):
        skl.fwd_partials(q1, k1[:, :, 64:], q2, k2[:, :, 64:], 100, 128)  # offset + shard past the sequence
    with pytest.raises(skl.StreamKLError):
        skl.fwd_partials(q1, k1, q2, k2, -1, 128)
    with pytest.raises(skl.StreamKLError):
        skl.fwd_partials(q1, k1[:, :, :32], q2, k2[:, :, :32], 0, 32, None, True)  # causal with N_Q > nk_total


def test_shard_module_on_one_gpu():
    """shard.py's head and key paths with a world of one (no process group): the library's kernels behind
    every call, against the unsharded calls."""
    from attention_kl_divergence_streamkl_gb300 import shard
    w = synth.Workload("shardmod", 1, 4, 256, 640, 128, True, 0.5, 91)
    inp = synth.make_inputs(w)
    q1, k1, q2, k2 = U.dev_inputs(inp)
    g = torch.from_numpy(inp["g"]).cuda()
    sc = w.softmax_scale
    kl, l1, l2 = skl.fwd(q1, k1, q2, k2, sc, True)
    hkl, hl1, hl2, loss = shard.heads_forward(q1, k1, q2, k2, sc, True, g)
    assert torch.equal(hkl, kl) and abs(float(loss) - float((g.double() * kl.double()).sum())) < 1e-9
    k1l, k0 = shard.local_keys(k1)
    k2l, _ = shard.local_keys(k2)
    assert (k0, k1l.shape[2]) == (0, w.NK)
    skl_, sl1, sl2 = shard.keys_forward(q1, k1l, q2, k2l, k0, w.NK, sc, True)
    assert float((skl_ - kl).abs().max()) < 2e-4 and float((sl1 - l1).abs().max()) < 2e-5
    for setting in (1, 2):
        dq, dk = shard.keys_backward(setting, q1, k1l, q2, k2l, k0, w.NK, sl1, sl2, skl_, g, sc, True)
        rq, rk = (skl.bwd_s1(q1, k1, q2, k2, l1, l2, g, sc, True, skl.BWD_FUSED) if setting == 1 else
                  skl.bwd_s2(q1, k1, q2, k2, l1, l2, kl, g, sc, True, skl.BWD_FUSED))
        U.assert_grad(U.np64(dq), U.np64(rq), f"setting {setting} dQ via shard.py")
        U.assert_grad(U.np64(dk), U.np64(rk), f"setting {setting} dK via shard.py")


def test_key_sharded_autograd_on_one_gpu():
    """keys_attention_kl with a world of one equals attention_kl: values and the gradients of all four inputs."""
    from attention_kl_divergence_streamkl_gb300 import shard
    w = synth.Workload("shardgrad", 1, 2, 200, 384, 64, True, 0.5, 92)
    inp = synth.make_inputs(w)
    base = U.dev_inputs(inp)
    a = [t.clone().requires_grad_() for t in base]
    b = [t.clone().requires_grad_() for t in base]
    la = skl.attention_kl(*a, w.softmax_scale, True, "mean")
    la.backward()
    kl = shard.keys_attention_kl(*b, 0, w.NK, w.softmax_scale, True)
    lb = kl.mean()
    lb.backward()
    assert abs(float(la) - float(lb)) < 1e-5
    for x, y, name in zip(a, b, ("q1", "k1", "q2", "k2")):
        U.assert_grad(U.np64(y.grad), U.np64(x.grad), f"{name} grad via keys_attention_kl")
