"""The multi-GPU partitions of shard.py on CPU: ranges, and two gloo ranks that
shard heads and keys, checked against the fp64 oracle on the whole problem.

The ranks compute with tests/shard_cpu_ops.py (the oracle's functions) in
place of the GPU kernels, so what is tested is the partition, the exchange
(all-reduce, all-gather) and the merge of the five-scalar partials; the
kernels behind the same calls are checked on one GPU in test_gpu_keyshard.py.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from attention_kl_divergence_streamkl_gb300 import shard, synth


@pytest.mark.parametrize("n,parts,align", [(1000, 3, 128), (65536, 8, 128), (100, 4, 128), (7, 2, 1), (70, 2, 16),
                                           (0, 3, 1)])
def test_split_range_covers_in_order(n, parts, align):
    rs = [shard.split_range(n, parts, r, align) for r in range(parts)]
    assert rs[0][0] == 0 and rs[-1][1] == n
    for (a, b), (c, d) in zip(rs, rs[1:]):
        assert b == c and a <= b
    for lo, hi in rs[:-1]:
        assert lo % align == 0 and hi % align == 0
    sizes = [-(-(hi - lo) // align) for lo, hi in rs]
    assert max(sizes) - min(sizes) <= 1


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(causal):
    w = synth.Workload("shard", 2, 3, 40, 70, 8, causal, 0.5, 41)
    inp = synth.make_inputs(w)
    ts = {k: torch.from_numpy(synth.bf16_bits_to_f64(inp[k])) for k in ("q1", "k1", "q2", "k2")}
    g = torch.from_numpy(np.random.default_rng(3).uniform(0.5, 1.5, (w.B, w.H, w.NQ)))
    return w, ts, g


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from tests.shard_cpu_ops import OPS
    res = {}
    for causal in (False, True):
        w, t, g = _inputs(causal)
        sc = w.softmax_scale
        # ---- heads: the loss is all-reduced, gradients stay local
        loc = {k: shard.local_heads(v) for k, v in t.items()}
        gl = shard.local_heads(g)
        kl, l1, l2, loss = shard.heads_forward(loc["q1"], loc["k1"], loc["q2"], loc["k2"], sc, causal, gl, ops=OPS)
        grads = {}
        for setting in (1, 2):
            dq, dk = shard.heads_backward(setting, loc["q1"], loc["k1"], loc["q2"], loc["k2"], l1, l2, kl, gl, sc,
                                          causal, ops=OPS)
            grads[setting] = (dq, dk)
        res[("heads", causal)] = (shard.head_range(w.H), kl, float(loss), grads)
        # ---- keys: partials all-gathered and merged; dQ all-reduced; dK local
        k1l, k0 = shard.local_keys(t["k1"], align=16)
        k2l, _ = shard.local_keys(t["k2"], align=16)
        kl, l1, l2 = shard.keys_forward(t["q1"], k1l, t["q2"], k2l, k0, w.NK, sc, causal, ops=OPS)
        grads = {}
        for setting in (1, 2):
            grads[setting] = shard.keys_backward(setting, t["q1"], k1l, t["q2"], k2l, k0, w.NK, l1, l2, kl, g, sc,
                                                 causal, ops=OPS)
        res[("keys", causal)] = ((k0, k0 + k1l.shape[2]), (kl, l1, l2), grads)
        # ---- the differentiable form: mean KL over all rows, gradients of every input
        ins = [t["q1"].clone().requires_grad_(), k1l.clone().requires_grad_(), t["q2"].clone().requires_grad_(),
               k2l.clone().requires_grad_()]
        kl = shard.keys_attention_kl(*ins, k0, w.NK, sc, causal, ops=OPS)
        kl.mean().backward()
        res[("autograd", causal)] = (float(kl.mean()), [x.grad.clone() for x in ins])
    out[rank] = res
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_heads_and_keys():
    from oracle import oracle as O
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    for causal in (False, True):
        w, t, g = _inputs(causal)
        sc = w.softmax_scale
        f = {k: v.numpy() for k, v in t.items()}
        rkl, rl1, rl2 = O.forward(f["q1"], f["k1"], f["q2"], f["k2"], sc, causal)
        ref = {s: O.backward(s, f["q1"], f["k1"], f["q2"], f["k2"], sc, causal, g.numpy()) for s in (1, 2)}
        # heads: every rank's loss is the whole job's sum of g KL; local values and grads are the owner's heads
        heads_seen = []
        for r in range(world):
            (h0, h1), kl, loss, grads = out[r][("heads", causal)]
            heads_seen.append((h0, h1))
            assert loss == pytest.approx(float((g.numpy() * rkl).sum()), rel=1e-12)
            assert np.allclose(kl.numpy(), rkl[:, h0:h1], atol=1e-12)
            for s in (1, 2):
                assert np.allclose(grads[s][0].numpy(), ref[s][0][:, h0:h1], atol=1e-12)
                assert np.allclose(grads[s][1].numpy(), ref[s][1][:, h0:h1], atol=1e-12)
        assert heads_seen == [(0, 1), (1, 3)]
        # keys: merged KL/LSE and dQ on every rank; dK of the owned keys
        ranges = []
        for r in range(world):
            (k0, k1), (kl, l1, l2), grads = out[r][("keys", causal)]
            ranges.append((k0, k1))
            assert np.allclose(kl.numpy(), rkl, atol=1e-12) and np.allclose(l1.numpy(), rl1, atol=1e-12)
            assert np.allclose(l2.numpy(), rl2, atol=1e-12)
            for s in (1, 2):
                dq, dk = grads[s]
                assert np.allclose(dq.numpy(), ref[s][0], atol=1e-12)
                assert np.allclose(dk.numpy(), ref[s][1][:, :, k0:k1], atol=1e-12)
        assert ranges == [(0, 32), (32, 70)]
        # autograd: g = 1 / (B H N_Q) per row; setting 2 gives the teacher's, setting 1 the student's gradients
        gm = np.full((w.B, w.H, w.NQ), 1.0 / (w.B * w.H * w.NQ))
        r1 = O.backward(1, f["q1"], f["k1"], f["q2"], f["k2"], sc, causal, gm)
        r2 = O.backward(2, f["q1"], f["k1"], f["q2"], f["k2"], sc, causal, gm)
        for r, (k0, k1) in enumerate(ranges):
            loss, (gq1, gk1, gq2, gk2) = out[r][("autograd", causal)]
            assert loss == pytest.approx(float(rkl.mean()), rel=1e-12)
            assert np.allclose(gq1.numpy(), r2[0], atol=1e-12) and np.allclose(gq2.numpy(), r1[0], atol=1e-12)
            assert np.allclose(gk1.numpy(), r2[1][:, :, k0:k1], atol=1e-12)
            assert np.allclose(gk2.numpy(), r1[1][:, :, k0:k1], atol=1e-12)


def test_a_rank_without_heads_calls_no_kernel():
    """More ranks than heads leaves a rank an empty head range; it returns empty
    values and gradients without calling the kernels (which refuse H = 0)."""
    import types

    def refuse(*a, **k):
        raise AssertionError("kernel called for an empty head range")

    ops = types.SimpleNamespace(fwd=refuse, bwd_s1=refuse, bwd_s2=refuse)
    assert shard.split_range(1, 2, 0) == (0, 0)
    q = torch.zeros((2, 0, 5, 8))
    k = torch.zeros((2, 0, 7, 8))
    kl, l1, l2, loss = shard.heads_forward(q, k, q, k, 0.5, False, ops=ops)
    assert kl.shape == (2, 0, 5) and l1.shape == (2, 0, 5) and float(loss) == 0.0
    for setting in (1, 2):
        dq, dk = shard.heads_backward(setting, q, k, q, k, l1, l2, kl, kl, 0.5, False, ops=ops)
        assert dq.shape == q.shape and dk.shape == k.shape
