"""Seeded input generator: bf16 rounding, determinism, per-head rebuild."""
import numpy as np
import torch

from attention_kl_divergence_streamkl_gb300 import synth


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10.0 ** rng.integers(-6, 6, 100000),
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 65504.0, -3.0e38], np.float32)])
    ours = synth.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = synth.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_generator_deterministic_and_headwise():
    w = synth.WORKLOADS["kl_b1h1_n128_d64"].with_(B=2, H=3, NQ=40, NK=56)
    a = synth.make_inputs(w, threads=1)
    b = synth.make_inputs(w, threads=4)
    for k in ("q1", "k1", "q2", "k2"):
        assert np.array_equal(a[k], b[k])
        for bb in range(w.B):
            for hh in range(w.H):
                assert np.array_equal(a[k][bb, hh], synth.head_slice(w, k, bb, hh))
    # student is the teacher plus noise of the stated size
    d = synth.bf16_bits_to_f64(a["q2"]) - synth.bf16_bits_to_f64(a["q1"])
    assert 0.25 < d.std() < 0.35  # sigma 0.3 on this workload
    assert abs(synth.bf16_bits_to_f64(a["k1"]).std() - 1.0) < 0.05
    assert np.allclose(a["g"], 1.0 / w.NQ)


def test_pair_counts_and_samples():
    assert synth.count_pairs(4096, 4096, True) == 4096 * 4097 // 2
    assert synth.count_pairs(65536, 65536, True) == 65536 * 65537 // 2
    assert synth.count_pairs(5, 9, True) == sum(min(9, i + 4 + 1) for i in range(5))
    w = synth.WORKLOADS["kl_b1h32_n65536_d128_causal"]
    rows = synth.sample_rows(w, 256, 1003)
    assert rows.shape == (256, 3)
    assert len({tuple(r) for r in rows}) == 256
    for i in (0, 1, 127, 128, 65535):
        assert i in set(rows[:, 2].tolist())


def test_head_rows_is_a_prefix_of_the_head():
    w = synth.WORKLOADS["kl_b1h1_n128_d64"].with_(B=2, H=2, NQ=50, NK=70)
    for k in ("q1", "k1", "q2", "k2"):
        full = synth.head_slice(w, k, 1, 1)
        assert np.array_equal(synth.head_rows(w, k, 1, 1, 17), full[:17])
