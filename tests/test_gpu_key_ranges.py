"""GPU parity of the fused backward run over key ranges (one launch per range,
dQ summed over the ranges in fp32), forced onto small shapes through the
STREAMKL_FUSED_KEY_TILES override and compared with the fp64 oracle.  The full
512K workload, where the ranges are the automatic choice, is covered in
test_gpu_parity."""
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


CASES = [
    # B, H, NQ, NK, D, causal, key tiles per range
    (2, 3, 300, 300, 128, True, 1),
    (2, 3, 300, 300, 128, True, 2),
    (1, 2, 77, 333, 64, False, 1),
    (1, 2, 260, 1000, 128, True, 3),
    (2, 1, 130, 513, 64, True, 2),
]


def bnhd(t):
    return t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)


@pytest.mark.parametrize("layout", ["contiguous", "bnhd"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}h{}q{}k{}d{}{}_t{}".format(*c[:5], "c" if c[5] else "", c[6]))
def test_fused_over_key_ranges_matches_oracle(case, layout, monkeypatch):
    B, H, NQ, NK, D, causal, tiles = case
    w = synth.Workload("ranges", B, H, NQ, NK, D, causal, 0.5, 300 + NQ + NK + tiles)
    inp = synth.make_inputs(w)
    ins = U.dev_inputs(inp)
    if layout == "bnhd":
        ins = [bnhd(t) for t in ins]
    q1, k1, q2, k2 = ins
    kl, l1, l2 = skl.fwd(q1, k1, q2, k2, w.softmax_scale, causal)
    g = torch.from_numpy(inp["g"]).cuda()
    monkeypatch.setenv("STREAMKL_FUSED_KEY_TILES", str(tiles))
    n_kt = -(-NK // 128)
    ranges = -(-n_kt // tiles)
    assert ranges > 1 or n_kt == 1
    want_ws = B * H * min(tiles * 128, NK) * D * 4 + (B * H * NQ * D * 4 if ranges > 1 else 0)
    assert skl.bwd_workspace_bytes(B, H, NQ, NK, D, skl.BWD_FUSED, causal) == want_ws
    Q1, K1, Q2, K2 = (U.f64(inp[k]) for k in ("q1", "k1", "q2", "k2"))
    for setting in (1, 2):
        rdq, rdk = O.backward(setting, Q1, K1, Q2, K2, w.softmax_scale, causal, inp["g"])
        if setting == 1:
            dq, dk = skl.bwd_s1(q1, k1, q2, k2, l1, l2, g, w.softmax_scale, causal, skl.BWD_FUSED)
        else:
            dq, dk = skl.bwd_s2(q1, k1, q2, k2, l1, l2, kl, g, w.softmax_scale, causal, skl.BWD_FUSED)
        U.assert_grad(U.np64(dq), rdq, f"{layout} t{tiles} setting {setting} dQ")
        U.assert_grad(U.np64(dk), rdk, f"{layout} t{tiles} setting {setting} dK")
