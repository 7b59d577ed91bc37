"""The C-ABI library: it loads, exports what include/streamkl.h declares, and its
host-side rules (validation, Split-K planning, backward path choice, workspace
sizes) behave as documented.  Nothing here launches a kernel."""
import ctypes
import os
import re

import pytest

from attention_kl_divergence_streamkl_gb300 import _lib as K
from attention_kl_divergence_streamkl_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "streamkl.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return K.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(streamkl_\w+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(K.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.streamkl_version() >= 100


def test_status_strings(lib):
    for code in range(6):
        assert K.status_string(code)
    assert "timed out" in K.status_string(K.ERR_TIMEOUT)


def fake_ptr(off=0):
    return ctypes.c_void_p(0x10000000 + off)


def call_fwd(lib, shape, q=None, kl=None):
    q = q or fake_ptr()
    kl = kl or fake_ptr(4096)
    return lib.streamkl_fwd(q, fake_ptr(64), fake_ptr(128), fake_ptr(192), shape, kl, fake_ptr(8192),
                            fake_ptr(12288), None)


@pytest.mark.parametrize("shape,code", [
    (dict(B=0, H=1, NQ=8, NK=8, D=64), K.ERR_INVALID),
    (dict(B=1, H=0, NQ=8, NK=8, D=64), K.ERR_INVALID),
    (dict(B=1, H=1, NQ=-1, NK=8, D=64), K.ERR_INVALID),
    (dict(B=1, H=1, NQ=8, NK=0, D=64), K.ERR_INVALID),
    (dict(B=1, H=1, NQ=8, NK=8, D=96), K.ERR_UNSUPPORTED),
    (dict(B=1, H=1, NQ=8, NK=8, D=256), K.ERR_UNSUPPORTED),
    (dict(B=1, H=1, NQ=9, NK=8, D=64, causal=True), K.ERR_INVALID),
    (dict(B=1, H=1, NQ=8, NK=8, D=64, scale=float("nan")), K.ERR_INVALID),
    (dict(B=1, H=1, NQ=8, NK=8, D=64, scale=float("inf")), K.ERR_INVALID),
    (dict(B=1, H=1, NQ=8, NK=2**31 - 1, D=64), K.ERR_UNSUPPORTED),
    (dict(B=65536, H=65536, NQ=8, NK=8, D=64), K.ERR_UNSUPPORTED),
    # B*H fits, but (query tiles + key tiles) x B*H blocks would not fit a grid
    (dict(B=1 << 15, H=1 << 15, NQ=256, NK=256, D=64), K.ERR_UNSUPPORTED),
    (dict(B=1, H=1 << 21, NQ=65536, NK=65536, D=64), K.ERR_UNSUPPORTED),
])
def test_fwd_rejects_bad_shapes_before_launch(lib, shape, code):
    assert call_fwd(lib, K.make_shape(**shape)) == code


def test_fwd_rejects_null_and_misaligned_pointers(lib):
    s = K.make_shape(1, 1, 8, 8, 64)
    assert lib.streamkl_fwd(None, fake_ptr(), fake_ptr(), fake_ptr(), s, fake_ptr(), fake_ptr(), fake_ptr(),
                            None) == K.ERR_INVALID
    assert call_fwd(lib, s, q=fake_ptr(8)) == K.ERR_INVALID  # Q not 16-byte aligned
    assert call_fwd(lib, s, kl=fake_ptr(2)) == K.ERR_INVALID  # fp32 output not 4-byte aligned


def test_empty_query_set_is_a_no_op(lib):
    # N_Q = 0: nothing to compute, no pointer is touched
    s = K.make_shape(2, 3, 0, 16, 128)
    assert lib.streamkl_fwd(None, None, None, None, s, None, None, None, None) == K.OK


def test_bwd_rejects_bad_mode_and_pointers(lib):
    s = K.make_shape(1, 1, 8, 8, 64)
    p = [fake_ptr(64 * i) for i in range(12)]
    assert lib.streamkl_bwd_s1(p[0], p[1], p[2], p[3], s, p[4], p[5], p[6], p[7], p[8], 7, None, 0,
                               None) == K.ERR_INVALID
    assert lib.streamkl_bwd_s2(p[0], p[1], p[2], p[3], s, p[4], p[5], None, p[6], p[7], p[8], K.BWD_SEPARATE,
                               None, 0, None) == K.ERR_INVALID  # setting 2 needs the saved KL
    assert lib.streamkl_bwd_s1(p[0], p[1], p[2], p[3], s, p[4], p[5], p[6], p[7], fake_ptr(2), K.BWD_SEPARATE,
                               None, 0, None) == K.ERR_INVALID  # dK misaligned
    # fused without (enough) workspace is refused before any launch
    assert lib.streamkl_bwd_s1(p[0], p[1], p[2], p[3], s, p[4], p[5], p[6], p[7], p[8], K.BWD_FUSED, None, 0,
                               None) == K.ERR_WORKSPACE
    assert lib.streamkl_bwd_s1(p[0], p[1], p[2], p[3], s, p[4], p[5], p[6], p[7], p[8], K.BWD_FUSED, fake_ptr(8),
                               1 << 20, None) == K.ERR_WORKSPACE  # misaligned workspace


def test_workspace_sizes(lib):
    n = ctypes.c_size_t()
    s = K.make_shape(8, 32, 4, 131072, 128)
    assert lib.streamkl_fwd_splitk_workspace(s, 19, ctypes.byref(n)) == K.OK
    assert n.value == 8 * 32 * 4 * 19 * 5 * 4
    s16 = K.make_shape(8, 32, 17, 131072, 128)
    assert lib.streamkl_fwd_splitk_workspace(s16, 19, ctypes.byref(n)) == K.ERR_UNSUPPORTED
    s = K.make_shape(2, 32, 4096, 8192, 128)
    assert lib.streamkl_bwd_workspace(s, K.BWD_SEPARATE, ctypes.byref(n)) == K.OK
    assert n.value == 0
    for mode in (K.BWD_DQ_ONLY, K.BWD_DK_ONLY):
        assert lib.streamkl_bwd_workspace(s, mode, ctypes.byref(n)) == K.OK
        assert n.value == 0
    assert lib.streamkl_bwd_workspace(s, 5, ctypes.byref(n)) == K.ERR_INVALID


def test_splitk_workspace_rejects_bad_split_counts(lib):
    p = [fake_ptr(64 * i) for i in range(8)]
    s = K.make_shape(1, 2, 3, 1000, 64)
    assert lib.streamkl_fwd_splitk(p[0], p[1], p[2], p[3], s, -1, p[4], 1 << 20, p[5], p[6], p[7],
                                   None) == K.ERR_INVALID
    assert lib.streamkl_fwd_splitk(p[0], p[1], p[2], p[3], s, 4, p[4], 2 * 3 * 4 * 20 - 1, p[5], p[6], p[7],
                                   None) == K.ERR_WORKSPACE
    assert lib.streamkl_fwd_splitk(p[0], p[1], p[2], p[3], s, 4, fake_ptr(8), 1 << 20, p[5], p[6], p[7],
                                   None) == K.ERR_WORKSPACE  # misaligned workspace


def _cost(bh, tiles, sms, s):
    slots = sms * 2
    waves = -(-bh * s // slots)
    return waves * (-(-tiles // s) + 2)


@pytest.mark.parametrize("bh,nk,sms", [(256, 131072, 152), (32, 4096, 152), (1, 100, 152), (7, 65536, 132),
                                       (1024, 64, 152)])
def test_splitk_plan_minimises_the_wave_model(lib, bh, nk, sms):
    s = K.splitk_plan(1, bh, 4, nk, 128, num_sms=sms)
    tiles = -(-nk // 64)
    assert 1 <= s <= tiles
    best = min(_cost(bh, tiles, sms, x) for x in range(1, min(tiles, 4096) + 1))
    assert _cost(bh, tiles, sms, s) == best
    ideal = bh * tiles / (sms * 2)
    if ideal >= 100:
        # with many tiles per slot the chosen split keeps the SMs >90% busy under the model
        assert ideal / _cost(bh, tiles, sms, s) > 0.9


def _live_rows_bytes(B, H, NQ, NK, D, sms):
    query_tiles = -(-NQ // 128)
    heads = min(B * H, -(-sms // query_tiles) + 1)
    return NK * D * 4 * heads


def _first_qtile(NQ, NK, k0, causal):
    need = k0 - (NK - NQ)
    return 0 if (not causal or need <= 0) else -(-(need + 1) // 128) - 1


def _fused_plan(B, H, NQ, NK, D, l2, sms, causal):
    """The fused backward's key-range rule, restated: every key at once while the live dK rows fit in L2, else
    the longest range whose live rows (counted with the last range's query tiles) fit in half of it."""
    n_kt, n_qt = -(-NK // 128), -(-NQ // 128)
    if _live_rows_bytes(B, H, NQ, NK, D, sms) <= l2:
        return 1, B * H * NK * D * 4
    n = 2
    while True:
        tiles = -(-n_kt // n)
        ranges = -(-n_kt // tiles)
        qtiles = max(1, n_qt - _first_qtile(NQ, NK, (ranges - 1) * tiles * 128, causal))
        heads = min(B * H, -(-sms // qtiles) + 1)
        if tiles <= 1 or min(tiles * 128, NK) * D * 4 * heads <= l2 // 2:
            break
        n += 1
    ranges = -(-n_kt // tiles)
    return ranges, B * H * min(tiles * 128, NK) * D * 4 + (B * H * NQ * D * 4 if ranges > 1 else 0)


def test_bwd_select_and_fused_plan(lib):
    l2, sms = 135528448, 152  # GB300
    assert K.bwd_select(1, 8, 524288, 524288, 128, l2, sms) == K.BWD_FUSED  # many query tiles: fused over ranges
    assert K.bwd_select(1, 32, 65536, 65536, 128, l2, sms, True) == K.BWD_FUSED
    # at most eight query tiles per head and several key ranges: the separate kernels
    assert K.bwd_select(1, 128, 128, 65536, 128, l2, sms) == K.BWD_SEPARATE
    assert K.bwd_select(1, 64, 256, 131072, 128, l2, sms) == K.BWD_SEPARATE
    assert K.bwd_select(1, 32, 512, 262144, 128, l2, sms) == K.BWD_SEPARATE  # four query tiles
    assert K.bwd_select(1, 8, 1024, 65536, 128, l2, sms) == K.BWD_SEPARATE  # eight
    assert K.bwd_select(1, 8, 1025, 65536, 128, l2, sms) == K.BWD_FUSED  # nine
    assert K.bwd_select(1, 8, 2048, 65536, 128, l2, sms) == K.BWD_FUSED
    # one key range: the separate path only while the fused grid (B*H*query tiles blocks) leaves SMs idle
    assert K.bwd_select(1, 1, 128, 128, 64, l2, sms) == K.BWD_SEPARATE
    assert K.bwd_select(1, 18, 1024, 1024, 128, l2, sms) == K.BWD_SEPARATE  # 144 fused blocks on 152 SMs
    assert K.bwd_select(1, 19, 1024, 1024, 128, l2, sms) == K.BWD_FUSED  # 152
    assert K.bwd_select(64, 32, 1024, 1024, 128, l2, sms) == K.BWD_FUSED
    assert K.bwd_select(0, 1, 8, 8, 64, l2, sms) == 0  # invalid shape
    assert K.bwd_select(1, 1, 8, 8, 64, l2, 0) == 0  # no SM count
    # one launch while the live dK rows (heads in flight x N_K x D x 4 B) fit in L2
    assert K.bwd_fused_plan(1, 1, 128, 128, 64, l2, sms, False) == (1, 128 * 64 * 4)
    assert K.bwd_fused_plan(2, 32, 4096, 8192, 128, l2, sms, False) == (1, 2 * 32 * 8192 * 128 * 4)
    assert K.bwd_fused_plan(1, 32, 65536, 65536, 128, l2, sms, True) == (1, 32 * 65536 * 128 * 4)  # live 64 MiB
    # the 512K workload: one head's rows alone are 256 MiB -> 8 ranges of 64K keys (2 heads x 32 MiB live),
    # workspace = one range's dK rows + the fp32 dQ accumulator
    assert K.bwd_fused_plan(1, 8, 524288, 524288, 128, l2, sms, True) == (8, 8 * 65536 * 512 + 8 * 524288 * 512)
    for B, H, NQ, NK, causal in [(1, 8, 100000, 100000, True), (1, 8, 131072, 131072, False), (1, 4, 1000, 200000, True),
                                 (1, 8, 140000, 140000, True), (64, 32, 256, 4096, False), (1, 8, 200000, 260000, True)]:
        for l2b in (l2, l2 // 8, 77 * 4096 * 512, 77 * 4096 * 512 - 1):
            assert K.bwd_fused_plan(B, H, NQ, NK, 128, l2b, sms, causal) == _fused_plan(B, H, NQ, NK, 128, l2b, sms,
                                                                                      causal), (B, H, NQ, NK, l2b)


def test_fused_range_override(lib, monkeypatch):
    l2, sms = 135528448, 152
    monkeypatch.setenv("STREAMKL_FUSED_KEY_TILES", "2")
    assert K.bwd_fused_plan(2, 3, 300, 1000, 64, l2, sms, True) == (4, 2 * 3 * 256 * 64 * 4 + 2 * 3 * 300 * 64 * 4)
    monkeypatch.setenv("STREAMKL_FUSED_KEY_TILES", "100")  # longer than N_K: one launch
    assert K.bwd_fused_plan(2, 3, 300, 1000, 64, l2, sms, True) == (1, 2 * 3 * 1000 * 64 * 4)
    monkeypatch.setenv("STREAMKL_FUSED_KEY_TILES", "0")  # not positive: ignored
    assert K.bwd_fused_plan(2, 3, 300, 1000, 64, l2, sms, True) == (1, 2 * 3 * 1000 * 64 * 4)


@pytest.mark.parametrize("qs,ks,code", [
    ((0, 0, 0), (0, 0, 0), K.OK),                                   # contiguous
    ((64 * 4 * 128, 128, 4 * 128), (4096 * 4 * 128, 128, 4 * 128), K.OK),  # [B, N, H, D] views
    ((0, 0, 0), (3 * 4096 * 4 * 128, 128, 3 * 4 * 128), K.OK),      # K sliced from a packed [B, N, 3, H, D]
    ((64 * 4 * 128, 128, 64), (0, 0, 0), K.ERR_INVALID),            # rows shorter than D
    ((64 * 4 * 128, 128, 4 * 128 + 4), (0, 0, 0), K.ERR_INVALID),   # not a multiple of 8 elements
    ((0, 0, 0), (-128, 128, 512), K.ERR_INVALID),                   # negative
    ((0, 0, 128), (0, 0, 0), K.ERR_INVALID),                        # partly zero
    ((1 << 38, 128, 512), (0, 0, 0), K.ERR_INVALID),                # beyond the tensor map's stride range
])
def test_stride_validation(lib, qs, ks, code):
    s = K.make_shape(2, 4, 64, 4096, 128, q_strides=qs, k_strides=ks)
    n = ctypes.c_size_t()
    assert lib.streamkl_bwd_workspace(s, K.BWD_SEPARATE, ctypes.byref(n)) == code
    if code != K.OK:  # the compute entry points refuse the same shapes before any launch
        assert call_fwd(lib, s) == code


def test_binding_reads_views_in_place():
    torch = pytest.importorskip("torch")
    np = pytest.importorskip("numpy")
    B_, N, H, D = 2, 48, 4, 64
    bnhd = torch.zeros(B_, N, H, D, dtype=torch.bfloat16)
    assert K._bhn_strides(bnhd.permute(0, 2, 1, 3)) == (N * H * D, D, H * D)
    qkv = torch.zeros(B_, N, 3, H, D, dtype=torch.bfloat16)
    assert K._bhn_strides(qkv[:, :, 1].permute(0, 2, 1, 3)) == (N * 3 * H * D, D, 3 * H * D)
    c = torch.zeros(B_, H, N, D, dtype=torch.bfloat16)
    assert K._bhn_strides(c) == (H * N * D, N * D, D)
    assert K._bhn_strides(c[:1, :1]) == (8, 8, D)  # extent-1 strides replaced by valid ones
    assert K._bhn_strides(c.transpose(2, 3)) is None  # D not contiguous
    buf = torch.zeros(B_ * H * N * D + 8, dtype=torch.bfloat16)
    assert K._bhn_strides(buf[4:4 + B_ * H * N * D].view(B_, H, N, D)) is None  # start not 16-byte aligned
    assert K._bhn_strides(c[:, :1].expand(B_, H, N, D)) is None  # zero stride
    assert K._bhn_strides(torch.as_strided(c, (B_, H, N, D), (H * N * D, N * D, 8, 1))) is None  # overlapping rows
    empty = torch.from_numpy(np.zeros((1, 2, 0, 64), np.int16)).view(torch.bfloat16)  # numpy gives zero strides
    assert K._bhn_strides(empty) == (2 * 64, 64, 64)
    # a mismatched pair is made contiguous together
    a, b, st = K._pair(bnhd.permute(0, 2, 1, 3), c)
    assert a.is_contiguous() and b.is_contiguous() and st == (H * N * D, N * D, D)
    g = K._grad_like(qkv[:, :, 0].permute(0, 2, 1, 3), (N * 3 * H * D, D, 3 * H * D), N)
    assert g.stride() == (N * 3 * H * D, D, 3 * H * D, 1)


def test_key_shard_entry_points_validate_before_any_launch(lib):
    """streamkl_fwd_partials / _bwd_keyshard / _merge_partials / _dq_from_partial reject bad shards and
    pointers synchronously (no device is touched on these paths)."""
    p = [fake_ptr(64 * i) for i in range(16)]
    s = K.make_shape(1, 2, 64, 32, 64, None, True)  # a 32-key shard of a longer sequence
    part = fake_ptr(1 << 12)
    # the shard must lie inside the sequence
    assert lib.streamkl_fwd_partials(p[0], p[1], p[2], p[3], s, -1, 128, part, None) == K.ERR_INVALID
    assert lib.streamkl_fwd_partials(p[0], p[1], p[2], p[3], s, 100, 128, part, None) == K.ERR_INVALID
    # causal needs N_Q <= nk_total (here 64 > 48), not N_Q <= the shard's keys
    assert lib.streamkl_fwd_partials(p[0], p[1], p[2], p[3], s, 16, 48, part, None) == K.ERR_INVALID
    assert lib.streamkl_fwd_partials(p[0], p[1], p[2], p[3], s, 0, 64, fake_ptr(2), None) == K.ERR_INVALID
    assert lib.streamkl_fwd_partials(None, p[1], p[2], p[3], s, 0, 64, part, None) == K.ERR_INVALID
    s0 = K.make_shape(1, 2, 0, 32, 64)
    assert lib.streamkl_fwd_partials(None, None, None, None, s0, 0, 64, None, None) == K.OK  # no rows: no-op
    # merge: at least one part, aligned rows
    sm = K.make_shape(1, 2, 64, 1, 64)
    assert lib.streamkl_merge_partials(part, 0, sm, p[4], p[5], p[6], None) == K.ERR_INVALID
    assert lib.streamkl_merge_partials(part, 2, sm, fake_ptr(1), p[5], p[6], None) == K.ERR_INVALID
    # backward on a shard: setting, dK, dQ-partial and workspace checks come first
    args = (p[0], p[1], p[2], p[3], s, 0, 64, p[4], p[5], p[6], p[7])
    assert lib.streamkl_bwd_keyshard(3, *args, p[8], p[9], p[10], 1 << 20, None) == K.ERR_INVALID
    assert lib.streamkl_bwd_keyshard(1, *args, p[8], fake_ptr(2), p[10], 1 << 20, None) == K.ERR_INVALID
    assert lib.streamkl_bwd_keyshard(1, *args, fake_ptr(4), p[9], p[10], 1 << 20, None) == K.ERR_INVALID
    assert lib.streamkl_bwd_keyshard(1, *args, p[8], p[9], None, 0, None) == K.ERR_WORKSPACE
    assert lib.streamkl_bwd_keyshard(2, p[0], p[1], p[2], p[3], s, 0, 64, p[4], p[5], None, p[7], p[8], p[9],
                                     p[10], 1 << 20, None) == K.ERR_INVALID  # setting 2 needs the merged KL
    # dQ from the summed partials: aligned buffers
    assert lib.streamkl_dq_from_partial(fake_ptr(4), sm, p[9], None) == K.ERR_INVALID
    assert lib.streamkl_dq_from_partial(p[8], sm, fake_ptr(2), None) == K.ERR_INVALID


def test_bwd_mutual_select(lib):
    """The mutual case: the mutual kernels while a head has at most 64 query tiles; a fused pass per setting
    otherwise."""
    l2, sms = 135528448, 152  # GB300
    S = lambda *a: K.bwd_mutual_select(*a, l2, sms)  # noqa: E731
    assert S(1, 32, 128, 65536, 128) == K.BWD_SEPARATE
    assert S(1, 8, 8192, 65536, 128) == K.BWD_SEPARATE  # 64 query tiles
    assert S(1, 8, 8193, 65536, 128) == K.BWD_FUSED  # 65
    assert S(2, 32, 4096, 4096, 128, True) == K.BWD_SEPARATE
    assert S(1, 32, 65536, 65536, 128, True) == K.BWD_FUSED
    assert S(1, 8, 524288, 524288, 128, True) == K.BWD_FUSED
    assert K.bwd_mutual_select(0, 1, 8, 8, 64, l2, sms) == 0
    assert K.bwd_mutual_select(1, 1, 8, 8, 64, l2, 0) == 0


def test_bwd_mutual_validates_before_any_launch(lib):
    s = K.make_shape(1, 1, 8, 8, 64)
    p = [fake_ptr(64 * i) for i in range(16)]
    ins, rows = p[:4], p[4:8]
    outs = p[8:12]
    n = ctypes.c_size_t(1)
    for mode in (K.BWD_DQ_ONLY, K.BWD_DK_ONLY, 9):
        assert lib.streamkl_bwd_mutual(*ins, s, *rows, *outs, mode, p[12], 1 << 20, None) == K.ERR_INVALID
        assert lib.streamkl_bwd_mutual_workspace(s, mode, ctypes.byref(n)) == K.ERR_INVALID
    assert lib.streamkl_bwd_mutual_workspace(s, K.BWD_SEPARATE, ctypes.byref(n)) == K.OK and n.value == 0
    for k in range(4):  # every output is required and 16-byte aligned
        bad = list(outs)
        bad[k] = None
        assert lib.streamkl_bwd_mutual(*ins, s, *rows, *bad, K.BWD_SEPARATE, None, 0, None) == K.ERR_INVALID
        bad[k] = fake_ptr(2)
        assert lib.streamkl_bwd_mutual(*ins, s, *rows, *bad, K.BWD_SEPARATE, None, 0, None) == K.ERR_INVALID
    assert lib.streamkl_bwd_mutual(*ins, s, rows[0], rows[1], None, rows[3], *outs, K.BWD_SEPARATE, None, 0,
                                   None) == K.ERR_INVALID  # the saved KL is required
    assert lib.streamkl_bwd_mutual(*ins, s, *rows, *outs, K.BWD_FUSED, None, 0, None) == K.ERR_WORKSPACE
    assert lib.streamkl_bwd_mutual(*ins, s, *rows, *outs, K.BWD_FUSED, fake_ptr(8), 1 << 20,
                                   None) == K.ERR_WORKSPACE  # misaligned workspace
