"""ctypes binding of libstreamkl (argument marshalling only).

Every step of the computation runs in the CUDA kernels of ``libstreamkl.so``;
this module only checks tensor metadata, allocates outputs and workspaces
through PyTorch's CUDA allocator, and passes raw pointers and the current CUDA
stream to the C entry points of the same names.  There is no CPU fallback: if
the library is missing, every call raises.

Inputs given as CPU tensors are copied to the current CUDA device on the
current stream (non-blocking from pinned memory) and the results are copied
back, so a host caller uses the same functions.

Device inputs need not be contiguous: any [B, H, N, D] view whose D is
contiguous, whose other strides are multiples of 8 elements and whose rows do
not overlap (a [B, N, H, D] tensor permuted, a slice of a packed QKV tensor) is
passed as it is, with its strides; the gradients come back with the strides of
the input they belong to.  Other views are copied to a contiguous tensor first.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libstreamkl.so")

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT, ERR_SCRATCH_LIMIT = range(7)
BWD_AUTO, BWD_FUSED, BWD_SEPARATE, BWD_DQ_ONLY, BWD_DK_ONLY = 0, 1, 2, 3, 4
SPLITK_MAX_NQ = 16


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("NQ", ctypes.c_int), ("NK", ctypes.c_int),
                ("D", ctypes.c_int), ("scale", ctypes.c_float), ("causal", ctypes.c_int),
                ("q_stride_b", ctypes.c_longlong), ("q_stride_h", ctypes.c_longlong),
                ("q_stride_n", ctypes.c_longlong), ("k_stride_b", ctypes.c_longlong),
                ("k_stride_h", ctypes.c_longlong), ("k_stride_n", ctypes.c_longlong)]


class StreamKLError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_P, _F, _S, _I, _SZ = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_LL = ctypes.c_longlong
# name -> (restype, argtypes); also the list of symbols include/streamkl.h declares
SIGNATURES = {
    "streamkl_fwd": (_I, [_P, _P, _P, _P, Shape, _F, _F, _F, _S]),
    "streamkl_fwd_splitk_workspace": (_I, [Shape, _I, ctypes.POINTER(_SZ)]),
    "streamkl_fwd_splitk": (_I, [_P, _P, _P, _P, Shape, _I, _P, _SZ, _F, _F, _F, _S]),
    "streamkl_fwd_splitk_plan": (_I, [Shape, _I, ctypes.POINTER(_I)]),
    "streamkl_fwd_splitk_noalloc": (_I, [_P, _P, _P, _P, Shape, _I, _F, _F, _F, _S]),
    "streamkl_fwd_partials": (_I, [_P, _P, _P, _P, Shape, _LL, _LL, _F, _S]),
    "streamkl_merge_partials": (_I, [_F, _I, Shape, _F, _F, _F, _S]),
    "streamkl_bwd_keyshard_workspace": (_I, [Shape, _LL, _LL, ctypes.POINTER(_SZ)]),
    "streamkl_bwd_keyshard": (_I, [_I, _P, _P, _P, _P, Shape, _LL, _LL, _F, _F, _F, _F, _F, _P, _P, _SZ, _S]),
    "streamkl_dq_from_partial": (_I, [_F, Shape, _P, _S]),
    "streamkl_bwd_workspace": (_I, [Shape, _I, ctypes.POINTER(_SZ)]),
    "streamkl_bwd_select": (_I, [Shape, _SZ, _I]),
    "streamkl_bwd_fused_plan": (_I, [Shape, _SZ, _I, ctypes.POINTER(_I), ctypes.POINTER(_SZ)]),
    "streamkl_bwd_s1": (_I, [_P, _P, _P, _P, Shape, _F, _F, _F, _P, _P, _I, _P, _SZ, _S]),
    "streamkl_bwd_s2": (_I, [_P, _P, _P, _P, Shape, _F, _F, _F, _F, _P, _P, _I, _P, _SZ, _S]),
    "streamkl_bwd_mutual": (_I, [_P, _P, _P, _P, Shape, _F, _F, _F, _F, _P, _P, _P, _P, _I, _P, _SZ, _S]),
    "streamkl_bwd_mutual_select": (_I, [Shape, _SZ, _I]),
    "streamkl_bwd_mutual_workspace": (_I, [Shape, _I, ctypes.POINTER(_SZ)]),
    "streamkl_status_string": (ctypes.c_char_p, [_I]),
    "streamkl_check_device_status": (_I, [_S]),
    "streamkl_debug_wait_timeout": (_I, [_I, _S]),
    "streamkl_version": (_I, []),
}

_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libstreamkl.so not found at {LIB_PATH}: build it with "
                               "attention_kl_divergence_streamkl_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().streamkl_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != OK:
        raise StreamKLError(status, where)


def make_shape(B, H, NQ, NK, D, scale=None, causal=False, q_strides=(0, 0, 0), k_strides=(0, 0, 0)) -> Shape:
    """The C shape; q_strides / k_strides are element strides along (b, h, n), zeros = contiguous."""
    return Shape(int(B), int(H), int(NQ), int(NK), int(D), float(scale or 0.0), int(bool(causal)),
                 *(int(x) for x in q_strides), *(int(x) for x in k_strides))


def _bhn_strides(t: torch.Tensor):
    """(b, h, n) element strides under which the library can read `t` in place, else None.

    D must be contiguous, the start 16-byte aligned, each stride of an extent > 1
    a positive multiple of 8 elements and the rows pairwise disjoint (sorted by
    stride, each stride covers the extent below it).  The stride of an extent-1
    dimension is never used to address anything; it is replaced by a valid one.
    """
    B, H, N, D = t.shape
    if t.numel() == 0:  # nothing is read; any valid strides do
        return max(H, 1) * max(N, 1) * D, max(N, 1) * D, D
    if t.stride(3) != 1 or t.data_ptr() % 16:
        return None
    dims = [(t.stride(i), t.size(i)) for i in range(4) if t.size(i) > 1]
    if any(st <= 0 for st, _ in dims):
        return None
    span = 0
    for st, n in sorted(dims):
        if st < span:
            return None
        span = st * n
    sn = t.stride(2) if t.size(2) > 1 else D
    sh = t.stride(1) if t.size(1) > 1 else 8
    sb = t.stride(0) if t.size(0) > 1 else 8
    if sn < D or any(x % 8 for x in (sb, sh, sn)):
        return None
    return sb, sh, sn


def _pair(a: torch.Tensor, b: torch.Tensor):
    """The two tensors of a pair (Q1/Q2 or K1/K2) and their shared (b, h, n) strides."""
    sa, sb = _bhn_strides(a), _bhn_strides(b)
    if sa is None or sa != sb:
        a, b = a.contiguous(), b.contiguous()
        sa = _bhn_strides(a)
        if sa is None:
            raise ValueError("inputs must be 16-byte aligned")
    return a, b, sa


def _grad_like(t: torch.Tensor, strides, rows) -> torch.Tensor:
    """A bf16 output with the (b, h, n) strides the library writes `t`'s gradient with."""
    B, H, _, D = t.shape
    return torch.empty_strided((B, H, rows, D), (strides[0], strides[1], strides[2], 1), dtype=torch.bfloat16,
                               device=t.device)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _prep(q1, k1, q2, k2):
    """Validates the four inputs; returns (device tensors, was_host, q strides, k strides)."""
    ts = [q1, k1, q2, k2]
    for t in ts:
        if t.dtype != torch.bfloat16:
            raise TypeError("Q1, K1, Q2, K2 must be bfloat16")
        if t.dim() != 4:
            raise ValueError("Q1, K1, Q2, K2 must be [B, H, N, D]")
    if q1.shape != q2.shape or k1.shape != k2.shape or q1.shape[:2] != k1.shape[:2] or q1.shape[3] != k1.shape[3]:
        raise ValueError(f"shape mismatch: Q1 {tuple(q1.shape)} K1 {tuple(k1.shape)} "
                         f"Q2 {tuple(q2.shape)} K2 {tuple(k2.shape)}")
    host = q1.device.type == "cpu"
    if host:
        dev = torch.device("cuda", torch.cuda.current_device())
        ts = [t.contiguous().to(dev, non_blocking=True) for t in ts]
    elif any(t.device != ts[0].device for t in ts):
        raise ValueError("inputs on different devices")
    q1, q2, qs = _pair(ts[0], ts[2])
    k1, k2, ks = _pair(ts[1], ts[3])
    return [q1, k1, q2, k2], host, qs, ks


def _rows(t: Optional[torch.Tensor], dev, shape3, name):
    if t is None:
        return None
    if t.dtype != torch.float32 or tuple(t.shape) != tuple(shape3):
        raise ValueError(f"{name} must be float32 of shape {tuple(shape3)}")
    return t.to(dev, non_blocking=True).contiguous()


def _back(ts, host):
    if not host:
        return ts
    out = tuple(t.to("cpu", non_blocking=True) for t in ts)
    torch.cuda.current_stream().synchronize()
    return out


def fwd(q1, k1, q2, k2, scale=None, causal=False):
    """KL, LSE1, LSE2 fp32 [B, H, N_Q] (one-pass forward)."""
    (q1, k1, q2, k2), host, qs, ks = _prep(q1, k1, q2, k2)
    B, H, NQ, D = q1.shape
    s = make_shape(B, H, NQ, k1.shape[2], D, scale, causal, qs, ks)
    kl, l1, l2 = (torch.empty((B, H, NQ), dtype=torch.float32, device=q1.device) for _ in range(3))
    _check(lib().streamkl_fwd(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), s, _ptr(kl), _ptr(l1), _ptr(l2),
                              _stream(q1.device)), "streamkl_fwd")
    return _back((kl, l1, l2), host)


def splitk_plan(B, H, NQ, NK, D, num_sms=0, causal=False) -> int:
    n = ctypes.c_int(0)
    _check(lib().streamkl_fwd_splitk_plan(make_shape(B, H, NQ, NK, D, None, causal), int(num_sms),
                                          ctypes.byref(n)), "streamkl_fwd_splitk_plan")
    return n.value


def fwd_splitk(q1, k1, q2, k2, scale=None, causal=False, num_splits=0):
    """Split-K forward for N_Q <= 16: KL, LSE1, LSE2 fp32 [B, H, N_Q]."""
    (q1, k1, q2, k2), host, qs, ks = _prep(q1, k1, q2, k2)
    B, H, NQ, D = q1.shape
    s = make_shape(B, H, NQ, k1.shape[2], D, scale, causal, qs, ks)
    nbytes = ctypes.c_size_t(0)
    _check(lib().streamkl_fwd_splitk_workspace(s, int(num_splits), ctypes.byref(nbytes)),
           "streamkl_fwd_splitk_workspace")
    ws = torch.empty(max(16, nbytes.value), dtype=torch.uint8, device=q1.device)
    kl, l1, l2 = (torch.empty((B, H, NQ), dtype=torch.float32, device=q1.device) for _ in range(3))
    _check(lib().streamkl_fwd_splitk(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), s, int(num_splits), _ptr(ws),
                                     nbytes.value, _ptr(kl), _ptr(l1), _ptr(l2), _stream(q1.device)),
           "streamkl_fwd_splitk")
    return _back((kl, l1, l2), host)


def fwd_partials(q1, k1, q2, k2, key_offset, nk_total, scale=None, causal=False):
    """Five scalars per row fp32 [B, H, N_Q, 5] over a key shard.

    k1, k2 hold the shard's keys, at global positions [key_offset, key_offset +
    k1.shape[2]) of a sequence of nk_total keys (the causal frontier is the
    global one).  Merge the shards' partials with merge_partials."""
    (q1, k1, q2, k2), host, qs, ks = _prep(q1, k1, q2, k2)
    B, H, NQ, D = q1.shape
    s = make_shape(B, H, NQ, k1.shape[2], D, scale, causal, qs, ks)
    part = torch.empty((B, H, NQ, 5), dtype=torch.float32, device=q1.device)
    _check(lib().streamkl_fwd_partials(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), s, int(key_offset), int(nk_total),
                                       _ptr(part), _stream(q1.device)), "streamkl_fwd_partials")
    return _back((part,), host)[0]


def merge_partials(parts, D, scale=None):
    """KL, LSE1, LSE2 fp32 [B, H, N_Q] from partial sets stacked as [S, B, H, N_Q, 5] (device)."""
    if parts.dtype != torch.float32 or parts.dim() != 5 or parts.shape[-1] != 5:
        raise ValueError("partials must be float32 [S, B, H, N_Q, 5]")
    parts = parts.contiguous()
    S, B, H, NQ, _ = parts.shape
    s = make_shape(B, H, NQ, 1, D, scale, False)
    kl, l1, l2 = (torch.empty((B, H, NQ), dtype=torch.float32, device=parts.device) for _ in range(3))
    _check(lib().streamkl_merge_partials(_ptr(parts), int(S), s, _ptr(kl), _ptr(l1), _ptr(l2),
                                         _stream(parts.device)), "streamkl_merge_partials")
    return kl, l1, l2


def bwd_keyshard(setting, q1, k1, q2, k2, key_offset, nk_total, lse1, lse2, kl, g, scale=None, causal=False):
    """Backward over a key shard: (unscaled fp32 dQ contribution [B, H, N_Q, D], bf16 dK of the shard's keys).

    lse1, lse2, kl are the merged values of the whole sequence; summing the
    dQ contributions of every shard and passing the sum to dq_from_partial gives dQ."""
    (q1, k1, q2, k2), host, qs, ks = _prep(q1, k1, q2, k2)
    B, H, NQ, D = q1.shape
    NK = k1.shape[2]
    dev = q1.device
    s = make_shape(B, H, NQ, NK, D, scale, causal, qs, ks)
    lse1 = _rows(lse1, dev, (B, H, NQ), "lse1")
    lse2 = _rows(lse2, dev, (B, H, NQ), "lse2")
    g = _rows(g, dev, (B, H, NQ), "g")
    kl = _rows(kl, dev, (B, H, NQ), "kl") if setting == 2 else None
    nbytes = ctypes.c_size_t(0)
    _check(lib().streamkl_bwd_keyshard_workspace(s, int(key_offset), int(nk_total), ctypes.byref(nbytes)),
           "streamkl_bwd_keyshard_workspace")
    ws = torch.empty(max(16, nbytes.value), dtype=torch.uint8, device=dev)
    dq = torch.empty((B, H, NQ, D), dtype=torch.float32, device=dev)
    dk = _grad_like(k1, ks, NK)
    _check(lib().streamkl_bwd_keyshard(int(setting), _ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), s, int(key_offset),
                                       int(nk_total), _ptr(lse1), _ptr(lse2), _ptr(kl), _ptr(g), _ptr(dq), _ptr(dk),
                                       _ptr(ws), nbytes.value, _stream(dev)), "streamkl_bwd_keyshard")
    return _back((dq, dk), host)


def dq_from_partial(dq_partial, q_like, scale=None):
    """bf16 dQ = scale * dq_partial, with the layout the library gives q_like's gradient."""
    if dq_partial.dtype != torch.float32 or dq_partial.dim() != 4:
        raise ValueError("dq_partial must be float32 [B, H, N_Q, D]")
    dq_partial = dq_partial.contiguous()
    B, H, NQ, D = dq_partial.shape
    qs = _bhn_strides(q_like) or (H * NQ * D, NQ * D, D)
    s = make_shape(B, H, NQ, 1, D, scale, False, qs)
    out = _grad_like(q_like, qs, NQ) if _bhn_strides(q_like) else torch.empty(
        (B, H, NQ, D), dtype=torch.bfloat16, device=dq_partial.device)
    _check(lib().streamkl_dq_from_partial(_ptr(dq_partial), s, _ptr(out), _stream(dq_partial.device)),
           "streamkl_dq_from_partial")
    return out


def bwd_select(B, H, NQ, NK, D, l2_bytes, num_sms, causal=False) -> int:
    return lib().streamkl_bwd_select(make_shape(B, H, NQ, NK, D, None, causal), int(l2_bytes), int(num_sms))


def bwd_fused_plan(B, H, NQ, NK, D, l2_bytes, num_sms, causal=False):
    """(key ranges, workspace bytes) of the fused backward on a device with this L2 and SM count."""
    n, ws = ctypes.c_int(0), ctypes.c_size_t(0)
    _check(lib().streamkl_bwd_fused_plan(make_shape(B, H, NQ, NK, D, None, causal), int(l2_bytes), int(num_sms),
                                         ctypes.byref(n), ctypes.byref(ws)), "streamkl_bwd_fused_plan")
    return n.value, ws.value


def bwd_workspace_bytes(B, H, NQ, NK, D, bwd_mode=BWD_AUTO, causal=False) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().streamkl_bwd_workspace(make_shape(B, H, NQ, NK, D, None, causal), int(bwd_mode),
                                        ctypes.byref(n)), "streamkl_bwd_workspace")
    return n.value


def _bwd(setting, q1, k1, q2, k2, lse1, lse2, kl, g, scale, causal, bwd_mode):
    (q1, k1, q2, k2), host, qs, ks = _prep(q1, k1, q2, k2)
    B, H, NQ, D = q1.shape
    NK = k1.shape[2]
    dev = q1.device
    s = make_shape(B, H, NQ, NK, D, scale, causal, qs, ks)
    lse1 = _rows(lse1, dev, (B, H, NQ), "lse1")
    lse2 = _rows(lse2, dev, (B, H, NQ), "lse2")
    g = _rows(g, dev, (B, H, NQ), "g")
    kl = _rows(kl, dev, (B, H, NQ), "kl") if setting == 2 else None
    nbytes = ctypes.c_size_t(0)
    _check(lib().streamkl_bwd_workspace(s, int(bwd_mode), ctypes.byref(nbytes)), "streamkl_bwd_workspace")
    ws = torch.empty(max(16, nbytes.value), dtype=torch.uint8, device=dev)
    dq = _grad_like(q1, qs, NQ) if bwd_mode != BWD_DK_ONLY else None
    dk = _grad_like(k1, ks, NK) if bwd_mode != BWD_DQ_ONLY else None
    if setting == 1:
        st = lib().streamkl_bwd_s1(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), s, _ptr(lse1), _ptr(lse2), _ptr(g),
                                   _ptr(dq), _ptr(dk), int(bwd_mode), _ptr(ws), nbytes.value, _stream(dev))
    else:
        st = lib().streamkl_bwd_s2(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), s, _ptr(lse1), _ptr(lse2), _ptr(kl),
                                   _ptr(g), _ptr(dq), _ptr(dk), int(bwd_mode), _ptr(ws), nbytes.value,
                                   _stream(dev))
    _check(st, f"streamkl_bwd_s{setting}")
    got = iter(_back(tuple(t for t in (dq, dk) if t is not None), host))
    return tuple(None if t is None else next(got) for t in (dq, dk))


def bwd_s1(q1, k1, q2, k2, lse1, lse2, g, scale=None, causal=False, bwd_mode=BWD_AUTO):
    """Setting 1 (P1 fixed): (dQ2, dK2) bf16."""
    return _bwd(1, q1, k1, q2, k2, lse1, lse2, None, g, scale, causal, bwd_mode)


def bwd_s2(q1, k1, q2, k2, lse1, lse2, kl, g, scale=None, causal=False, bwd_mode=BWD_AUTO):
    """Setting 2 (P2 fixed): (dQ1, dK1) bf16."""
    return _bwd(2, q1, k1, q2, k2, lse1, lse2, kl, g, scale, causal, bwd_mode)


def bwd_mutual_select(B, H, NQ, NK, D, l2_bytes, num_sms, causal=False) -> int:
    """AUTO's path for the mutual case (BWD_SEPARATE = the mutual kernels, BWD_FUSED = a fused pass per setting)."""
    return lib().streamkl_bwd_mutual_select(make_shape(B, H, NQ, NK, D, None, causal), int(l2_bytes), int(num_sms))


def bwd_mutual(q1, k1, q2, k2, lse1, lse2, kl, g, scale=None, causal=False, bwd_mode=BWD_AUTO):
    """Gradients of all four inputs (the mutual case): (dQ1, dK1, dQ2, dK2) bf16.

    bwd_mode BWD_SEPARATE rebuilds each logit tile pair once for both settings;
    BWD_FUSED runs one fused pass per setting; BWD_AUTO picks by shape.
    """
    (q1, k1, q2, k2), host, qs, ks = _prep(q1, k1, q2, k2)
    B, H, NQ, D = q1.shape
    NK = k1.shape[2]
    dev = q1.device
    s = make_shape(B, H, NQ, NK, D, scale, causal, qs, ks)
    lse1 = _rows(lse1, dev, (B, H, NQ), "lse1")
    lse2 = _rows(lse2, dev, (B, H, NQ), "lse2")
    kl = _rows(kl, dev, (B, H, NQ), "kl")
    g = _rows(g, dev, (B, H, NQ), "g")
    nbytes = ctypes.c_size_t(0)
    _check(lib().streamkl_bwd_mutual_workspace(s, int(bwd_mode), ctypes.byref(nbytes)),
           "streamkl_bwd_mutual_workspace")
    ws = torch.empty(max(16, nbytes.value), dtype=torch.uint8, device=dev)
    dq1, dq2 = _grad_like(q1, qs, NQ), _grad_like(q2, qs, NQ)
    dk1, dk2 = _grad_like(k1, ks, NK), _grad_like(k2, ks, NK)
    _check(lib().streamkl_bwd_mutual(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), s, _ptr(lse1), _ptr(lse2), _ptr(kl),
                                     _ptr(g), _ptr(dq1), _ptr(dk1), _ptr(dq2), _ptr(dk2), int(bwd_mode), _ptr(ws),
                                     nbytes.value, _stream(dev)),
           "streamkl_bwd_mutual")
    return _back((dq1, dk1, dq2, dk2), host)


def check_device_status(device=None) -> int:
    """Synchronises the current stream and returns (and clears) the device status."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    return lib().streamkl_check_device_status(_stream(dev))


def debug_wait_timeout(timeout_us: int) -> int:
    dev = torch.device("cuda", torch.cuda.current_device())
    return lib().streamkl_debug_wait_timeout(int(timeout_us), _stream(dev))
