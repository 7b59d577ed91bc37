"""The allocation-free Split-K entry point, streamkl_fwd_splitk_noalloc.

It serves callers that cannot allocate device memory (the GPU's memory is
owned by a host application or serving runtime, or a decode loop's budget is
fixed up front): it keeps the split partials in a static device array built
into the library instead of a caller-provided workspace.  This test calls it
through the C-ABI and compares it with streamkl_fwd_splitk (caller workspace)
on two calls in a row, using the tolerances of the other parity tests.  It
runs last (file name) and builds/loads the library itself, so it passes both
alone in a fresh process and after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

import attention_kl_divergence_streamkl_gb300 as skl
from attention_kl_divergence_streamkl_gb300 import _lib as K
from attention_kl_divergence_streamkl_gb300 import build, synth
from tests import parity_util as U

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(L, ins, w, splits):
    out = [torch.full((w.B, w.H, w.NQ), float("nan"), device="cuda") for _ in range(3)]
    s = K.make_shape(w.B, w.H, w.NQ, w.NK, w.D, w.softmax_scale, w.causal)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = L.streamkl_fwd_splitk_noalloc(*(_p(t) for t in ins), s, splits, *(_p(t) for t in out), stream)
    return st, out


def test_noalloc_splitk_matches_workspace_entry_point_on_two_calls():
    """Two calls in a row on different problems: the second (fewer heads, other split count, other values)
    finds the first one's partials in the shared scratch and must still match the workspace entry point on
    its own inputs, so a partial that the second call failed to write would show up."""
    build.build()
    L = skl.lib()
    problems = [(synth.Workload("noalloc", 2, 8, 5, 3000, 128, True, 0.5, 21), 7),
                (synth.Workload("noalloc_b", 1, 6, 4, 2900, 128, False, 0.5, 23), 5)]
    for call, (w, splits) in enumerate(problems):
        ins = U.dev_inputs(synth.make_inputs(w))
        ref = skl.fwd_splitk(*ins, w.softmax_scale, w.causal, num_splits=splits)
        st, out = _noalloc(L, ins, w, splits)
        assert st == K.OK, K.status_string(st)
        torch.cuda.synchronize()
        U.assert_rows(*(U.np64(x) for x in out), *(U.np64(x) for x in ref), f"call {call}")
    assert skl.check_device_status() == K.OK


def test_noalloc_auto_splits_and_limit():
    build.build()
    L = skl.lib()
    w = synth.Workload("noalloc2", 1, 4, 16, 8192, 64, False, 0.5, 22)
    ins = U.dev_inputs(synth.make_inputs(w))
    ref = skl.fwd_splitk(*ins, w.softmax_scale, w.causal)
    st, out = _noalloc(L, ins, w, 0)
    assert st == K.OK, K.status_string(st)
    torch.cuda.synchronize()
    U.assert_rows(*(U.np64(x) for x in out), *(U.np64(x) for x in ref), "auto splits")
    # partials beyond the fixed scratch are refused before any launch
    too_many = (4 << 20) // (w.B * w.H * w.NQ * 5 * 4) + 1
    st, out = _noalloc(L, ins, w, too_many)
    assert st == K.ERR_SCRATCH_LIMIT
    assert np.isnan(U.np64(out[0])).all()  # nothing was written
