"""libstreamkl: fused one-pass attention KL divergence on one GB300 (sm_103a).

Python surface over the C-ABI library ``libstreamkl.so`` (see
``include/streamkl.h``).  The shared library is loaded on first use and every
call fails loudly if it is missing; nothing here computes on the CPU.
"""
from ._lib import (BWD_AUTO, BWD_DK_ONLY, BWD_DQ_ONLY, BWD_FUSED, BWD_SEPARATE, SPLITK_MAX_NQ,  # noqa: F401
                   Shape, StreamKLError,
                   bwd_fused_plan, bwd_keyshard, bwd_mutual, bwd_mutual_select, bwd_s1, bwd_s2, bwd_select, bwd_workspace_bytes,
                   check_device_status, debug_wait_timeout, dq_from_partial,
                   fwd, fwd_partials, fwd_splitk, lib, make_shape, merge_partials, splitk_plan, status_string)
from .autograd import attention_kl  # noqa: E402,F401
