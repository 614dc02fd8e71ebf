"""GB300 (sm_103a) speculative-decoding verification.

The verification pass runs in the CUDA library ``libspecverify.so`` behind the
C ABI of ``include/spec_verify.h``; this package is its build step and a thin
binding. Nothing here computes the method on the CPU: if the library is not
built, every call raises.
"""
from ._native import build, lib, LIB_PATH  # noqa: F401
from .api import (  # noqa: F401
    BF16, F32, FLY, GREEDY, MAX_K, MAX_V, MODES, STOCHASTIC, IrlsState, SpecError, Workspace, av_budget,
    confidence, device_status, estimator_update, irls_accumulate, irls_refit, make_params, ngram_draft, verify,
    workspace_size,
)
