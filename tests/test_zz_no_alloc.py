"""spec_verify_static: the entry point for callers that cannot allocate device
memory (for example code running under a framework that owns every device
allocation, so it has no way to hand spec_verify a workspace). It uses a
fixed scratch array inside the library instead. These tests call it through
the C ABI and check it against spec_verify, which takes a caller workspace.

This file is collected last on purpose: if its GPU test fails, a run that
stops at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import speculative_decoding_token_verify_gb300 as sv
from speculative_decoding_token_verify_gb300 import _native

import workloads
from helpers import tol_for

STATIC_BYTES = 16 << 20


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_static_entry_rejects_oversized_calls():
    """Calls whose scratch would not fit the static array are refused on the
    host with SPEC_ERR_UNSUPPORTED before anything is enqueued."""
    L = _native.lib()
    p = sv.make_params(B=4096, K=8, V=152064, dtype=sv.F32, mode="stochastic")
    assert L.spec_workspace_size(ctypes.byref(p)) > STATIC_BYTES
    fake = ctypes.c_void_p(0x7f0000000000)
    rc = L.spec_verify_static(ctypes.byref(p), fake, fake, fake, fake, fake, fake, None, None, None,
                              None, None)
    assert rc == sv.api.SPEC_ERR_UNSUPPORTED
    assert b"static" in L.spec_last_error()
    assert L.spec_verify_static(None, fake, fake, fake, fake, fake, fake, None, None, None, None,
                                None) == sv.api.SPEC_ERR_INVALID_ARG


def _static_call(inp, mode, est, **kw):
    """spec_verify_static through the C ABI, outputs allocated here."""
    L = _native.lib()
    zt, zd, x = inp["zt"], inp["zd"], inp["x"]
    u = inp["u"] if mode == "stochastic" else None
    B, K1, V = zt.shape
    K = K1 - 1
    dev = zt.device
    out = dict(out_tokens=torch.full((B, K + 1), -7, dtype=torch.int32, device=dev),
               accepted_len=torch.full((B,), -7, dtype=torch.int32, device=dev),
               pos_stats=torch.full((B, K + 1, 4), 7.0, device=dev),
               feature=torch.full((B, K), 7.0, device=dev),
               conf=torch.full((B, K), 7.0, device=dev))
    dt = sv.BF16 if zt.dtype == torch.bfloat16 else sv.F32
    p = sv.make_params(B, K, V, dt, mode, kw.get("fly_theta", 0.3), kw.get("fly_window", 6), V, V)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    rc = L.spec_verify_static(ctypes.byref(p), _p(zt), _p(zd), _p(x), _p(u), _p(out["out_tokens"]),
                              _p(out["accepted_len"]), _p(out["pos_stats"]), _p(est), _p(out["feature"]),
                              _p(out["conf"]), stream)
    assert rc == 0, _native.last_error()
    torch.cuda.synchronize()
    return out


def _compare(a, b, dtype):
    assert torch.equal(a["out_tokens"], b["out_tokens"])
    assert torch.equal(a["accepted_len"], b["accepted_len"])
    tol = tol_for(dtype)
    for k in ("pos_stats", "feature", "conf"):
        x = a[k].cpu().numpy().astype(np.float64)
        y = b[k].cpu().numpy().astype(np.float64)
        same = (np.isnan(x) & np.isnan(y)) | (x == y)
        assert (same | (np.abs(x - y) <= tol * np.maximum(1.0, np.abs(y)))).all(), k


@pytest.mark.gpu
def test_static_entry_matches_spec_verify_twice():
    """Two calls in a row, each checked against spec_verify on the same
    inputs; the second call must not see the first call's leftovers."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    w = workloads.ESTIMATOR.scaled(B=48)
    est = torch.tensor([1.0] + [0.0] * w.K, dtype=torch.float32, device=dev)
    for seed, mode in ((2101, "stochastic"), (2102, "stochastic")):
        inp = workloads.make_inputs(w, seed, dev)
        got = _static_call(inp, mode, est)
        ref = sv.verify(inp["zt"], inp["zd"], inp["x"], inp["u"], mode=mode, est_params=est,
                        want_pos_stats=True, want_feature=True, want_conf=True)
        torch.cuda.synchronize()
        _compare(got, ref, w.dtype)
