"""spec_verify_static: the entry point for callers that cannot allocate device
memory (for example code running under a framework that owns every device
allocation, so it has no way to hand spec_verify a workspace). It uses a
fixed scratch array inside the library instead. These tests call it through
the C ABI and check it against spec_verify, which takes a caller workspace.

This file is collected last on purpose: if its GPU test fails, a run that
stops at the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import speculative_decoding_token_verify_gb300 as sv
from speculative_decoding_token_verify_gb300 import _native

import helpers as hv
import workloads
from helpers import poison_f32, poison_i32

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
    """spec_verify_static through the C ABI, outputs allocated here and
    poisoned, so an entry the call never writes cannot pass."""
    L = _native.lib()
    zt, x = inp["zt"], inp["x"]
    zd = inp["zd"] if (mode == "stochastic" or est is not None) else None
    u = inp["u"] if mode == "stochastic" else None
    B, K1, V = zt.shape
    K = K1 - 1
    dev = zt.device
    out = dict(out_tokens=poison_i32((B, K + 1), dev), accepted_len=poison_i32((B,), dev),
               pos_stats=poison_f32((B, K + 1, 4), dev))
    if zd is not None:
        out["feature"] = poison_f32((B, K), dev)
        out["conf"] = poison_f32((B, K), dev) if est is not None else None
    dt = sv.BF16 if zt.dtype == torch.bfloat16 else sv.F32
    p = sv.make_params(B, K, V, dt, mode, kw.get("fly_theta", 0.3), kw.get("fly_window", 6), V, V)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    rc = L.spec_verify_static(ctypes.byref(p), _p(zt), _p(zd), _p(x), _p(u), _p(out["out_tokens"]),
                              _p(out["accepted_len"]), _p(out["pos_stats"]), _p(est), _p(out.get("feature")),
                              _p(out.get("conf")), stream)
    assert rc == 0, _native.last_error()
    torch.cuda.synchronize()
    return {k: v for k, v in out.items() if v is not None}


def _static_status():
    v = ctypes.c_int32(-1)
    assert _native.lib().spec_static_device_status(ctypes.byref(v)) == 0, _native.last_error()
    return int(v.value)


def _bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t


def _same_bits(a, b):
    """Both calls run the same kernels on the same inputs, and every output is
    deterministic, so the two must agree bit for bit (NaNs included)."""
    for k in a:
        assert torch.equal(_bits(a[k]), _bits(b[k])), k


@pytest.mark.gpu
def test_static_entry_matches_spec_verify_call_after_call():
    """Calls in a row, each checked bit for bit against spec_verify (caller
    workspace) on the same inputs: a larger batch first, then smaller ones,
    in the stochastic, greedy and FLy rules, so that nothing a larger call
    left in the shared array (draw records, partials, slice sums) can leak
    into a later, smaller one. The static status word reads clean after each."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    cases = [(workloads.ESTIMATOR.scaled(B=96), 2101, "stochastic"),
             (workloads.ESTIMATOR.scaled(B=20), 2102, "stochastic"),
             (workloads.FLY.scaled(B=32), 2103, "fly"),
             (workloads.ESTIMATOR.scaled(B=20), 2104, "greedy"),
             (workloads.LLAMA3_VOCAB.scaled(B=8), 2105, "stochastic")]
    for w, seed, mode in cases:
        inp = workloads.make_inputs(w, seed, dev)
        est = torch.tensor([1.0] + [0.0] * w.K, dtype=torch.float32, device=dev) if mode == "stochastic" else None
        kw = dict(fly_theta=w.fly_theta, fly_window=w.fly_window) if mode == "fly" else {}
        got = _static_call(inp, mode, est, **kw)
        assert _static_status() == 0
        zd = inp["zd"] if mode == "stochastic" else None
        ref = hv.verify(inp["zt"], zd, inp["x"], inp["u"] if mode == "stochastic" else None, mode=mode,
                        est_params=est, want_pos_stats=True, want_feature=zd is not None,
                        want_conf=est is not None, **kw)
        torch.cuda.synchronize()
        ref = {k: ref[k] for k in got}
        _same_bits(got, ref)


@pytest.mark.gpu
def test_static_status_word_reports_device_errors():
    """A draft token outside [0, V) raises SPEC_ERR_BAD_TOKEN in the static
    call's status word, read through spec_static_device_status; the next
    clean call clears it."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    w = workloads.TINY
    inp = workloads.make_inputs(w, 2110, dev)
    inp["x"] = inp["x"].clone()
    inp["x"][1, 2] = w.V + 3
    _static_call(inp, "stochastic", None)
    assert _static_status() == sv.api.SPEC_ERR_BAD_TOKEN
    _static_call(workloads.make_inputs(w, 2111, dev), "stochastic", None)
    assert _static_status() == 0
