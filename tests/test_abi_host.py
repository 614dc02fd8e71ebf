"""CPU tests of the C ABI boundary: the library loads, exports every symbol
include/spec_verify.h declares, lays out spec_verify_params as the header
does, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

import speculative_decoding_token_verify_gb300 as sv
from speculative_decoding_token_verify_gb300 import _native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def L():
    _native.build()
    return _native.lib()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 8
    out = subprocess.run(["nm", "-D", "--defined-only", _native.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (spec_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    assert set(names) == set(_native.SIGNATURES), "binding signatures out of sync with the header"
    assert "spec_internal_set_error" not in exported


def test_checked_build_exports_the_same_calls(L):
    """The checked variant (index checks in the kernels) exports every call
    the header declares, like the default build."""
    _native.build()
    out = subprocess.run(["nm", "-D", "--defined-only", _native.CHECKED_LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (spec_\w+)", out))
    missing = [n for n in _declared() if n not in exported]
    assert not missing, f"declared but not exported by the checked build: {missing}"


def test_params_struct_layout_matches_header():
    prog = r"""
#include <stdio.h>
#include <stddef.h>
#include "spec_verify.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu\n", sizeof(spec_verify_params),
         offsetof(spec_verify_params, fly_window), offsetof(spec_verify_params, fly_theta),
         offsetof(spec_verify_params, reserved), offsetof(spec_verify_params, t_row_stride),
         offsetof(spec_verify_params, d_row_stride));
  return 0;
}
"""
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "t.c")
        exe = os.path.join(d, "t")
        open(c, "w").write(prog)
        subprocess.check_call(["gcc", "-I", os.path.dirname(HEADER), c, "-o", exe])
        got = list(map(int, subprocess.check_output([exe]).split()))
    P = _native.VerifyParams
    want = [ctypes.sizeof(P), P.fly_window.offset, P.fly_theta.offset, P.reserved.offset,
            P.t_row_stride.offset, P.d_row_stride.offset]
    assert got == want


def test_version_and_error_strings(L):
    assert L.spec_version().startswith(b"specverify")
    assert L.spec_last_error() is not None


def _params(**kw):
    base = dict(B=4, K=4, V=1024, dtype=sv.F32, mode="stochastic")
    base.update(kw)
    return sv.make_params(**base)


def test_workspace_size(L):
    p = _params()
    n = L.spec_workspace_size(ctypes.byref(p))
    assert n > 0 and n % 16 == 0
    big = L.spec_workspace_size(ctypes.byref(_params(B=400)))
    assert big > n
    assert L.spec_workspace_size(None) == 0
    assert L.spec_workspace_size(ctypes.byref(_params(K=0))) == 0
    assert L.spec_workspace_size(ctypes.byref(_params(V=1))) == 0
    assert L.spec_confidence_workspace_size(4, 4, 1024, sv.BF16) > 0
    assert L.spec_confidence_workspace_size(4, 4, 1024, 7) == 0


# Fake, non-null device addresses: every case below must be rejected by host
# validation before any pointer is used or any CUDA call is made.
_FAKE = 0x7f0000000000


def _call(L, p, zt=_FAKE, zd=_FAKE, x=_FAKE, u=_FAKE, out=_FAKE, acc=_FAKE, est=None, feat=None,
          conf=None, ws=_FAKE, ws_bytes=1 << 30):
    P = ctypes.c_void_p
    return L.spec_verify(ctypes.byref(p) if p is not None else None, P(zt), P(zd), P(x), P(u), P(out),
                         P(acc), None, P(est) if est else None, P(feat) if feat else None,
                         P(conf) if conf else None, P(ws), ctypes.c_size_t(ws_bytes), None)


@pytest.mark.parametrize("case,code", [
    ("null_params", 1), ("B0", 1), ("K0", 2), ("K32", 2), ("V1", 2), ("Vbig", 2), ("dtype", 2),
    ("mode", 2), ("reserved", 1), ("stride", 1), ("null_target", 1), ("null_tokens", 1),
    ("null_out", 1), ("stochastic_no_draft", 1), ("stochastic_no_u", 1), ("conf_no_est", 1),
    ("feature_no_draft", 1), ("fly_window0", 1), ("fly_theta_nan", 1), ("misaligned_f32", 1),
    ("ws_null", 1), ("ws_misaligned", 1), ("ws_small", 1),
])
def test_host_validation(L, case, code):
    p = _params()
    kw = {}
    if case == "null_params":
        p = None
    elif case == "B0":
        p.B = 0
    elif case == "K0":
        p.K = 0
    elif case == "K32":
        p.K = 32
    elif case == "V1":
        p.V = 1
    elif case == "Vbig":
        p.V = (1 << 20) + 1
    elif case == "dtype":
        p.dtype = 5
    elif case == "mode":
        p.mode = 9
    elif case == "reserved":
        p.reserved = 1
    elif case == "stride":
        p.t_row_stride = 1000
    elif case == "null_target":
        kw["zt"] = 0
    elif case == "null_tokens":
        kw["x"] = 0
    elif case == "null_out":
        kw["out"] = 0
    elif case == "stochastic_no_draft":
        kw["zd"] = 0
    elif case == "stochastic_no_u":
        kw["u"] = 0
    elif case == "conf_no_est":
        kw["conf"] = _FAKE
    elif case == "feature_no_draft":
        p.mode = sv.GREEDY
        kw.update(zd=0, feat=_FAKE)
    elif case == "fly_window0":
        p.mode = sv.FLY
        p.fly_window = 0
    elif case == "fly_theta_nan":
        p.mode = sv.FLY
        p.fly_theta = float("nan")
    elif case == "misaligned_f32":
        kw["zt"] = _FAKE + 2
    elif case == "ws_null":
        kw["ws"] = 0
    elif case == "ws_misaligned":
        kw["ws"] = _FAKE + 8
    elif case == "ws_small":
        kw["ws_bytes"] = 64
    rc = _call(L, p, **kw)
    assert rc == code
    assert L.spec_last_error()


def test_confidence_and_estimator_validation(L):
    P = ctypes.c_void_p
    assert L.spec_confidence(4, 0, 100, 0, P(_FAKE), 0, None, P(_FAKE), None, P(_FAKE), 1 << 20, None) == 2
    assert L.spec_confidence(4, 2, 100, 0, None, 0, None, P(_FAKE), None, P(_FAKE), 1 << 20, None) == 1
    assert L.spec_confidence(4, 2, 100, 0, P(_FAKE), 0, P(_FAKE), P(_FAKE), None, P(_FAKE), 1 << 20,
                             None) == 1          # est without conf
    assert L.spec_confidence(4, 2, 100, 0, P(_FAKE), 50, None, P(_FAKE), None, P(_FAKE), 1 << 20,
                             None) == 1          # stride < V
    assert L.spec_estimator_update(4, 0, P(_FAKE), P(_FAKE), P(_FAKE), 0.05, None, None, None) == 2
    assert L.spec_estimator_update(4, 2, P(_FAKE), P(_FAKE), None, 0.05, None, None, None) == 1
    assert L.spec_estimator_update(-1, 2, P(_FAKE), P(_FAKE), P(_FAKE), 0.05, None, None, None) == 1
    assert L.spec_estimator_update(4, 2, None, P(_FAKE), P(_FAKE), 0.05, None, None, None) == 1
    v = ctypes.c_int32()
    assert L.spec_get_device_status(None, ctypes.byref(v)) == 1


def test_irls_validation(L):
    P = ctypes.c_void_p
    assert L.spec_irls_state_size(0) == 0 and L.spec_irls_state_size(1025) == 0
    assert L.spec_irls_state_size(8) == (4 * 8 + 3) * 8
    assert L.spec_irls_reset(0, P(_FAKE), None) == 2
    assert L.spec_irls_reset(4, None, None) == 1
    assert L.spec_irls_accumulate(4, 0, P(_FAKE), P(_FAKE), P(_FAKE), P(_FAKE), None) == 2
    assert L.spec_irls_accumulate(-1, 2, P(_FAKE), P(_FAKE), P(_FAKE), P(_FAKE), None) == 1
    assert L.spec_irls_accumulate(4, 2, None, P(_FAKE), P(_FAKE), P(_FAKE), None) == 1
    assert L.spec_irls_accumulate(4, 2, P(_FAKE), P(_FAKE), None, P(_FAKE), None) == 1
    assert L.spec_irls_accumulate(4, 2, P(_FAKE), P(_FAKE), P(_FAKE), None, None) == 1
    assert L.spec_irls_accumulate(4, 2, P(_FAKE), P(_FAKE), P(_FAKE), P(_FAKE + 4), None) == 1   # misaligned
    assert L.spec_irls_refit(1025, P(_FAKE), P(_FAKE), 1.0, None, None) == 2
    assert L.spec_irls_refit(4, None, P(_FAKE), 1.0, None, None) == 1
    assert L.spec_irls_refit(4, P(_FAKE), None, 1.0, None, None) == 1
    assert L.spec_irls_refit(4, P(_FAKE), P(_FAKE), -1.0, None, None) == 1
    assert L.spec_irls_refit(4, P(_FAKE), P(_FAKE), float("nan"), None, None) == 1
    assert L.spec_irls_refit(4, P(_FAKE), P(_FAKE), float("inf"), None, None) == 1
    assert L.spec_last_error()


def test_av_and_ragged_validation(L):
    P = ctypes.c_void_p
    F = P(_FAKE)
    assert L.spec_av_budget(0, 4, F, F, F, F, F, None, None, None) == 1
    assert L.spec_av_budget(4, 0, F, F, F, F, F, None, None, None) == 1
    assert L.spec_av_budget(1024, 17, F, F, F, F, F, None, None, None) == 2      # B*K > 16384
    assert L.spec_av_budget(4, 4, None, F, F, F, F, None, None, None) == 1
    assert L.spec_av_budget(4, 4, F, F, F, None, F, None, None, None) == 1
    assert L.spec_av_budget(4, 4, F, F, F, F, None, None, None, None) == 1
    p = sv.make_params(4, 2, 1000, 1)
    assert L.spec_verify_ragged(ctypes.byref(p), F, F, F, None, F, F, F, None, None, None, None, F, 1 << 24,
                                None) == 1
    assert L.spec_verify_temperature(ctypes.byref(p), F, F, F, None, None, F, F, F, None, None, None, None, F,
                                     1 << 24, None) == 1                         # inv_temperature NULL
    assert b"inv_temperature" in L.spec_last_error()
    p.mode = 7
    assert L.spec_verify_temperature(ctypes.byref(p), F, F, F, None, F, F, F, F, None, None, None, None, F,
                                     1 << 24, None) == 2                         # unknown mode
    p.mode = 0
    assert L.spec_estimator_update_ragged(4, 2, F, F, None, F, 0.05, None, None, None) == 1
    assert L.spec_irls_accumulate_ragged(4, 2, F, F, None, F, F, None) == 1
    assert L.spec_ngram_draft(-1, 8, F, F, 1, 2, 4, F, F, None) == 1
    assert L.spec_ngram_draft(4, 8, F, F, 0, 2, 4, F, F, None) == 1
    assert L.spec_ngram_draft(4, 8, F, F, 3, 2, 4, F, F, None) == 1
    assert L.spec_ngram_draft(4, 8, F, F, 1, 2, 0, F, F, None) == 1
    assert L.spec_ngram_draft(4, 8, None, F, 1, 2, 4, F, F, None) == 1
    assert L.spec_ngram_draft(0, 8, None, None, 1, 2, 4, None, None, None) == 0
    assert L.spec_last_error() is not None


def test_missing_library_fails_loudly(monkeypatch):
    monkeypatch.setattr(_native, "_lib", None)
    monkeypatch.setattr(_native, "LIB_PATH", "/nonexistent/libspecverify.so")
    with pytest.raises(RuntimeError, match="missing"):
        _native.lib()


def test_python_binding_rejects_bad_tensors():
    import torch
    zt = torch.zeros((2, 3, 8))                      # CPU tensor: refused before the ABI
    with pytest.raises(ValueError):
        sv.verify(zt, None, torch.zeros((2, 2), dtype=torch.int32), None, mode="greedy")


@pytest.mark.parametrize("B", [(1 << 24) + 1, 1 << 25, 700_000_000])
def test_batches_beyond_the_limit_are_refused(L, B):
    """B > SPEC_MAX_B (2^24) is refused on the host, in every mode, before any
    pointer is used: the draw record of the stochastic rule packs the
    sequence index as 64 b + 2 n + bonus in a 32-bit int, which would
    overflow at B >= 2^25. spec_workspace_size returns 0 for such B."""
    for mode in ("stochastic", "greedy", "fly"):
        p = _params(B=B, K=1, V=2, mode=mode)
        assert L.spec_workspace_size(ctypes.byref(p)) == 0
        assert _call(L, p) == sv.api.SPEC_ERR_UNSUPPORTED
        assert b"B must be <=" in L.spec_last_error()
    assert L.spec_confidence_workspace_size(B, 1, 2, sv.F32) == 0
    ok = _params(B=1 << 24, K=1, V=2)
    assert L.spec_workspace_size(ctypes.byref(ok)) > 0


def test_wait_limit_hook_round_trips(L):
    prev = L.spec_debug_set_wait_limit(123)
    try:
        assert prev == 1 << 20
        assert L.spec_debug_set_wait_limit(0) == 123
    finally:
        L.spec_debug_set_wait_limit(prev)
    assert L.spec_debug_set_wait_limit(prev) == prev
