"""fp64 CPU oracle of the speculative-decoding verification pass.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s ``cpu_baseline`` / reference arm may import this package. The
product library (``speculative_decoding_token_verify_gb300``) never imports it
and shares no code with it.

The arithmetic lives in ``spec_oracle.c`` (plain C, double precision, loops in
ascending index order). This module only compiles it with gcc and marshals
numpy arrays through ctypes. Logits are passed either as ``float32`` arrays or
as ``uint16`` arrays holding raw bfloat16 bits.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_LIB = os.path.join(_HERE, "libspec_oracle.so")

F32, BF16 = 0, 1
STOCHASTIC, GREEDY, FLY = 0, 1, 2

FLAG_Q_ZERO = 1
FLAG_Z_ZERO = 2
FLAG_CDF_FALLBACK = 4
FLAG_REST_ZERO = 8
FLAG_BAD_ROW = 16
FLAG_NUCLEUS = 32

_lib = None


def build(force: bool = False) -> str:
    """Compile spec_oracle.c into a shared library next to it (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    _lib = bind(ctypes.CDLL(_LIB))
    return _lib


def bind(lib):
    """Declare the argument and result types of every oracle entry point on a
    loaded copy of the library (the one built here, or a test's variant)."""
    P = ctypes.c_void_p
    i32, i64, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.oracle_verify.argtypes = [i32, i32, i32, ctypes.c_int, ctypes.c_int, P, i64, P, i64,
                                  P, P, dbl, i32, P, P, P, P, P, P, P, P, P, P, P, P, dbl,
                                  P, P, P, P, P, ctypes.c_int]
    lib.oracle_verify.restype = ctypes.c_int
    lib.oracle_confidence.argtypes = [i32, i32, i32, ctypes.c_int, P, i64, P, P, P, P, ctypes.c_int]
    lib.oracle_confidence.restype = ctypes.c_int
    lib.oracle_estimator_update.argtypes = [i32, i32, P, P, P, P, dbl, P, P]
    lib.oracle_estimator_update.restype = ctypes.c_int
    lib.oracle_estimator_loss.argtypes = [i32, i32, P, P, P, P]
    lib.oracle_irls_accumulate.restype = ctypes.c_int
    lib.oracle_irls_accumulate.argtypes = [i32, i32, P, P, P, P, P, P, P]
    lib.oracle_ngram_draft.restype = ctypes.c_int
    lib.oracle_ngram_draft.argtypes = [i32, i32, P, P, i32, i32, i32, P, P]
    lib.oracle_av_budget.restype = ctypes.c_int
    lib.oracle_av_budget.argtypes = [i32, i32, P, P, P, P, P, P, P, P]
    lib.oracle_irls_refit.restype = ctypes.c_int
    lib.oracle_irls_refit.argtypes = [i32, P, P, P, dbl, P, P]
    lib.oracle_estimator_loss.restype = dbl
    lib.oracle_row_stats.argtypes = [i64, i32, ctypes.c_int, P, i64, P, P, P, P, ctypes.c_int]
    lib.oracle_row_stats.restype = ctypes.c_int
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _logits(z):
    z = np.ascontiguousarray(z)
    if z.dtype == np.float32:
        return z, F32
    if z.dtype == np.uint16:
        return z, BF16
    raise TypeError(f"logits must be float32 or uint16 (raw bf16 bits), got {z.dtype}")


def verify(zt, zd, x, u, mode=STOCHASTIC, fly_theta=0.3, fly_window=6, est_params=None,
           nthreads=1, want_cdf=False, draft_len=None, inv_temp=None, top_p=1.0, force=None,
           nuc_shift=None):
    """Verify B sequences. zt [B,K+1,V], zd [B,K,V] or None, x [B,K] int32,
    u [B,K+1] float32 or None, draft_len [B] int32 in [0, K] or None (drafts
    submitted for verification per sequence; None: all K), inv_temp [B]
    float32 > 0 or None (per-sequence inverse sampling temperature), top_p in
    (0, 1] (nucleus truncation of every processed row; 1: none).

    Returns a dict of numpy arrays: out_tokens [B,K+1] int32, accepted_len [B],
    pos_stats [B,K+1,4] (lse_t, h_t, log_ratio, f), feature [B,K], conf [B,K]
    (NaN without est_params), margin_acc [B] (acceptance / FLy-gate margin),
    margin_cdf [B] (margin of the final draw), margin [B] (the smaller of the
    two), flags [B], and with want_cdf the normalised running sum of each
    final draw's weights, cdf [B,V].

    Per-position report (for parity checks of a computation that decided a
    position in doubt the other way): margin_pos [B,K] (the margin of each
    decision the scan takes, +inf where none is taken), natural_pos [B,K]
    (the rule's decision there: 1 accept / gate open, 0 reject / gate
    closed, -1 none), nuc_doubt [B,2K+1] (top-p: bit 1 the group at a row's
    z* may be dropped, bit 2 the next group down may be added; rows are
    target 0..K, then draft 0..K-1). Overrides: force [B,K] int (-1: the
    rule; 0/1: that decision where the scan reaches the position), nuc_shift
    [B,2K+1] int (0: the natural nucleus boundary; -1 / +1: one tie group
    up / down).
    """
    lib = _load()
    zt, dt = _logits(zt)
    B, K1, V = zt.shape
    K = K1 - 1
    if zd is not None:
        zd, dd = _logits(zd)
        assert dd == dt and zd.shape == (B, K, V)
    x = np.ascontiguousarray(x, dtype=np.int32)
    assert x.shape == (B, K)
    if u is not None:
        u = np.ascontiguousarray(u, dtype=np.float32)
        assert u.shape == (B, K + 1)
    est = None if est_params is None else np.ascontiguousarray(est_params, dtype=np.float64)
    out = dict(
        out_tokens=np.empty((B, K + 1), np.int32),
        accepted_len=np.empty(B, np.int32),
        pos_stats=np.empty((B, K + 1, 4), np.float64),
        feature=np.full((B, K), np.nan),
        conf=np.full((B, K), np.nan),
        margin_acc=np.empty(B, np.float64),
        margin_cdf=np.empty(B, np.float64),
        flags=np.empty(B, np.int32),
        margin_pos=np.empty((B, K), np.float64),
        natural_pos=np.empty((B, K), np.int32),
        nuc_doubt=np.empty((B, 2 * K + 1), np.int32),
    )
    if force is not None:
        force = np.ascontiguousarray(force, dtype=np.int32)
        assert force.shape == (B, K)
    if nuc_shift is not None:
        nuc_shift = np.ascontiguousarray(nuc_shift, dtype=np.int32)
        assert nuc_shift.shape == (B, 2 * K + 1)
    cdf = np.full((B, V), np.nan) if want_cdf else None
    if draft_len is not None:
        draft_len = np.ascontiguousarray(draft_len, dtype=np.int32)
        assert draft_len.shape == (B,)
    if inv_temp is not None:
        inv_temp = np.ascontiguousarray(inv_temp, dtype=np.float32)
        assert inv_temp.shape == (B,)
    rc = lib.oracle_verify(B, K, V, dt, mode, _ptr(zt), V, _ptr(zd), V, _ptr(x), _ptr(u),
                           float(fly_theta), int(fly_window), _ptr(est),
                           _ptr(out["out_tokens"]), _ptr(out["accepted_len"]),
                           _ptr(out["pos_stats"]), _ptr(out["conf"]) if est is not None else None,
                           _ptr(out["feature"]) if zd is not None else None,
                           _ptr(out["margin_acc"]), _ptr(out["margin_cdf"]), _ptr(cdf),
                           _ptr(out["flags"]), _ptr(draft_len), _ptr(inv_temp), float(top_p),
                           _ptr(force), _ptr(nuc_shift), _ptr(out["margin_pos"]), _ptr(out["natural_pos"]),
                           _ptr(out["nuc_doubt"]), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_verify rejected its arguments")
    out["margin"] = np.minimum(out["margin_acc"], out["margin_cdf"])
    if want_cdf:
        out["cdf"] = cdf
    return out


def confidence(zd, est_params=None, nthreads=1):
    """feature [B,K] = logit(q_max) of each draft row; conf [B,K] if est_params."""
    lib = _load()
    zd, dt = _logits(zd)
    B, K, V = zd.shape
    est = None if est_params is None else np.ascontiguousarray(est_params, dtype=np.float64)
    feat = np.empty((B, K), np.float64)
    conf = np.full((B, K), np.nan)
    flags = np.empty(B, np.int32)
    rc = lib.oracle_confidence(B, K, V, dt, _ptr(zd), V, _ptr(est), _ptr(feat),
                               _ptr(conf) if est is not None else None, _ptr(flags), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_confidence rejected its arguments")
    return feat, conf, flags


def _draft_len(draft_len, B):
    if draft_len is None:
        return None
    d = np.ascontiguousarray(draft_len, dtype=np.int32)
    assert d.shape == (B,)
    return d


def estimator_update(feature, accepted_len, params, lr, draft_len=None):
    """One gradient step; returns (new_params [K+1], grad [K+1], counts [K+1])."""
    lib = _load()
    f = np.ascontiguousarray(feature, dtype=np.float64)
    B, K = f.shape
    n = np.ascontiguousarray(accepted_len, dtype=np.int32)
    dl = _draft_len(draft_len, B)
    p = np.array(params, dtype=np.float64, copy=True)
    assert p.shape == (K + 1,)
    g = np.empty(K + 1, np.float64)
    c = np.empty(K + 1, np.int64)
    rc = lib.oracle_estimator_update(B, K, _ptr(f), _ptr(n), _ptr(dl), _ptr(p), float(lr), _ptr(g), _ptr(c))
    if rc != 0:
        raise ValueError("oracle_estimator_update rejected its arguments")
    return p, g, c


def estimator_loss(feature, accepted_len, params, draft_len=None):
    lib = _load()
    f = np.ascontiguousarray(feature, dtype=np.float64)
    B, K = f.shape
    n = np.ascontiguousarray(accepted_len, dtype=np.int32)
    p = np.ascontiguousarray(params, dtype=np.float64)
    return lib.oracle_estimator_loss(B, K, _ptr(f), _ptr(n), _ptr(_draft_len(draft_len, B)), _ptr(p))


def irls_zero(K):
    """An empty IRLS round: (g [K+1], H [K+1, K+1], n [K+1])."""
    return np.zeros(K + 1), np.zeros((K + 1, K + 1)), np.zeros(K + 1, np.int64)


def irls_accumulate(feature, accepted_len, params, state, draft_len=None):
    """Add one decoding step's labels to an IRLS round ``state`` (in place)."""
    lib = _load()
    f = np.ascontiguousarray(feature, dtype=np.float64)
    B, K = f.shape
    nacc = np.ascontiguousarray(accepted_len, dtype=np.int32)
    dl = _draft_len(draft_len, B)
    p = np.ascontiguousarray(params, dtype=np.float64)
    g, H, n = state
    assert g.shape == (K + 1,) and H.shape == (K + 1, K + 1) and n.shape == (K + 1,)
    assert g.flags.c_contiguous and H.flags.c_contiguous and n.flags.c_contiguous
    rc = lib.oracle_irls_accumulate(B, K, _ptr(f), _ptr(nacc), _ptr(dl), _ptr(p), _ptr(g), _ptr(H), _ptr(n))
    if rc != 0:
        raise ValueError("oracle_irls_accumulate rejected its arguments")
    return state


def irls_refit(state, params, damping):
    """Refit at the end of a round; returns (new_params [K+1], applied step [K+1])."""
    lib = _load()
    g, H, n = state
    K = g.shape[0] - 1
    p = np.array(params, dtype=np.float64, copy=True)
    step = np.empty(K + 1, np.float64)
    rc = lib.oracle_irls_refit(K, _ptr(g), _ptr(H), _ptr(n), float(damping), _ptr(p), _ptr(step))
    if rc != 0:
        raise ValueError("oracle_irls_refit rejected its arguments (%d)" % rc)
    return p, step


def ngram_draft(ctx, lengths, n_min, n_max, K):
    """Prompt-lookup drafts: returns (draft_tokens [B,K] int32, -1 padded;
    draft_len [B] int32)."""
    lib = _load()
    c = np.ascontiguousarray(ctx, dtype=np.int32)
    B, ld = c.shape
    ln = np.ascontiguousarray(lengths, dtype=np.int32)
    assert ln.shape == (B,)
    toks = np.empty((B, K), np.int32)
    dl = np.empty(B, np.int32)
    rc = lib.oracle_ngram_draft(B, ld, _ptr(c), _ptr(ln), int(n_min), int(n_max), int(K), _ptr(toks), _ptr(dl))
    if rc != 0:
        raise ValueError("oracle_ngram_draft rejected its arguments")
    return toks, dl


def av_budget(conf, draft_cost, verify_cost):
    """Adaptive-verification pruning: returns a dict with draft_len [B] int32,
    budget (int), survival [B,K] float32, objective [B*K+1] and gap (relative
    gap between the best and second-best objective)."""
    lib = _load()
    c = np.ascontiguousarray(conf, dtype=np.float32)
    B, K = c.shape
    dc = np.ascontiguousarray(draft_cost, dtype=np.float32)
    vc = np.ascontiguousarray(verify_cost, dtype=np.float32)
    assert dc.shape == (B * K + 1,) and vc.shape == (B * K + 1,)
    dl = np.empty(B, np.int32)
    bud = np.zeros(1, np.int32)
    sv = np.empty((B, K), np.float32)
    obj = np.empty(B * K + 1, np.float32)
    gap = np.zeros(1, np.float64)
    rc = lib.oracle_av_budget(B, K, _ptr(c), _ptr(dc), _ptr(vc), _ptr(dl), _ptr(bud), _ptr(sv), _ptr(obj),
                              _ptr(gap))
    if rc != 0:
        raise ValueError("oracle_av_budget rejected its arguments")
    return dict(draft_len=dl, budget=int(bud[0]), survival=sv, objective=obj, gap=float(gap[0]))


def row_stats(z, nthreads=1):
    """Per-row (lse, normalised entropy, argmax, logit(q_max)) of z [..., V]."""
    lib = _load()
    z, dt = _logits(z)
    V = z.shape[-1]
    rows = int(np.prod(z.shape[:-1]))
    lse = np.empty(rows, np.float64)
    h = np.empty(rows, np.float64)
    am = np.empty(rows, np.int32)
    fq = np.empty(rows, np.float64)
    rc = lib.oracle_row_stats(rows, V, dt, _ptr(z), V, _ptr(lse), _ptr(h), _ptr(am), _ptr(fq),
                              int(nthreads))
    if rc != 0:
        raise ValueError("oracle_row_stats rejected its arguments")
    shp = z.shape[:-1]
    return lse.reshape(shp), h.reshape(shp), am.reshape(shp), fq.reshape(shp)
