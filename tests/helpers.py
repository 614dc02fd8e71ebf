"""Shared helpers: run the CUDA path and the oracle on the same seeded bytes
and compare them under the tolerances stated in the design notes.

Tolerances (token ids and accepted lengths are exact):
* a sequence whose oracle acceptance margin |u_i - min(1, p/q)| (FLy: |h - theta|)
  is below FLAG_MARGIN (1e-5) is "flagged": its accepted length may differ;
* a final inverse-CDF draw whose u lies within FLAG_MARGIN of a boundary of
  the oracle's CDF is "flagged": the GPU's token may differ from the oracle's,
  but must still be valid, i.e. its interval in the oracle's fp64 CDF lies
  within FLAG_MARGIN of u;
* log-domain values (lse, log-ratio, logit(q_max)):
  |gpu - oracle| <= tol * max(1, |oracle|);
* normalised entropy and confidence: |gpu - oracle| <= tol * max(|oracle|, 0.1);
  tol = 1e-5 for fp32 logits, 2e-3 for bf16 logits.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads

FLAG_MARGIN = 1e-5


def tol_for(dtype) -> float:
    return 2e-3 if dtype in ("bf16", torch.bfloat16) else 1e-5


def oracle_run(inp, mode, fly_theta=0.3, fly_window=6, est=None, with_draft=True, nthreads=8, draft_len=None,
               inv_temp=None, top_p=1.0):
    zt = workloads.to_numpy_logits(inp["zt"])
    zd = workloads.to_numpy_logits(inp["zd"]) if with_draft else None
    x = inp["x"].cpu().numpy()
    u = inp["u"].cpu().numpy() if mode == oracle.STOCHASTIC else None
    r = oracle.verify(zt, zd, x, u, mode=mode, fly_theta=fly_theta, fly_window=fly_window,
                      est_params=None if est is None else np.asarray(est, np.float64),
                      nthreads=nthreads, want_cdf=mode == oracle.STOCHASTIC, draft_len=draft_len,
                      inv_temp=inv_temp, top_p=top_p)
    if u is not None:
        r["u_final"] = u[:, -1].astype(np.float64)
    return r


def _close_log(g, r, tol):
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    both_nan = (np.isnan(g) & np.isnan(r)) | (g == r)      # equal infinities match
    err = np.abs(g - r)
    lim = tol * np.maximum(1.0, np.abs(r))
    bad = ~both_nan & ~(err <= lim)
    return bad, np.nanmax(np.where(both_nan, 0.0, err / lim)) if g.size else 0.0


def _close_unit(g, r, tol):
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    both_nan = (np.isnan(g) & np.isnan(r)) | (g == r)
    err = np.abs(g - r)
    lim = tol * np.maximum(np.abs(r), 0.1)
    bad = ~both_nan & ~(err <= lim)
    return bad, np.nanmax(np.where(both_nan, 0.0, err / lim)) if g.size else 0.0


def compare(gpu: dict, ref: dict, dtype, check_pos_stats=True, check_feature=False,
            check_conf=False, flag_margin=FLAG_MARGIN, max_flagged_frac=0.02, doubt_frac=None):
    """Assert parity; returns a summary dict (flagged counts, mismatches, worst
    float error as a fraction of its tolerance).

    doubt_frac (top-p): sequences whose nucleus boundary the oracle marks as
    in doubt (flag FLAG_NUCLEUS) may differ in their floats, since the GPU may
    place that boundary one tie group off; at most max(1, doubt_frac * the
    number of such sequences) of them may, and every other sequence must meet
    the tolerances."""
    tol = tol_for(dtype)
    n_g = gpu["accepted_len"].cpu().numpy()
    t_g = gpu["out_tokens"].cpu().numpy()
    n_r = ref["accepted_len"]
    t_r = ref["out_tokens"]
    B, K1 = t_r.shape
    acc_flag = ref["margin_acc"] < flag_margin
    cdf_flag = ref["margin_cdf"] < flag_margin
    # accepted length and accepted prefix: exact unless the acceptance is flagged
    pre_bad = np.array([n_g[b] != n_r[b] or (t_g[b, :n_r[b]] != t_r[b, :n_r[b]]).any()
                        or (t_g[b, n_r[b] + 1:] != -1).any() for b in range(B)])
    bad = pre_bad & ~acc_flag
    assert not bad.any(), (
        f"{int(bad.sum())} unflagged sequences differ, e.g. b={int(np.flatnonzero(bad)[0])}: "
        f"gpu n={n_g[bad][0]} toks={t_g[bad][0]} vs oracle n={n_r[bad][0]} toks={t_r[bad][0]}")
    # the final token: exact, or valid within the flag margin of the oracle's CDF
    same_n = ~pre_bad
    fin_g = t_g[np.arange(B), np.minimum(n_r, K1 - 1)]
    fin_r = t_r[np.arange(B), n_r]
    tok_diff = same_n & (fin_g != fin_r)
    bad = tok_diff & ~cdf_flag
    assert not bad.any(), (
        f"{int(bad.sum())} unflagged final tokens differ, e.g. b={int(np.flatnonzero(bad)[0])}: "
        f"gpu {fin_g[bad][0]} vs oracle {fin_r[bad][0]} (margin {ref['margin_cdf'][bad][0]:.3g})")
    for b in np.flatnonzero(tok_diff):
        c = ref["cdf"][b]
        v = int(fin_g[b])
        assert 0 <= v < c.shape[0], f"b={b}: token {v} out of range"
        lo = c[v - 1] if v > 0 else 0.0
        hi = c[v]
        uu = ref["u_final"][b]
        assert lo - flag_margin <= uu <= hi + flag_margin, (
            f"b={b}: gpu token {v} has oracle interval [{lo}, {hi}) far from u={uu}")
    assert acc_flag.sum() <= max(1, max_flagged_frac * B), (
        f"too many acceptance-flagged sequences: {int(acc_flag.sum())} of {B}")
    summary = dict(B=B, flagged_accept=int(acc_flag.sum()), flagged_cdf=int(cdf_flag.sum()),
                   mismatched=int((pre_bad | tok_diff).sum()), token_diff_flagged=int(tok_diff.sum()))
    doubt = np.zeros(B, bool)
    if doubt_frac is not None:
        doubt = (ref["flags"] & oracle.FLAG_NUCLEUS) != 0
        summary["nucleus_doubt"] = int(doubt.sum())
    float_bad_doubt = np.zeros(B, bool)

    def _check(bad, name):
        per_seq = bad.reshape(B, -1).any(1)
        assert not (per_seq & ~doubt).any(), f"{name} out of tolerance at {np.argwhere(bad)[:3].tolist()}"
        float_bad_doubt[:] |= per_seq & doubt

    if check_pos_stats:
        ps = gpu["pos_stats"].cpu().numpy()
        rp = ref["pos_stats"]
        for k, (name, fn) in enumerate((("lse", _close_log), ("entropy", _close_unit),
                                        ("log_ratio", _close_log), ("feature", _close_log))):
            bad, worst = fn(ps[..., k], rp[..., k], tol)
            _check(bad, f"pos_stats[{name}]")
            summary[f"worst_{name}"] = float(worst)
    if check_feature:
        bad, worst = _close_log(gpu["feature"].cpu().numpy(), ref["feature"], tol)
        _check(bad, "feature")
        summary["worst_feature_out"] = float(worst)
    if check_conf:
        bad, worst = _close_unit(gpu["conf"].cpu().numpy(), ref["conf"], tol)
        _check(bad, "conf")
        summary["worst_conf"] = float(worst)
    if doubt_frac is not None:
        nb = int(float_bad_doubt.sum())
        summary["nucleus_doubt_float_diff"] = nb
        assert nb <= max(1, doubt_frac * doubt.sum()), (
            f"{nb} of {int(doubt.sum())} sequences with a nucleus boundary in doubt differ in their floats")
    return summary
