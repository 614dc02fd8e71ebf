"""Shared helpers: run the CUDA path and the oracle on the same seeded bytes
and compare them under the tolerances stated in the design notes.

Tolerances (token ids and accepted lengths are exact):
* a sequence whose oracle decision margin is below FLAG_MARGIN (1e-5) is
  "flagged": its tokens may differ, and every mismatch must be flagged;
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


def oracle_run(inp, mode, fly_theta=0.3, fly_window=6, est=None, with_draft=True, nthreads=8):
    zt = workloads.to_numpy_logits(inp["zt"])
    zd = workloads.to_numpy_logits(inp["zd"]) if with_draft else None
    x = inp["x"].cpu().numpy()
    u = inp["u"].cpu().numpy() if mode == oracle.STOCHASTIC else None
    return oracle.verify(zt, zd, x, u, mode=mode, fly_theta=fly_theta, fly_window=fly_window,
                         est_params=None if est is None else np.asarray(est, np.float64),
                         nthreads=nthreads)


def _close_log(g, r, tol):
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    both_nan = np.isnan(g) & np.isnan(r)
    err = np.abs(g - r)
    lim = tol * np.maximum(1.0, np.abs(r))
    bad = ~both_nan & ~(err <= lim)
    return bad, np.nanmax(np.where(both_nan, 0.0, err / lim)) if g.size else 0.0


def _close_unit(g, r, tol):
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    both_nan = np.isnan(g) & np.isnan(r)
    err = np.abs(g - r)
    lim = tol * np.maximum(np.abs(r), 0.1)
    bad = ~both_nan & ~(err <= lim)
    return bad, np.nanmax(np.where(both_nan, 0.0, err / lim)) if g.size else 0.0


def compare(gpu: dict, ref: dict, dtype, check_pos_stats=True, check_feature=False,
            check_conf=False, flag_margin=FLAG_MARGIN, max_flagged_frac=0.05):
    """Assert parity; returns a summary dict (flagged count, worst float error
    as a fraction of its tolerance)."""
    tol = tol_for(dtype)
    n_g = gpu["accepted_len"].cpu().numpy()
    t_g = gpu["out_tokens"].cpu().numpy()
    flagged = ref["margin"] < flag_margin
    mism = (n_g != ref["accepted_len"]) | (t_g != ref["out_tokens"]).any(1)
    unexplained = mism & ~flagged
    assert not unexplained.any(), (
        f"{int(unexplained.sum())} unflagged sequences differ, e.g. b={int(np.flatnonzero(unexplained)[0])}: "
        f"gpu n={n_g[unexplained][0]} toks={t_g[unexplained][0]} vs oracle n="
        f"{ref['accepted_len'][unexplained][0]} toks={ref['out_tokens'][unexplained][0]}")
    assert flagged.mean() <= max_flagged_frac, f"too many flagged sequences: {flagged.mean():.3f}"
    summary = dict(B=len(n_g), flagged=int(flagged.sum()), mismatched=int(mism.sum()))
    if check_pos_stats:
        ps = gpu["pos_stats"].cpu().numpy()
        rp = ref["pos_stats"]
        for k, (name, fn) in enumerate((("lse", _close_log), ("entropy", _close_unit),
                                        ("log_ratio", _close_log), ("feature", _close_log))):
            bad, worst = fn(ps[..., k], rp[..., k], tol)
            assert not bad.any(), f"pos_stats[{name}] out of tolerance at {np.argwhere(bad)[:3].tolist()}"
            summary[f"worst_{name}"] = float(worst)
    if check_feature:
        bad, worst = _close_log(gpu["feature"].cpu().numpy(), ref["feature"], tol)
        assert not bad.any(), "feature out of tolerance"
        summary["worst_feature_out"] = float(worst)
    if check_conf:
        bad, worst = _close_unit(gpu["conf"].cpu().numpy(), ref["conf"], tol)
        assert not bad.any(), "conf out of tolerance"
        summary["worst_conf"] = float(worst)
    return summary
