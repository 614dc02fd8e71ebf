"""Shared helpers: run the CUDA path and the oracle on the same seeded bytes
and compare them under the tolerances stated in the design notes.

The parity rule ("Speculative Decoding: ...", "Математика верификации": accept
x_i iff u_i < min(1, p(x_i)/q(x_i)); "Training-Free Loosely Speculative
Decoding", 2.A.1: the gate reads h_j >= theta). The GPU decides in fp32 and
the oracle in fp64, so a decision whose oracle margin is below FLAG_MARGIN
(1e-5) may go either way. Every sequence whose GPU result differs from the
oracle's is checked completely:

* the oracle is re-run on that sequence with the GPU's decisions imposed
  (stochastic: accept before the GPU's stop, reject at it; FLy: the gates
  before the stop open, the one at the stop as the rule or closed), and with
  a top-p nucleus boundary moved one tie group where the oracle says it is in
  doubt that way;
* every imposed decision that differs from the rule's own must lie within
  the flag margin there, and the re-run must reproduce the GPU's accepted
  length and prefix exactly;
* the GPU's final token must be the re-run's, or lie within the flag margin
  of u in the re-run's fp64 CDF of the stop row the GPU chose;
* every float must meet its tolerance against the re-run.

Sequences that differ are counted; a test bounds their number. Floats:
* log-domain values (lse, log-ratio, logit(q_max)):
  |gpu - oracle| <= tol * max(1, |oracle|);
* normalised entropy and confidence: |gpu - oracle| <= tol * max(|oracle|, 0.1);
  tol = 1e-5 for fp32 logits, 2e-3 for bf16 logits. The plain relative
  error of h and conf (rows where the oracle's value is above 1e-30) is
  reported as well.

Outputs and workspaces handed to the GPU are filled with a poison pattern
first (bytes 0x7F: the int 2139062143, the float 3.4e38), so an entry the
library never writes cannot pass.
"""
from __future__ import annotations

import itertools

import numpy as np
import torch

import oracle
import speculative_decoding_token_verify_gb300 as sv
import workloads

FLAG_MARGIN = 1e-5
POISON_I32 = 0x7F7F7F7F


def tol_for(dtype) -> float:
    return 2e-3 if dtype in ("bf16", torch.bfloat16) else 1e-5


# ---------------------------------------------------------------------------
# poisoned outputs
# ---------------------------------------------------------------------------

def poison_i32(shape, device):
    return torch.full(shape, POISON_I32, dtype=torch.int32, device=device)


def poison_f32(shape, device):
    return poison_i32(shape, device).view(torch.float32)


def poisoned_workspace(nbytes, device):
    ws = sv.Workspace(device)
    ws.buf = torch.full((max(int(nbytes), 16),), 0x7F, dtype=torch.uint8, device=device)
    return ws


def verify(target_logits, draft_logits, draft_tokens, uniforms, mode="stochastic", fly_theta=0.3, fly_window=6,
           want_pos_stats=False, want_feature=False, want_conf=False, **kw):
    """sv.verify with every output and the workspace poisoned beforehand."""
    zt = target_logits
    dev = zt.device
    B, K1, V = zt.shape
    K = K1 - 1
    out = {"out_tokens": poison_i32((B, K1), dev), "accepted_len": poison_i32((B,), dev)}
    if want_pos_stats:
        out["pos_stats"] = poison_f32((B, K1, 4), dev)
    if want_feature:
        out["feature"] = poison_f32((B, K), dev)
    if want_conf:
        out["conf"] = poison_f32((B, K), dev)
    if "workspace" not in kw:
        p = sv.api.make_params(B, K, V, sv.api._dtype_code(zt), mode, fly_theta, fly_window)
        kw["workspace"] = poisoned_workspace(sv.api.workspace_size(p), dev)
    return sv.verify(zt, draft_logits, draft_tokens, uniforms, mode=mode, fly_theta=fly_theta,
                     fly_window=fly_window, want_pos_stats=want_pos_stats, want_feature=want_feature,
                     want_conf=want_conf, out=out, **kw)


def confidence(draft_logits, est_params=None, **kw):
    """sv.confidence with its outputs and workspace poisoned beforehand."""
    B, K, V = draft_logits.shape
    dev = draft_logits.device
    out = {"feature": poison_f32((B, K), dev)}
    if est_params is not None:
        out["conf"] = poison_f32((B, K), dev)
    if "workspace" not in kw:
        n = sv.api._native.lib().spec_confidence_workspace_size(B, K, V, sv.api._dtype_code(draft_logits))
        kw["workspace"] = poisoned_workspace(n, dev)
    return sv.confidence(draft_logits, est_params, out=out, **kw)


# ---------------------------------------------------------------------------
# the oracle
# ---------------------------------------------------------------------------

def oracle_run(inp, mode, fly_theta=0.3, fly_window=6, est=None, with_draft=True, nthreads=8, draft_len=None,
               inv_temp=None, top_p=1.0):
    zt = workloads.to_numpy_logits(inp["zt"])
    zd = workloads.to_numpy_logits(inp["zd"]) if with_draft else None
    x = inp["x"].cpu().numpy()
    u = inp["u"].cpu().numpy() if mode == oracle.STOCHASTIC else None
    est_np = None if est is None else np.asarray(est, np.float64)
    dl = None if draft_len is None else np.asarray(draft_len, np.int32)
    it = None if inv_temp is None else np.asarray(inv_temp, np.float32)
    kw = dict(mode=mode, fly_theta=fly_theta, fly_window=fly_window, est_params=est_np,
              want_cdf=mode == oracle.STOCHASTIC, top_p=top_p)
    r = oracle.verify(zt, zd, x, u, nthreads=nthreads, draft_len=dl, inv_temp=it, **kw)
    if u is not None:
        r["u_final"] = u[:, -1].astype(np.float64)
    r["mode"] = mode
    r["draft_len"] = dl if dl is not None else np.full(x.shape[0], x.shape[1], np.int32)

    def rerun(b, force=None, nuc_shift=None):
        s = slice(b, b + 1)
        rr = oracle.verify(zt[s], None if zd is None else zd[s], x[s], None if u is None else u[s], nthreads=1,
                           draft_len=None if dl is None else dl[s], inv_temp=None if it is None else it[s],
                           force=None if force is None else np.asarray(force, np.int32)[None],
                           nuc_shift=None if nuc_shift is None else np.asarray(nuc_shift, np.int32)[None], **kw)
        return rr

    r["_rerun"] = rerun
    return r


# ---------------------------------------------------------------------------
# comparison
# ---------------------------------------------------------------------------

def _err_log(g, r, tol):
    """Error of g against r as a multiple of its log-domain tolerance
    (0 where both are NaN or equal, e.g. equal infinities)."""
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    same = (np.isnan(g) & np.isnan(r)) | (g == r)
    with np.errstate(invalid="ignore"):
        e = np.abs(g - r) / (tol * np.maximum(1.0, np.abs(r)))
    return np.where(same, 0.0, np.where(np.isnan(e), np.inf, e))


def _err_unit(g, r, tol):
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    same = (np.isnan(g) & np.isnan(r)) | (g == r)
    with np.errstate(invalid="ignore"):
        e = np.abs(g - r) / (tol * np.maximum(np.abs(r), 0.1))
    return np.where(same, 0.0, np.where(np.isnan(e), np.inf, e))


def _rel(g, r, floor=1e-30):
    """Largest plain relative error |g - r| / |r| over entries with |r| > floor."""
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    m = np.isfinite(r) & (np.abs(r) > floor) & np.isfinite(g)
    return float((np.abs(g[m] - r[m]) / np.abs(r[m])).max()) if m.any() else 0.0


class _Floats:
    """The float outputs under check, per sequence, as multiples of their tolerance."""

    def __init__(self, gpu, tol, check_pos_stats, check_feature, check_conf):
        self.tol = tol
        self.items = []
        if check_pos_stats:
            ps = gpu["pos_stats"].cpu().numpy()
            for k, (name, fn) in enumerate((("lse", _err_log), ("entropy", _err_unit),
                                            ("log_ratio", _err_log), ("feature", _err_log))):
                self.items.append((f"pos_stats[{name}]", ps[..., k], lambda r, k=k: r["pos_stats"][..., k], fn))
        if check_feature:
            self.items.append(("feature", gpu["feature"].cpu().numpy(), lambda r: r["feature"], _err_log))
        if check_conf:
            self.items.append(("conf", gpu["conf"].cpu().numpy(), lambda r: r["conf"], _err_unit))

    def errors(self, ref, rows=None):
        """{name: error array [n, ...]} of the GPU sequences `rows` (all if
        None) against ref (whose first axis matches)."""
        out = {}
        for name, g, get, fn in self.items:
            gg = g if rows is None else g[rows]
            out[name] = fn(gg, get(ref), self.tol)
        return out

    @staticmethod
    def seq_ok(errs):
        B = next(iter(errs.values())).shape[0] if errs else 0
        ok = np.ones(B, bool)
        for e in errs.values():
            ok &= (e.reshape(B, -1) <= 1.0).all(1)
        return ok


def _final_ok(tok, rr_tok, cdf, uu, flag_margin):
    """The final token equals the reference's, or its interval in the fp64
    CDF of the same draw lies within the flag margin of u."""
    if tok == rr_tok:
        return True
    if cdf is None or not (0 <= tok < cdf.shape[0]):
        return False
    lo = cdf[tok - 1] if tok > 0 else 0.0
    return lo - flag_margin <= uu <= cdf[tok] + flag_margin


def _forces(mode, n_g, K, kb):
    """Decision paths to impose for a GPU accepted length n_g."""
    if mode == oracle.STOCHASTIC:
        f = np.full(K, -1, np.int32)
        f[:n_g] = 1
        if n_g < kb:
            f[n_g] = 0
        return [f]
    if mode == oracle.FLY:
        f = np.full(K, -1, np.int32)
        f[:n_g] = 1
        out = [f]
        if n_g < kb:
            f2 = f.copy()
            f2[n_g] = 0
            out.append(f2)
        return out
    return [None]   # greedy: integer decisions, nothing to impose


def _resolve(b, gpu_np, ref, floats, flag_margin, tol):
    """Check a sequence whose GPU result differs from the oracle's: is it the
    oracle's result along some decision path that differs only at positions
    in doubt (and, under top-p, for some nucleus boundaries in doubt)?
    Returns None if so, else a description of the failure."""
    n_all, t_all = gpu_np
    n_g = int(n_all[b])
    t_g = t_all[b]
    K = t_g.shape[0] - 1
    kb = int(ref["draft_len"][b])
    mode = ref["mode"]
    if not (0 <= n_g <= kb):
        return f"accepted length {n_g} outside [0, {kb}]"
    # nucleus boundaries in doubt: pick, row by row, a placement that the
    # GPU's floats agree with (rows' statistics depend on their own boundary)
    doubt = ref["nuc_doubt"][b] if "nuc_doubt" in ref else np.zeros(2 * K + 1, np.int32)
    shifts = np.zeros(2 * K + 1, np.int32)
    if doubt.any():
        alts = {}
        for sgn, bit in ((-1, 1), (1, 2)):
            sv_ = np.where((doubt & bit) != 0, sgn, 0).astype(np.int32)
            if sv_.any():
                alts[sgn] = ref["_rerun"](b, nuc_shift=sv_)
        base = floats.errors({k: v[b:b + 1] for k, v in ref.items() if isinstance(v, np.ndarray)}, rows=[b])
        for row in np.flatnonzero(doubt):
            def row_ok(errs):
                ok = True
                for name, e in errs.items():
                    e = e[0]
                    if name.startswith("pos_stats"):
                        if row <= K and name in ("pos_stats[lse]", "pos_stats[entropy]"):
                            ok &= bool((e[row] <= 1.0).all())
                        if row > K and name == "pos_stats[feature]":
                            ok &= bool((e[row - K - 1] <= 1.0).all())
                    elif row > K:
                        ok &= bool((e[row - K - 1] <= 1.0).all())
                return ok
            if row_ok(base):
                continue
            for sgn, rr in alts.items():
                if doubt[row] & (1 if sgn < 0 else 2) and row_ok(floats.errors(rr, rows=[b])):
                    shifts[row] = sgn
                    break
            else:
                return f"row {row}: floats match no placement of its nucleus boundary in doubt"
    fails = []
    for force in _forces(mode, n_g, K, kb):
        rr = ref["_rerun"](b, force=force, nuc_shift=shifts if shifts.any() else None)
        why = None
        if int(rr["accepted_len"][0]) != n_g:
            why = f"imposed path gives n={int(rr['accepted_len'][0])}, gpu n={n_g}"
        elif (rr["out_tokens"][0, :n_g] != t_g[:n_g]).any() or (t_g[n_g + 1:] != -1).any():
            why = "prefix or padding differs"
        else:
            if force is not None:
                imp = (force >= 0) & (rr["natural_pos"][0] >= 0) & (rr["natural_pos"][0] != force)
                big = imp & ~(rr["margin_pos"][0] < flag_margin)
                if big.any():
                    i = int(np.flatnonzero(big)[0])
                    why = (f"position {i} decided against the rule with margin "
                           f"{rr['margin_pos'][0, i]:.3g} >= {flag_margin}")
            if why is None:
                cdf = rr["cdf"][0] if "cdf" in rr else None
                uu = ref["u_final"][b] if "u_final" in ref else 0.0
                if not _final_ok(int(t_g[n_g]), int(rr["out_tokens"][0, n_g]), cdf, uu, flag_margin):
                    why = f"final token {int(t_g[n_g])} vs {int(rr['out_tokens'][0, n_g])} outside the CDF margin"
            if why is None:
                errs = floats.errors(rr, rows=[b])
                bad = [k for k, e in errs.items() if not (e <= 1.0).all()]
                if bad:
                    why = f"floats out of tolerance on the imposed path: {bad}"
        if why is None:
            return None
        fails.append(why)
    return "; ".join(fails)


def compare(gpu: dict, ref: dict, dtype, check_pos_stats=True, check_feature=False, check_conf=False,
            flag_margin=FLAG_MARGIN, max_diff=None):
    """Assert parity (see the module docstring); returns a summary dict.

    max_diff bounds the sequences whose results differ from the oracle's
    (each of them checked in full along the GPU's decision path); default
    2 + 1% of B."""
    tol = tol_for(dtype)
    n_g = gpu["accepted_len"].cpu().numpy()
    t_g = gpu["out_tokens"].cpu().numpy()
    n_r = ref["accepted_len"]
    t_r = ref["out_tokens"]
    B, K1 = t_r.shape
    assert n_g.shape == (B,) and t_g.shape == (B, K1)
    floats = _Floats(gpu, tol, check_pos_stats, check_feature, check_conf)
    # decisions and tokens against the oracle's own path
    same_path = np.array([n_g[b] == n_r[b] and (t_g[b, :n_r[b]] == t_r[b, :n_r[b]]).all()
                          and (t_g[b, n_r[b] + 1:] == -1).all() for b in range(B)])
    fin_ok = np.zeros(B, bool)
    for b in np.flatnonzero(same_path):
        cdf = ref["cdf"][b] if "cdf" in ref else None
        uu = ref["u_final"][b] if "u_final" in ref else 0.0
        fin_ok[b] = _final_ok(int(t_g[b, n_r[b]]), int(t_r[b, n_r[b]]), cdf, uu, flag_margin)
    errs = floats.errors(ref)
    f_ok = _Floats.seq_ok(errs) if errs else np.ones(B, bool)
    differ = np.flatnonzero(~(same_path & fin_ok & f_ok))
    failures = {}
    for b in differ:
        why = _resolve(int(b), (n_g, t_g), ref, floats, flag_margin, tol)
        if why is not None:
            failures[int(b)] = why
    assert not failures, (
        f"{len(failures)} sequences fail parity, e.g. b={next(iter(failures))}: {next(iter(failures.values()))}; "
        f"gpu n={n_g[next(iter(failures))]} toks={t_g[next(iter(failures))]} vs oracle "
        f"n={n_r[next(iter(failures))]} toks={t_r[next(iter(failures))]}")
    limit = max_diff if max_diff is not None else 2 + int(0.01 * B)
    assert len(differ) <= limit, f"{len(differ)} of {B} sequences differ from the oracle (limit {limit})"
    same_tok = same_path & (t_g[np.arange(B), np.minimum(n_r, K1 - 1)] == t_r[np.arange(B), n_r])
    summary = dict(B=B, flagged_accept=int((ref["margin_acc"] < flag_margin).sum()),
                   flagged_cdf=int((ref["margin_cdf"] < flag_margin).sum()),
                   differ=int(len(differ)), differ_path=int((~same_path).sum()),
                   differ_token=int((same_path & ~same_tok).sum()),
                   differ_floats=int((~f_ok).sum()))
    if "nuc_doubt" in ref and (ref["nuc_doubt"] != 0).any():
        summary["nucleus_doubt"] = int((ref["nuc_doubt"] != 0).any(1).sum())
    for name, e in errs.items():
        summary[f"worst_{name}"] = float(np.max(np.where(np.isfinite(e), e, 0.0))) if e.size else 0.0
    if check_pos_stats:
        ps = gpu["pos_stats"].cpu().numpy()
        summary["rel_entropy"] = _rel(ps[..., 1], ref["pos_stats"][..., 1])
    if check_conf:
        summary["rel_conf"] = _rel(gpu["conf"].cpu().numpy(), ref["conf"])
    return summary


def record(name, summary):
    """Append a parity summary (flagged and differing counts) to the JSON-lines
    file named by SPEC_PARITY_LOG, if set."""
    import json
    import os

    path = os.environ.get("SPEC_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": name, **summary}) + "\n")
