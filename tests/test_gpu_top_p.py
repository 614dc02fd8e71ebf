"""GPU parity of top-p (nucleus) processed verification (spec_verify_top_p)
against the fp64 oracle, through the C ABI.

"Verificación Adaptativa sin una cabeza de confianza", "Benchmarks" (serving
samples with top-p 0.95); "Speculative Decoding: ...", "Математика
верификации" (lossless for the processed p and q). Inputs are seeded; drafts
come from the temperature-processed q of the generator, so a draft can fall
outside q's nucleus (the q(x) = 0 reading then applies on both sides).
Tolerances and the flagged-margin rule (which covers the nucleus boundary)
are those of tests/helpers.py.
"""
import numpy as np
import pytest
import torch
from scipy import special

import oracle
import speculative_decoding_token_verify_gb300 as sv
import workloads
from helpers import compare, oracle_run
import helpers as hv

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()
    yield


def _est(K):
    return torch.tensor([1.0] + [0.0] * K, dtype=torch.float32, device=DEV)


def _run(inp, mode, top_p, s=None, with_draft=True, est=None, draft_len=None, **kw):
    out = hv.verify(inp["zt"], inp["zd"] if with_draft else None, inp["x"],
                    inp["u"] if mode == "stochastic" else None, mode=mode, est_params=est,
                    want_pos_stats=True, want_feature=with_draft, want_conf=est is not None and with_draft,
                    inv_temperature=s, top_p=top_p, draft_len=draft_len, **kw)
    torch.cuda.synchronize()
    return out


def _wl(B, K, V, dt, lo=None, hi=None, **kw):
    return workloads.Workload(f"topp_B{B}_K{K}_V{V}_{dt}", B=B, K=K, V=V, dtype=dt, mode="stochastic",
                              sigma_t=3.0, sigma_d=1.0,
                              inv_temp_range=None if lo is None else (lo, hi), **kw)


def _cmp(g, r, dt, **kw):
    """compare() for top-p runs. A nucleus boundary in doubt (a tie group
    holding over 1e-6 of the nucleus, within 1e-5 relative of top_p; common
    with bf16 ties at 128K vocabularies) may be placed one tie group off by
    the GPU; compare() then checks the sequence in full against the oracle
    with that boundary moved. Such sequences may differ from the oracle's
    natural result, on top of the usual bound."""
    B = len(r["accepted_len"])
    doubt = int((r["nuc_doubt"] != 0).any(1).sum())
    return compare(g, r, dt, max_diff=2 + int(0.01 * B) + doubt, **kw)


def _oracle(inp, mode, top_p, temp=True, **kw):
    s = inp["inv_temp"].cpu().numpy() if temp and "inv_temp" in inp else None
    return oracle_run(inp, mode, inv_temp=s, top_p=top_p, **kw)


@pytest.mark.parametrize("B,K,V,dt,top_p", [(16, 4, 1000, "f32", 0.95), (12, 8, 128256, "bf16", 0.95),
                                            (8, 5, 33333, "f32", 0.5), (24, 3, 4097, "bf16", 0.8),
                                            (6, 2, 2, "f32", 0.7)])
def test_all_modes_match_oracle(B, K, V, dt, top_p):
    w = _wl(B, K, V, dt, 0.5, 2.0)
    inp = workloads.make_inputs(w, 5100 + B + K, DEV)
    s = inp["inv_temp"]
    g = _run(inp, "stochastic", top_p, s, est=_est(K))
    r = _oracle(inp, oracle.STOCHASTIC, top_p, est=np.r_[1.0, np.zeros(K)])
    print(_cmp(g, r, dt, check_feature=True, check_conf=True))
    for with_draft in (True, False):
        g = _run(inp, "greedy", top_p, s, with_draft=with_draft)
        r = _oracle(inp, oracle.GREEDY, top_p, with_draft=with_draft)
        _cmp(g, r, dt)
        g = _run(inp, "fly", top_p, s, with_draft=with_draft, fly_theta=0.3, fly_window=2)
        r = _oracle(inp, oracle.FLY, top_p, fly_theta=0.3, fly_window=2, with_draft=with_draft)
        _cmp(g, r, dt)
    assert sv.device_status(g["_workspace"]) == 0


@pytest.mark.parametrize("top_p", [1e-6, 0.3, 0.999])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_top_p_range_without_temperature(top_p, dt):
    w = _wl(32, 4, 2049, dt)
    inp = workloads.make_inputs(w, 5200, DEV)
    g = _run(inp, "stochastic", top_p, est=_est(4))
    r = _oracle(inp, oracle.STOCHASTIC, top_p, est=np.r_[1.0, np.zeros(4)])
    print(top_p, _cmp(g, r, dt, check_feature=True, check_conf=True))


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_ties_at_the_boundary(dt):
    """Logits on a coarse grid: many tokens tie at the nucleus boundary."""
    w = _wl(24, 3, 3000, dt)
    inp = workloads.make_inputs(w, 5300, DEV)
    inp["zt"] = (torch.round(inp["zt"].float() * 2) / 2).to(inp["zt"].dtype)
    inp["zd"] = (torch.round(inp["zd"].float() * 2) / 2).to(inp["zd"].dtype)
    for tp in (0.6, 0.9):
        g = _run(inp, "stochastic", tp, est=_est(3))
        r = _oracle(inp, oracle.STOCHASTIC, tp, est=np.r_[1.0, np.zeros(3)])
        _cmp(g, r, dt, check_feature=True, check_conf=True)


@pytest.mark.parametrize("V", [128256, 152064])
def test_large_fp32_rows(V):
    """fp32 rows of 501 KB and 594 KB: the row kernel's significand shift
    grows with the tokens a warp bins (5 and 6 bits)."""
    w = _wl(6, 3, V, "f32", 0.5, 2.0)
    inp = workloads.make_inputs(w, 5450 + V % 97, DEV)
    g = _run(inp, "stochastic", 0.9, inp["inv_temp"], est=_est(3))
    r = _oracle(inp, oracle.STOCHASTIC, 0.9, est=np.r_[1.0, np.zeros(3)])
    print(V, _cmp(g, r, "f32", check_feature=True, check_conf=True))


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_nucleus_reference_and_boundary_paths(dt):
    """Rows that take each path of the nucleus selection, next to ordinary
    rows: a spike far above the first units' maximum (the mass bins are taken
    again against the row max), a masked head (no maximum in the first units:
    the bins wait for the row max), and a narrow row centred on 0 (in bf16 the
    boundary bin then spans far more than 256 keys: a coarse key round
    first)."""
    w = _wl(8, 3, 50000, dt)
    inp = workloads.make_inputs(w, 5800, DEV)
    zt, zd = inp["zt"], inp["zd"]
    zt[0, :, 40000] = 45.0
    zd[0, :, 40001] = 45.0
    zt[1, :, :20000] = float("-inf")
    zd[1, :, :20000] = float("-inf")
    inp["x"][1] = 20000 + inp["x"][1] % 30000
    zt[2] = (zt[2].float() * 0.05).to(zt.dtype)
    zd[2] = (zd[2].float() * 0.05).to(zd.dtype)
    for tp in (0.5, 0.95):
        g = _run(inp, "stochastic", tp, est=_est(3))
        r = _oracle(inp, oracle.STOCHASTIC, tp, est=np.r_[1.0, np.zeros(3)])
        print(tp, _cmp(g, r, dt, check_feature=True, check_conf=True))
        assert sv.device_status(g["_workspace"]) == 0


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_vocabularies_beyond_the_row_kernel(dt):
    """V = 300000: a warp bins more tokens than 32-bit counters hold at a
    2^-18 significand, so the pass takes the 64-bit histogram kernel."""
    w = _wl(3, 2, 300000, dt, 0.5, 2.0)
    inp = workloads.make_inputs(w, 5900, DEV)
    g = _run(inp, "stochastic", 0.9, inp["inv_temp"], est=_est(2))
    r = _oracle(inp, oracle.STOCHASTIC, 0.9, est=np.r_[1.0, np.zeros(2)])
    print(_cmp(g, r, dt, check_feature=True, check_conf=True))
    assert sv.device_status(g["_workspace"]) == 0


def test_masked_and_flat_rows():
    w = _wl(8, 3, 1000, "f32")
    inp = workloads.make_inputs(w, 5400, DEV)
    inp["zt"][0, :, 500:] = float("-inf")            # masked tail
    inp["zd"][0, :, 500:] = float("-inf")
    inp["x"][0] = inp["x"][0] % 500
    inp["zt"][1] = 0.25                              # a flat row: every token tied
    inp["zd"][1] = -1.0
    g = _run(inp, "stochastic", 0.9, est=_est(3))
    r = _oracle(inp, oracle.STOCHASTIC, 0.9, est=np.r_[1.0, np.zeros(3)])
    _cmp(g, r, "f32", check_feature=True, check_conf=True)
    assert sv.device_status(g["_workspace"]) == 0


def test_ragged_with_top_p_and_temperature():
    w = _wl(40, 6, 32000, "bf16", 0.5, 2.0)
    inp = workloads.make_inputs(w, 5500, DEV)
    s = inp["inv_temp"]
    dl = np.random.default_rng(3).integers(0, 7, 40).astype(np.int32)
    dl[:3] = [0, 6, 1]
    g = _run(inp, "stochastic", 0.95, s, est=_est(6), draft_len=torch.tensor(dl, device=DEV))
    r = _oracle(inp, oracle.STOCHASTIC, 0.95, est=np.r_[1.0, np.zeros(6)], draft_len=dl)
    _cmp(g, r, "bf16", check_feature=True, check_conf=True)


def test_full_size_estimator_shape_sampled():
    """B=256, K=8, V=128256 bf16 at top-p 0.95 and per-sequence temperatures,
    in the launch configuration the benchmark times; the oracle checks a
    sample of sequences."""
    w = workloads.ESTIMATOR.scaled(inv_temp_range=(0.5, 2.0))
    inp = workloads.make_inputs(w, 5600, DEV)
    g = _run(inp, "stochastic", 0.95, inp["inv_temp"], est=_est(w.K))
    idx = torch.linspace(0, w.B - 1, 32).long().unique()
    sub = {k: v[idx.to(v.device)] for k, v in inp.items()}
    r = _oracle(sub, oracle.STOCHASTIC, 0.95, nthreads=16, est=np.r_[1.0, np.zeros(w.K)])
    gs = {k: g[k][idx.to(DEV)] for k in ("accepted_len", "out_tokens", "pos_stats", "feature", "conf")}
    s = _cmp(gs, r, w.dtype, check_feature=True, check_conf=True)
    print(s)
    hv.record("top_p0.95_" + w.name + "_sampled32", s)


def test_top_p_one_is_the_temperature_path_and_runs_repeat():
    w = _wl(16, 4, 50000, "bf16", 0.5, 2.0)
    inp = workloads.make_inputs(w, 5700, DEV)
    s = inp["inv_temp"]
    a = _run(inp, "stochastic", 1.0, s, est=_est(4))
    b = _run(inp, "stochastic", None, s, est=_est(4))
    for k in ("out_tokens", "accepted_len", "feature", "conf"):
        assert torch.equal(a[k], b[k]), k
    c1 = _run(inp, "stochastic", 0.9, s, est=_est(4))
    c2 = _run(inp, "stochastic", 0.9, s, est=_est(4))
    for k in ("out_tokens", "accepted_len", "feature", "conf"):
        assert torch.equal(c1[k], c2[k]), k
    assert torch.equal(c1["pos_stats"].nan_to_num(7.0), c2["pos_stats"].nan_to_num(7.0))


def _nucleus_np(z, tp):
    p = special.softmax(z.astype(np.float64))
    order = np.argsort(-z, kind="stable")
    cum = np.cumsum(p[order])
    k = min(int(np.searchsorted(cum, tp)), len(z) - 1)
    m = z >= z[order[k]]
    q = p * m
    return q / q.sum()


def test_gpu_lossless_chi_square_under_top_p():
    """1e6 identical sequences at top-p 0.8 with drafts from the draft's
    nucleus: the first emitted token follows the target's nucleus."""
    from scipy import stats
    rng = np.random.default_rng(2026)
    V, K, N, tp = 16, 2, 1_000_000, 0.8
    zt1 = rng.normal(0, 1.5, (K + 1, V)).astype(np.float32)
    zd1 = (zt1[:K] + rng.normal(0, 1.0, (K, V))).astype(np.float32)
    p = np.array([_nucleus_np(zt1[i], tp) for i in range(K + 1)])
    q = np.array([_nucleus_np(zd1[i], tp) for i in range(K)])
    x = np.stack([rng.choice(V, size=N, p=q[i]) for i in range(K)], 1).astype(np.int32)
    u = rng.random((N, K + 1), dtype=np.float32)
    zt = torch.from_numpy(zt1).to(DEV).expand(N, K + 1, V).contiguous()
    zd = torch.from_numpy(zd1).to(DEV).expand(N, K, V).contiguous()
    g = hv.verify(zt, zd, torch.from_numpy(x).to(DEV), torch.from_numpy(u).to(DEV), top_p=tp)
    torch.cuda.synchronize()
    toks = g["out_tokens"].cpu().numpy()
    n = g["accepted_len"].cpu().numpy()
    nz = p[0] > 0
    c0 = np.bincount(toks[:, 0], minlength=V)
    assert c0[~nz].sum() == 0
    e = p[0][nz] * N
    assert stats.chi2.sf(((c0[nz] - e) ** 2 / e).sum(), nz.sum() - 1) > 1e-4
    a = np.minimum(p[0], q[0]).sum()
    assert abs((n >= 1).mean() - a) < 5 * np.sqrt(a * (1 - a) / N)
