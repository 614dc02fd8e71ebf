"""GPU parity of temperature-processed verification (spec_verify_temperature)
against the fp64 oracle, through the C ABI.

"Verificación Adaptativa sin una cabeza de confianza", "Benchmarks" (serving
samples at a temperature); "Speculative Decoding: ...", "Математика
верификации" (the rule is lossless for the processed p and q). Inputs are
seeded: per-sequence inverse temperatures log-uniform on a range, drafts drawn
from the processed q. Tolerances and the flagged-margin rule are those of
tests/helpers.py.
"""
import numpy as np
import pytest
import torch

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


def _run(inp, mode, s, with_draft=True, est=None, draft_len=None, **kw):
    out = hv.verify(inp["zt"], inp["zd"] if with_draft else None, inp["x"],
                    inp["u"] if mode == "stochastic" else None, mode=mode, est_params=est,
                    want_pos_stats=True, want_feature=with_draft, want_conf=est is not None and with_draft,
                    inv_temperature=s, draft_len=draft_len, **kw)
    torch.cuda.synchronize()
    return out


def _wl(B, K, V, dt, lo, hi, **kw):
    return workloads.Workload(f"temp_B{B}_K{K}_V{V}_{dt}", B=B, K=K, V=V, dtype=dt, mode="stochastic",
                              sigma_t=3.0, sigma_d=1.0, inv_temp_range=(lo, hi), **kw)


@pytest.mark.parametrize("B,K,V,dt", [(16, 4, 1000, "f32"), (12, 8, 128256, "bf16"), (8, 5, 33333, "f32"),
                                      (24, 3, 4097, "bf16")])
def test_all_modes_match_oracle(B, K, V, dt):
    w = _wl(B, K, V, dt, 0.25, 4.0)
    inp = workloads.make_inputs(w, 4100 + B + K, DEV)
    s = inp["inv_temp"]
    s_np = s.cpu().numpy()
    est = _est(K)
    g = _run(inp, "stochastic", s, est=est)
    r = oracle_run(inp, oracle.STOCHASTIC, est=np.r_[1.0, np.zeros(K)], inv_temp=s_np)
    print(compare(g, r, dt, check_feature=True, check_conf=True))
    for with_draft in (True, False):
        g = _run(inp, "greedy", s, with_draft=with_draft)
        r = oracle_run(inp, oracle.GREEDY, with_draft=with_draft, inv_temp=s_np)
        compare(g, r, dt)
        g = _run(inp, "fly", s, with_draft=with_draft, fly_theta=0.3, fly_window=2)
        r = oracle_run(inp, oracle.FLY, fly_theta=0.3, fly_window=2, with_draft=with_draft, inv_temp=s_np)
        compare(g, r, dt)
    assert sv.device_status(g["_workspace"]) == 0


@pytest.mark.parametrize("s_val", [1e-4, 0.01, 0.3, 3.0, 100.0, 1e4])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_extreme_temperatures(s_val, dt):
    """Both ends of the supported range: near-uniform rows (s = 1e-4) and
    one-hot rows (s = 1e4, where the draw becomes the argmax)."""
    w = _wl(32, 4, 2049, dt, s_val, s_val)
    inp = workloads.make_inputs(w, 4200, DEV)
    s = inp["inv_temp"]
    g = _run(inp, "stochastic", s, est=_est(4))
    r = oracle_run(inp, oracle.STOCHASTIC, est=np.r_[1.0, np.zeros(4)], inv_temp=s.cpu().numpy())
    print(s_val, compare(g, r, dt, check_feature=True, check_conf=True))
    assert sv.device_status(g["_workspace"]) == 0


def test_ragged_with_temperature():
    w = _wl(40, 6, 32000, "bf16", 0.5, 2.0)
    inp = workloads.make_inputs(w, 4300, DEV)
    s = inp["inv_temp"]
    dl = np.random.default_rng(3).integers(0, 7, 40).astype(np.int32)
    dl[:3] = [0, 6, 1]
    g = _run(inp, "stochastic", s, est=_est(6), draft_len=torch.tensor(dl, device=DEV))
    r = oracle_run(inp, oracle.STOCHASTIC, est=np.r_[1.0, np.zeros(6)], inv_temp=s.cpu().numpy(), draft_len=dl)
    compare(g, r, "bf16", check_feature=True, check_conf=True)
    g = _run(inp, "fly", s, draft_len=torch.tensor(dl, device=DEV), fly_theta=0.4, fly_window=1)
    r = oracle_run(inp, oracle.FLY, fly_theta=0.4, fly_window=1, inv_temp=s.cpu().numpy(), draft_len=dl)
    compare(g, r, "bf16")


def test_full_size_estimator_shape_sampled():
    """B=256, K=8, V=128256 bf16 at per-sequence temperatures, in the launch
    configuration the benchmark times; the oracle checks a sample of
    sequences."""
    w = workloads.ESTIMATOR.scaled(inv_temp_range=(0.5, 2.0))
    inp = workloads.make_inputs(w, 4400, DEV)
    g = _run(inp, "stochastic", inp["inv_temp"], est=_est(w.K))
    idx = torch.linspace(0, w.B - 1, 40).long().unique()
    sub = {k: v[idx.to(v.device)] for k, v in inp.items()}
    r = oracle_run(sub, oracle.STOCHASTIC, nthreads=16, est=np.r_[1.0, np.zeros(w.K)],
                   inv_temp=sub["inv_temp"].cpu().numpy())
    gs = {k: g[k][idx.to(DEV)] for k in ("accepted_len", "out_tokens", "pos_stats", "feature", "conf")}
    s = compare(gs, r, w.dtype, check_feature=True, check_conf=True)
    print(s)
    hv.record("temperature_" + w.name + "_sampled40", s)


def test_unit_temperature_agrees_with_the_default_path():
    """s = 1 through the temperature variant (difference-first exponents)
    against spec_verify (fused exponents): statistics within a few fp32
    roundings, decisions equal wherever the oracle does not flag them."""
    w = workloads.LLAMA3_VOCAB.scaled(B=16)
    inp = workloads.make_inputs(w, 4500, DEV)
    one = torch.ones(w.B, dtype=torch.float32, device=DEV)
    a = _run(inp, "stochastic", one, est=_est(w.K))
    b = hv.verify(inp["zt"], inp["zd"], inp["x"], inp["u"], est_params=_est(w.K), want_pos_stats=True,
                  want_feature=True, want_conf=True)
    torch.cuda.synchronize()
    pa, pb = a["pos_stats"].nan_to_num(7.0), b["pos_stats"].nan_to_num(7.0)
    assert torch.allclose(pa, pb, rtol=2e-6, atol=2e-6)
    assert torch.allclose(a["conf"], b["conf"], rtol=2e-6, atol=1e-7)
    r = oracle_run(inp, oracle.STOCHASTIC)
    flagged = (r["margin_acc"] < 1e-5) | (r["margin_cdf"] < 1e-5)
    same = (a["out_tokens"] == b["out_tokens"]).all(1).cpu().numpy()
    assert (same | flagged).all()


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_power_of_two_temperature_equals_scaled_logits_on_gpu(dt):
    """s = 2 on z against s = 1 on 2z (exact in fp32 and bf16): every step of
    the temperature variant scales exactly, so every output is the same bits."""
    w = _wl(24, 6, 50000, dt, 1.0, 1.0)
    inp = workloads.make_inputs(w, 4600, DEV)
    two = torch.full((w.B,), 2.0, dtype=torch.float32, device=DEV)
    one = torch.ones(w.B, dtype=torch.float32, device=DEV)
    a = _run(inp, "stochastic", two, est=_est(w.K))
    dbl = dict(inp, zt=inp["zt"] * 2, zd=inp["zd"] * 2)
    b = _run(dbl, "stochastic", one, est=_est(w.K))
    for k in ("out_tokens", "accepted_len", "feature", "conf"):
        assert torch.equal(a[k], b[k]), k
    assert torch.equal(a["pos_stats"].nan_to_num(7.0), b["pos_stats"].nan_to_num(7.0))


def test_out_of_range_temperature_sets_status_and_runs_at_one():
    w = _wl(8, 4, 1000, "f32", 1.0, 1.0)
    inp = workloads.make_inputs(w, 4700, DEV)
    s = torch.tensor([1.0, 0.0, float("nan"), -2.0, 1e5, 1.0, 5e-5, 1.0], device=DEV)
    g = _run(inp, "stochastic", s)
    assert sv.device_status(g["_workspace"]) == sv.api.SPEC_ERR_BAD_TEMPERATURE
    r = oracle_run(inp, oracle.STOCHASTIC, inv_temp=np.ones(8, np.float32))
    compare(g, r, "f32")
    ok = _run(inp, "stochastic", torch.ones(8, device=DEV))
    assert sv.device_status(ok["_workspace"]) == 0


def test_gpu_lossless_chi_square_at_a_temperature():
    """1e6 identical sequences at s = 0.6: the first emitted token follows
    softmax(s z_0) and the first acceptance rate is sum min(p, q) of the
    processed distributions."""
    from scipy import stats
    rng = np.random.default_rng(2025)
    V, K, N, s = 16, 2, 1_000_000, 0.6
    zt1 = rng.normal(0, 2.5, (K + 1, V)).astype(np.float32)
    zd1 = (zt1[:K] + rng.normal(0, 1.5, (K, V))).astype(np.float32)

    def soft(z):
        e = np.exp(s * (z.astype(np.float64) - z.max(-1, keepdims=True)))
        return e / e.sum(-1, keepdims=True)
    p, q = soft(zt1), soft(zd1)
    x = np.stack([rng.choice(V, size=N, p=q[i]) for i in range(K)], 1).astype(np.int32)
    u = rng.random((N, K + 1), dtype=np.float32)
    zt = torch.from_numpy(zt1).to(DEV).expand(N, K + 1, V).contiguous()
    zd = torch.from_numpy(zd1).to(DEV).expand(N, K, V).contiguous()
    g = hv.verify(zt, zd, torch.from_numpy(x).to(DEV), torch.from_numpy(u).to(DEV),
                  inv_temperature=torch.full((N,), s, dtype=torch.float32, device=DEV))
    torch.cuda.synchronize()
    toks = g["out_tokens"].cpu().numpy()
    n = g["accepted_len"].cpu().numpy()

    def pval(counts, probs):
        e = probs * counts.sum()
        return stats.chi2.sf(((counts - e) ** 2 / e).sum(), len(probs) - 1)

    assert pval(np.bincount(toks[:, 0], minlength=V), p[0]) > 1e-4
    assert pval(np.bincount(toks[n >= 1, 1], minlength=V), p[1]) > 1e-4
    a = np.minimum(p[0], q[0]).sum()
    assert abs((n >= 1).mean() - a) < 5 * np.sqrt(a * (1 - a) / N)
