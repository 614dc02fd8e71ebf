"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs. Token ids and accepted lengths must match exactly
except on sequences the oracle flags (decision margin < 1e-5); floats within
the tolerances of tests/helpers.py.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_token_verify_gb300 as sv
import workloads
from helpers import compare, oracle_run, tol_for
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


def _run(inp, mode="stochastic", with_draft=True, est=None, **kw):
    out = hv.verify(inp["zt"], inp["zd"] if with_draft else None, inp["x"],
                    inp["u"] if mode == "stochastic" else None, mode=mode, est_params=est,
                    want_pos_stats=True, want_feature=with_draft, want_conf=est is not None and with_draft,
                    **kw)
    torch.cuda.synchronize()
    return out


# ---------------------------------------------------------------------------
# Workloads (scaled in B for the element-by-element cases)
# ---------------------------------------------------------------------------

def test_tiny_all_modes():
    w = workloads.TINY
    inp = workloads.make_inputs(w, 1001, DEV)
    est = _est(w.K)
    g = _run(inp, "stochastic", est=est)
    r = oracle_run(inp, oracle.STOCHASTIC, est=np.r_[1.0, np.zeros(w.K)])
    compare(g, r, w.dtype, check_feature=True, check_conf=True)
    for with_draft in (True, False):
        g = _run(inp, "greedy", with_draft=with_draft)
        r = oracle_run(inp, oracle.GREEDY, with_draft=with_draft)
        compare(g, r, w.dtype)
        g = _run(inp, "fly", with_draft=with_draft, fly_theta=0.3, fly_window=2)
        r = oracle_run(inp, oracle.FLY, fly_theta=0.3, fly_window=2, with_draft=with_draft)
        compare(g, r, w.dtype)
    assert sv.device_status(g["_workspace"]) == 0


@pytest.mark.parametrize("wl,B", [(workloads.LLAMA3_VOCAB, 12), (workloads.ESTIMATOR, 10),
                                  (workloads.FLY, 12)])
def test_workloads_scaled(wl, B):
    w = wl.scaled(B=B)
    inp = workloads.make_inputs(w, 2000 + B, DEV)
    if w.mode == "fly":
        g = _run(inp, "fly", with_draft=True, fly_theta=w.fly_theta, fly_window=w.fly_window)
        r = oracle_run(inp, oracle.FLY, fly_theta=w.fly_theta, fly_window=w.fly_window)
        compare(g, r, w.dtype, check_feature=True)
        g = _run(inp, "fly", with_draft=False, fly_theta=w.fly_theta, fly_window=w.fly_window)
        r = oracle_run(inp, oracle.FLY, fly_theta=w.fly_theta, fly_window=w.fly_window, with_draft=False)
        compare(g, r, w.dtype)
    else:
        est = _est(w.K)
        g = _run(inp, "stochastic", est=est)
        r = oracle_run(inp, oracle.STOCHASTIC, est=np.r_[1.0, np.zeros(w.K)])
        compare(g, r, w.dtype, check_feature=True, check_conf=True)


@pytest.mark.parametrize("wl", [workloads.LLAMA3_VOCAB, workloads.ESTIMATOR, workloads.FLY],
                         ids=lambda w: w.name)
def test_workloads_full_size(wl):
    """Every sequence of the full-size workload, in the configuration the
    benchmark times."""
    w = wl
    seed = {workloads.LLAMA3_VOCAB.name: 1002, workloads.ESTIMATOR.name: 1003,
            workloads.FLY.name: 1004}[w.name]
    inp = workloads.make_inputs(w, seed, DEV)
    if w.mode == "fly":
        g = _run(inp, "fly", with_draft=False, fly_theta=w.fly_theta, fly_window=w.fly_window)
        r = oracle_run(inp, oracle.FLY, fly_theta=w.fly_theta, fly_window=w.fly_window,
                       with_draft=False, nthreads=16)
        s = compare(g, r, w.dtype)
    else:
        est = _est(w.K) if w.with_confidence else None
        g = _run(inp, "stochastic", est=est)
        r = oracle_run(inp, oracle.STOCHASTIC, nthreads=16,
                       est=None if est is None else np.r_[1.0, np.zeros(w.K)])
        s = compare(g, r, w.dtype, check_feature=True, check_conf=est is not None)
        if w.with_confidence:
            # one estimator step on the GPU's own verification results, on
            # both sides (every sequence, whatever the flagged decisions did)
            p = _est(w.K)
            sv.estimator_update(g["feature"], g["accepted_len"], p, w.estimator_lr)
            newp, _, _ = oracle.estimator_update(g["feature"].cpu().numpy().astype(np.float64),
                                                 g["accepted_len"].cpu().numpy(),
                                                 np.r_[1.0, np.zeros(w.K)], w.estimator_lr)
            np.testing.assert_allclose(p.cpu().numpy(), newp, rtol=1e-5, atol=1e-6)
        # the benchmark's own launch asks for features and confidences only
        # (no pos_stats): same bits as the launch checked above
        b = hv.verify(inp["zt"], inp["zd"], inp["x"], inp["u"], est_params=est, want_feature=True,
                      want_conf=est is not None)
        torch.cuda.synchronize()
        for k in ("out_tokens", "accepted_len", "feature") + (("conf",) if est is not None else ()):
            x_, y_ = g[k], b[k]
            if x_.dtype == torch.float32:
                x_, y_ = x_.view(torch.int32), y_.view(torch.int32)
            assert torch.equal(x_, y_), k
    print(w.name, s)
    hv.record(w.name, s)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_queue_tail_geometry_full_vocab(dt):
    """64 sequences of the estimator workload at its full vocabulary. In
    stochastic mode the queue's last ~80 MB of logits (the last 20 sequences
    here) stream in smaller tiles than the rest: 64 KB tiles, 4 per row for
    bf16 (8 for fp32), then 32 KB tiles. Every sequence, on both sides of that
    boundary, must match the oracle, in a full launch and in a ragged
    (pruned) launch of the same batch."""
    w = workloads.ESTIMATOR.scaled(B=64, dtype=dt)
    inp = workloads.make_inputs(w, 4064, DEV)
    g = _run(inp, "stochastic", est=_est(w.K))
    r = oracle_run(inp, oracle.STOCHASTIC, nthreads=16, est=np.r_[1.0, np.zeros(w.K)])
    compare(g, r, w.dtype, check_feature=True, check_conf=True)
    dl = np.random.default_rng(64).integers(0, w.K + 1, size=w.B).astype(np.int32)
    g2 = _run(inp, "stochastic", draft_len=torch.tensor(dl, device=DEV))
    r2 = oracle_run(inp, oracle.STOCHASTIC, nthreads=16, draft_len=dl)
    compare(g2, r2, w.dtype)
    assert sv.device_status(g2["_workspace"]) == 0


@pytest.mark.parametrize("B,K,V,dt", [(1024, 8, 152064, "f32"), (512, 4, 32000, "bf16"),
                                      (32, 8, 128256, "f32")])
def test_sweep_points_sampled(B, K, V, dt):
    """Largest sweep points at full size; the oracle checks a sample of
    sequences (their rows copied out one by one)."""
    w = workloads.Workload(f"sweep_B{B}_K{K}_V{V}_{dt}", B=B, K=K, V=V, dtype=dt, mode="stochastic")
    inp = workloads.make_inputs(w, 3000 + B + K, DEV)
    g = hv.verify(inp["zt"], inp["zd"], inp["x"], inp["u"], want_pos_stats=True)
    torch.cuda.synchronize()
    idx = torch.linspace(0, B - 1, min(B, 48)).long().unique()
    sub = {k: v[idx.to(v.device)] for k, v in inp.items()}
    r = oracle_run(sub, oracle.STOCHASTIC, nthreads=16)
    gs = {k: g[k][idx.to(DEV)] for k in ("accepted_len", "out_tokens", "pos_stats")}
    s = compare(gs, r, dt)
    print(w.name, s)
    hv.record(w.name + f"_sampled{len(idx)}", s)


# ---------------------------------------------------------------------------
# Edge cases
# ---------------------------------------------------------------------------

def _rand_inputs(B, K, V, dt, seed, sigma=3.0, noise=1.0, device=DEV):
    w = workloads.Workload("edge", B=B, K=K, V=V, dtype=dt, mode="stochastic", sigma_t=sigma,
                           sigma_d=noise)
    return workloads.make_inputs(w, seed, device)


@pytest.mark.parametrize("V", [2, 3, 7, 17, 1000, 2049, 4097, 33333])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_small_and_ragged_vocab(V, dt):
    for K, B in ((1, 5), (3, 4)):
        inp = _rand_inputs(B, K, V, dt, seed=V * 7 + K)
        g = _run(inp, "stochastic", est=_est(K))
        r = oracle_run(inp, oracle.STOCHASTIC, est=np.r_[1.0, np.zeros(K)])
        compare(g, r, dt, check_feature=True, check_conf=True)
        g = _run(inp, "greedy")
        r = oracle_run(inp, oracle.GREEDY)
        compare(g, r, dt)
        g = _run(inp, "fly", fly_theta=0.2, fly_window=1)
        r = oracle_run(inp, oracle.FLY, fly_theta=0.2, fly_window=1)
        compare(g, r, dt)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_misaligned_rows_and_base(dt):
    B, K, V = 6, 3, 5001
    base = _rand_inputs(B, K, V + 3, dt, seed=77)
    # rows of V elements with a row stride of V+3, and a base shifted by one element
    zt_big = base["zt"].reshape(-1)[1:1 + B * (K + 1) * (V + 3) - 3]
    zt = torch.as_strided(zt_big, (B, K + 1, V), ((K + 1) * (V + 3), V + 3, 1))
    zd = base["zd"][:, :, :V]
    x = torch.remainder(base["x"], V).to(torch.int32)
    inp = dict(zt=zt, zd=zd, x=x, u=base["u"])
    g = _run(inp, "stochastic")
    ref_inp = dict(zt=zt.contiguous(), zd=zd.contiguous(), x=x, u=base["u"])
    r = oracle_run(ref_inp, oracle.STOCHASTIC)
    compare(g, r, dt)
    g = _run(inp, "greedy")
    compare(g, oracle_run(ref_inp, oracle.GREEDY), dt)


def test_masked_logits():
    B, K, V = 16, 4, 3000
    inp = _rand_inputs(B, K, V, "f32", seed=5)
    gen = torch.Generator(device=DEV).manual_seed(9)
    mask = torch.rand(inp["zt"].shape, generator=gen, device=DEV) < 0.3
    inp["zt"] = inp["zt"].masked_fill(mask, float("-inf"))
    mask_d = torch.rand(inp["zd"].shape, generator=gen, device=DEV) < 0.3
    inp["zd"] = inp["zd"].masked_fill(mask_d, float("-inf"))
    # draft tokens must have q > 0: redraw them from the masked draft rows
    gum = -torch.log(-torch.log(torch.rand(inp["zd"].shape, generator=gen, device=DEV)))
    inp["x"] = (inp["zd"] + gum).argmax(-1).to(torch.int32)
    g = _run(inp, "stochastic", est=_est(K))
    r = oracle_run(inp, oracle.STOCHASTIC, est=np.r_[1.0, np.zeros(K)])
    compare(g, r, "f32", check_feature=True, check_conf=True)
    g = _run(inp, "fly", fly_theta=0.4, fly_window=1)
    compare(g, oracle_run(inp, oracle.FLY, fly_theta=0.4, fly_window=1), "f32")
    assert sv.device_status(g["_workspace"]) == 0


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_p_equals_q_bonus_draws(dt):
    B, K, V = 64, 5, 20000
    inp = _rand_inputs(B, K, V, dt, seed=12)
    inp["zd"] = inp["zt"][:, :K].contiguous()
    g = _run(inp, "stochastic")
    assert (g["accepted_len"] == K).all()
    compare(g, oracle_run(inp, oracle.STOCHASTIC), dt)


def test_peaked_rows_logit_qmax():
    # q_max -> 1: the complement mass is tiny and must not cancel
    B, K, V = 8, 3, 50000
    inp = _rand_inputs(B, K, V, "f32", seed=31, sigma=1.0)
    for spike in (20.0, 30.0, 40.0):
        zd = inp["zd"].clone()
        zd[:, :, 123] += spike
        zt = inp["zt"].clone()
        zt[:, :, 456] += spike
        cur = dict(zt=zt, zd=zd, x=inp["x"], u=inp["u"])
        g = _run(cur, "stochastic")
        r = oracle_run(cur, oracle.STOCHASTIC)
        compare(g, r, "f32", check_feature=True)


def test_max_K_and_many_sequences():
    inp = _rand_inputs(3, sv.MAX_K, 3000, "bf16", seed=4, noise=0.05)
    g = _run(inp, "stochastic", est=_est(sv.MAX_K))
    compare(g, oracle_run(inp, oracle.STOCHASTIC, est=np.r_[1.0, np.zeros(sv.MAX_K)]), "bf16",
            check_conf=True)
    g = _run(inp, "fly", fly_theta=0.1, fly_window=3)
    compare(g, oracle_run(inp, oracle.FLY, fly_theta=0.1, fly_window=3), "bf16")
    inp = _rand_inputs(5000, 2, 64, "f32", seed=8)
    g = _run(inp, "stochastic")
    compare(g, oracle_run(inp, oracle.STOCHASTIC), "f32")


def test_greedy_ties_bf16():
    B, K, V = 32, 6, 9000
    gen = torch.Generator(device=DEV).manual_seed(3)
    zt = torch.randint(-4, 5, (B, K + 1, V), generator=gen, device=DEV).to(torch.bfloat16)
    am = zt.float().argmax(-1)
    # torch's argmax does not promise the first maximal index: take it explicitly
    first = (zt.float() == zt.float().amax(-1, keepdim=True)).float().argmax(-1)
    x = torch.where(torch.rand((B, K), generator=gen, device=DEV) < 0.85, first[:, :K],
                    torch.randint(0, V, (B, K), generator=gen, device=DEV)).to(torch.int32)
    inp = dict(zt=zt, zd=None, x=x, u=None)
    g = hv.verify(zt, None, x, None, mode="greedy", want_pos_stats=True)
    torch.cuda.synchronize()
    r = oracle_run(dict(zt=zt, zd=zt[:, :K], x=x, u=None), oracle.GREEDY, with_draft=False)
    compare(g, r, "bf16")
    del am, inp


def test_fly_with_a_closed_gate_is_greedy_full_size():
    """A property that holds at any size: normalised entropy never exceeds 1,
    so at theta > 1 FLy defers nothing and equals greedy exact match, bit
    for bit, on the full FLy workload (B=128, K=15, V=152064, bf16)."""
    w = workloads.FLY
    inp = workloads.make_inputs(w, 1009, DEV)
    g = hv.verify(inp["zt"], None, inp["x"], None, mode="greedy")
    for W in (1, 4):
        f = hv.verify(inp["zt"], None, inp["x"], None, mode="fly", fly_theta=1.5, fly_window=W)
        torch.cuda.synchronize()
        assert torch.equal(f["accepted_len"], g["accepted_len"])
        assert torch.equal(f["out_tokens"], g["out_tokens"])


@pytest.mark.parametrize("wl", [workloads.ESTIMATOR, workloads.FLY.scaled(B=64),
                                workloads.Workload("sweep_B512_K8_V152064_f32", B=512, K=8, V=152064,
                                                   dtype="f32", mode="stochastic")],
                         ids=lambda w: w.name)
def test_deterministic_bits(wl):
    """Repeated launches on the same inputs give identical bits (fixed
    reduction orders, no float atomics, no races between the copy engine and
    the lanes)."""
    inp = workloads.make_inputs(wl, 99, DEV)
    mode = wl.mode
    kw = dict(fly_theta=wl.fly_theta, fly_window=wl.fly_window) if mode == "fly" else {}
    runs = [_run(inp, mode, est=_est(wl.K), **kw) for _ in range(4)]
    for k in ("out_tokens", "accepted_len", "pos_stats", "feature", "conf"):
        ref = runs[0][k]
        ref = ref.view(torch.int32) if ref.dtype == torch.float32 else ref
        for other in runs[1:]:
            o = other[k].view(torch.int32) if other[k].dtype == torch.float32 else other[k]
            assert torch.equal(ref, o), k


def test_bad_token_and_bad_row_status():
    B, K, V = 4, 3, 1000
    inp = _rand_inputs(B, K, V, "f32", seed=1)
    x = inp["x"].clone()
    x[1, 1] = V + 5
    x[2, 0] = -1
    inp["x"] = x
    g = _run(inp, "stochastic")
    assert sv.device_status(g["_workspace"]) == sv.api.SPEC_ERR_BAD_TOKEN
    n = g["accepted_len"].cpu().numpy()
    assert n[1] <= 1 and n[2] == 0
    g = _run(inp, "greedy")
    assert sv.device_status(g["_workspace"]) == sv.api.SPEC_ERR_BAD_TOKEN
    inp = _rand_inputs(B, K, V, "f32", seed=2)
    inp["zt"][0, 0, :] = float("-inf")
    g = _run(inp, "stochastic")
    assert sv.device_status(g["_workspace"]) == sv.api.SPEC_ERR_BAD_ROW
    # a clean call resets the status word
    g = _run(_rand_inputs(B, K, V, "f32", seed=3), "stochastic")
    assert sv.device_status(g["_workspace"]) == 0


@pytest.mark.parametrize("case", ["estimator", "masked_f32", "greedy_bf16", "fly_bf16", "temperature"])
def test_outputs_do_not_depend_on_pos_stats(case):
    """Target rows fold the entropy moment only when something reads it
    (pos_stats, or FLy's gate). Tokens, accepted lengths, features and
    confidences must be the same bits with and without pos_stats requested,
    on ordinary, masked (-inf) and temperature-processed rows."""
    kw = {}
    if case == "estimator":
        inp = workloads.make_inputs(workloads.ESTIMATOR.scaled(B=40), 7101, DEV)
        mode, K = "stochastic", workloads.ESTIMATOR.K
    elif case == "masked_f32":
        inp = _rand_inputs(16, 4, 3000, "f32", seed=7102)
        gen = torch.Generator(device=DEV).manual_seed(7)
        inp["zt"] = inp["zt"].masked_fill(torch.rand(inp["zt"].shape, generator=gen, device=DEV) < 0.3,
                                          float("-inf"))
        mode, K = "stochastic", 4
    elif case == "greedy_bf16":
        inp = _rand_inputs(24, 6, 50000, "bf16", seed=7103)
        mode, K = "greedy", 6
    elif case == "fly_bf16":
        inp = workloads.make_inputs(workloads.FLY.scaled(B=16), 7104, DEV)
        mode, K = "fly", workloads.FLY.K
        kw = dict(fly_theta=0.3, fly_window=6)
    else:
        w = workloads.ESTIMATOR.scaled(B=24, inv_temp_range=(0.5, 2.0))
        inp = workloads.make_inputs(w, 7105, DEV)
        mode, K = "stochastic", w.K
        kw = dict(inv_temperature=inp["inv_temp"])
    est = _est(K)
    u = inp["u"] if mode == "stochastic" else None
    runs = [hv.verify(inp["zt"], inp["zd"], inp["x"], u, mode=mode, est_params=est, want_pos_stats=ps,
                      want_feature=True, want_conf=True, **kw) for ps in (True, False)]
    torch.cuda.synchronize()
    for k in ("out_tokens", "accepted_len", "feature", "conf"):
        a, b = runs[0][k], runs[1][k]
        if a.dtype == torch.float32:
            a, b = a.view(torch.int32), b.view(torch.int32)
        assert torch.equal(a, b), k


def test_a_residual_wait_that_runs_out_sets_timeout():
    """Failure detection without a fault. With the poll limit of the bounded
    residual wait set to 0 (spec_debug_set_wait_limit), every warp that would
    wait for a sequence's draw gives up at once: it raises SPEC_ERR_TIMEOUT in
    the status word and returns, so the launch ends with the draws undone
    (those output slots keep the poison they were given). The host reads the
    status. The next call, at the default limit, is clean and matches the
    oracle, and the accepted lengths (decided before any wait) agree."""
    L = sv._native.lib()
    B, K, V = 8, 3, 5000
    inp = _rand_inputs(B, K, V, "f32", seed=41)
    prev = L.spec_debug_set_wait_limit(0)
    try:
        t = _run(inp, "stochastic")
    finally:
        L.spec_debug_set_wait_limit(prev)
    assert sv.device_status(t["_workspace"]) == sv.api.SPEC_ERR_TIMEOUT
    n_t = t["accepted_len"].cpu().numpy()
    toks = t["out_tokens"].cpu().numpy()
    assert (toks[np.arange(B), n_t] == hv.POISON_I32).all()   # no draw was made
    g = _run(inp, "stochastic")
    assert sv.device_status(g["_workspace"]) == 0
    compare(g, oracle_run(inp, oracle.STOCHASTIC), "f32")
    np.testing.assert_array_equal(n_t, g["accepted_len"].cpu().numpy())


# ---------------------------------------------------------------------------
# Losslessness on the GPU: 1e6 sequences in one call, V = 16
# ---------------------------------------------------------------------------

def test_gpu_lossless_chi_square():
    from scipy import stats
    rng = np.random.default_rng(2024)
    V, K, N = 16, 2, 1_000_000
    zt1 = rng.normal(0, 1.5, (K + 1, V)).astype(np.float32)
    zd1 = (zt1[:K] + rng.normal(0, 1.0, (K, V))).astype(np.float32)
    p = np.exp(zt1 - zt1.max(-1, keepdims=True).astype(np.float64))
    p /= p.sum(-1, keepdims=True)
    q = np.exp(zd1 - zd1.max(-1, keepdims=True).astype(np.float64))
    q /= q.sum(-1, keepdims=True)
    x = np.stack([rng.choice(V, size=N, p=q[i]) for i in range(K)], 1).astype(np.int32)
    u = rng.random((N, K + 1), dtype=np.float32)
    zt = torch.from_numpy(zt1).to(DEV).expand(N, K + 1, V).contiguous()
    zd = torch.from_numpy(zd1).to(DEV).expand(N, K, V).contiguous()
    g = hv.verify(zt, zd, torch.from_numpy(x).to(DEV), torch.from_numpy(u).to(DEV))
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


# ---------------------------------------------------------------------------
# Estimator and confidence entry points
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("B,K", [(256, 8), (1, 1), (1000, 15), (0, 4), (64, 16), (300, 24)])
def test_estimator_update_parity(B, K):
    rng = np.random.default_rng(B * 31 + K)
    f = rng.normal(-3.0, 1.5, (B, K)).astype(np.float32)
    n = rng.integers(0, K + 1, B).astype(np.int32)
    p0 = np.r_[0.9, rng.normal(0, 0.3, K)].astype(np.float32)
    pt = torch.from_numpy(p0.copy()).to(DEV)
    ft = torch.from_numpy(f).to(DEV) if B else torch.empty((0, K), dtype=torch.float32, device=DEV)
    nt = torch.from_numpy(n).to(DEV) if B else torch.empty((0,), dtype=torch.int32, device=DEV)
    grad, cnt = sv.estimator_update(ft, nt, pt, 0.05, want_grad=True)
    torch.cuda.synchronize()
    newp, g_ref, c_ref = oracle.estimator_update(f.astype(np.float64).reshape(B, K), n,
                                                 p0.astype(np.float64), 0.05)
    assert (cnt.cpu().numpy() == c_ref).all()
    np.testing.assert_allclose(grad.cpu().numpy(), g_ref, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(pt.cpu().numpy(), newp, rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_confidence_entry_point(dt):
    w = workloads.ESTIMATOR.scaled(B=20, dtype=dt)
    inp = workloads.make_inputs(w, 404, DEV)
    est = torch.tensor([0.53, 0.4, 0.3, 0.2, 0.1, 0.0, -0.1, -0.2, -0.3], dtype=torch.float32, device=DEV)
    feat, conf = hv.confidence(inp["zd"], est)
    torch.cuda.synchronize()
    f_ref, c_ref, _ = oracle.confidence(workloads.to_numpy_logits(inp["zd"]),
                                        est.cpu().numpy().astype(np.float64), nthreads=8)
    tol = tol_for(dt)
    np.testing.assert_allclose(feat.cpu().numpy(), f_ref, rtol=tol, atol=tol)
    np.testing.assert_allclose(conf.cpu().numpy(), c_ref, rtol=tol, atol=1e-6)
    feat2, none = hv.confidence(inp["zd"])
    torch.cuda.synchronize()
    assert none is None and torch.equal(feat2, feat)
