"""The checked build (SPEC_CHECKED, libspecverify_checked.so) on the edge
cases: its kernels check every index they derive (work item, sequence, row,
tile, draw slot, slice, token) against the buffer it addresses and raise
SPEC_ERR_INDEX instead of making an access that a check rejects. Here no
check may fail (status 0), and every output must be the same bits as the
default build's, on poisoned outputs and workspaces (tests/helpers.py).

The cases: tiny and ragged vocabularies, rows that start off any 16-byte
boundary, masked (-inf) logits, the largest K, a pruned (ragged) batch, the
queue's tail of smaller tiles, temperature and top-p processing (both
nucleus kernels), greedy and FLy, and the confidence pass.
"""
import numpy as np
import pytest
import torch

import helpers as hv
import speculative_decoding_token_verify_gb300 as sv
import workloads
from speculative_decoding_token_verify_gb300 import _native

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()
    _native.build()
    yield


def _bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t


def _both(monkeypatch, fn):
    """fn() under the default library, then under the checked one; returns
    both results and the checked run's status word."""
    ref = fn()
    torch.cuda.synchronize()
    with monkeypatch.context() as m:
        m.setattr(_native, "_lib", _native.lib_checked())
        got = fn()
        torch.cuda.synchronize()
        status = sv.device_status(got["_workspace"]) if "_workspace" in got else 0
    return ref, got, status


def _same(ref, got, keys=("out_tokens", "accepted_len", "pos_stats", "feature", "conf")):
    for k in keys:
        if k in ref:
            assert torch.equal(_bits(ref[k]), _bits(got[k])), k


def _rand(B, K, V, dt, seed, **kw):
    w = workloads.Workload("checked", B=B, K=K, V=V, dtype=dt, mode="stochastic", **kw)
    return workloads.make_inputs(w, seed, DEV)


def _est(K):
    return torch.tensor([1.0] + [0.0] * K, dtype=torch.float32, device=DEV)


@pytest.mark.parametrize("V", [2, 7, 17, 2049, 33333])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_small_and_ragged_vocab(monkeypatch, V, dt):
    inp = _rand(5, 3, V, dt, seed=9100 + V)
    for mode in ("stochastic", "greedy", "fly"):
        ref, got, st = _both(monkeypatch, lambda: hv.verify(
            inp["zt"], inp["zd"], inp["x"], inp["u"] if mode == "stochastic" else None, mode=mode,
            fly_theta=0.2, fly_window=1, est_params=_est(3), want_pos_stats=True, want_feature=True,
            want_conf=True))
        assert st == 0, (mode, st)
        _same(ref, got)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_misaligned_rows_masked_logits_and_max_K(monkeypatch, dt):
    B, K, V = 6, 3, 5001
    base = _rand(B, K, V + 3, dt, seed=9200)
    zt_big = base["zt"].reshape(-1)[1:1 + B * (K + 1) * (V + 3) - 3]
    zt = torch.as_strided(zt_big, (B, K + 1, V), ((K + 1) * (V + 3), V + 3, 1))
    zd = base["zd"][:, :, :V]
    x = torch.remainder(base["x"], V).to(torch.int32)
    ref, got, st = _both(monkeypatch, lambda: hv.verify(zt, zd, x, base["u"], want_pos_stats=True))
    assert st == 0
    _same(ref, got)
    inp = _rand(16, 4, 3000, dt, seed=9201)
    gen = torch.Generator(device=DEV).manual_seed(5)
    inp["zt"] = inp["zt"].masked_fill(torch.rand(inp["zt"].shape, generator=gen, device=DEV) < 0.3, float("-inf"))
    ref, got, st = _both(monkeypatch, lambda: hv.verify(inp["zt"], inp["zd"], inp["x"], inp["u"],
                                                         est_params=_est(4), want_pos_stats=True,
                                                         want_feature=True, want_conf=True))
    assert st == 0
    _same(ref, got)
    inp = _rand(3, sv.MAX_K, 3000, dt, seed=9202, sigma_d=0.05)
    ref, got, st = _both(monkeypatch, lambda: hv.verify(inp["zt"], inp["zd"], inp["x"], inp["u"],
                                                         want_pos_stats=True))
    assert st == 0
    _same(ref, got)


def test_pruned_batch_and_queue_tail(monkeypatch):
    w = workloads.ESTIMATOR.scaled(B=64)
    inp = workloads.make_inputs(w, 9300, DEV)
    dl = torch.tensor(np.random.default_rng(3).integers(0, w.K + 1, w.B).astype(np.int32), device=DEV)
    for draft_len in (None, dl):
        ref, got, st = _both(monkeypatch, lambda: hv.verify(inp["zt"], inp["zd"], inp["x"], inp["u"],
                                                             est_params=_est(w.K), want_feature=True,
                                                             want_conf=True, draft_len=draft_len))
        assert st == 0
        _same(ref, got)


@pytest.mark.parametrize("top_p", [None, 0.9])
def test_temperature_and_top_p(monkeypatch, top_p):
    for V, dt in ((128256, "bf16"), (5003, "f32")):
        w = workloads.Workload("checked_t", B=8, K=4, V=V, dtype=dt, mode="stochastic", inv_temp_range=(0.5, 2.0))
        inp = workloads.make_inputs(w, 9400 + V, DEV)
        ref, got, st = _both(monkeypatch, lambda: hv.verify(inp["zt"], inp["zd"], inp["x"], inp["u"],
                                                             est_params=_est(4), want_pos_stats=True,
                                                             want_feature=True, want_conf=True,
                                                             inv_temperature=inp["inv_temp"], top_p=top_p))
        assert st == 0
        _same(ref, got)


def test_fly_full_width_and_confidence(monkeypatch):
    inp = workloads.make_inputs(workloads.FLY.scaled(B=16), 9500, DEV)
    ref, got, st = _both(monkeypatch, lambda: hv.verify(inp["zt"], None, inp["x"], None, mode="fly",
                                                         fly_theta=0.3, fly_window=6, want_pos_stats=True))
    assert st == 0
    _same(ref, got)
    est = _est(workloads.FLY.K)
    a = hv.confidence(inp["zd"], est)
    torch.cuda.synchronize()
    with monkeypatch.context() as m:
        m.setattr(_native, "_lib", _native.lib_checked())
        b = hv.confidence(inp["zd"], est)
        torch.cuda.synchronize()
    assert torch.equal(_bits(a[0]), _bits(b[0])) and torch.equal(_bits(a[1]), _bits(b[1]))
