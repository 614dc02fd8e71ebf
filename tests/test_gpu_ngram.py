"""GPU parity of n-gram (prompt-lookup) drafting (spec_ngram_draft), alone and
as the drafter of FLy verification, against the oracle.

"Speculative Decoding: как черновая модель ускоряет генерацию LLM без потери
качества", "N-gram (prompt lookup)"; "Training-Free Loosely Speculative
Decoding", "Aceleração Multinível" (FLy drafts with prompt lookup). Integer
work: the drafts are compared exactly; the verification uses the parity
contract of tests/helpers.py.
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import compare
import helpers as hv

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _sv():
    import speculative_decoding_token_verify_gb300 as sv
    sv.build()
    return sv


def _contexts(rng, B, ld, vocab, plant=True):
    ctx = rng.integers(0, vocab, (B, ld)).astype(np.int32)
    if plant:
        for b in range(0, B, 2):
            n = min(int(rng.integers(4, 40)), ld // 2)
            a = int(rng.integers(0, ld // 2 - n + 1))
            if n > 0:
                ctx[b, ld - n:] = ctx[b, a:a + n]
    lens = rng.integers(0, ld + 1, B).astype(np.int32)
    lens[: min(B, 4)] = [0, 1, 2, ld][: min(B, 4)]
    return ctx, lens


@pytest.mark.parametrize("B,ld,vocab,n_min,n_max,K", [(1, 5, 3, 1, 2, 3), (64, 512, 7, 1, 4, 8),
                                                       (256, 4096, 50, 2, 6, 8), (33, 1000, 2, 1, 8, 40),
                                                       (128, 2048, 32000, 1, 3, 5)])
def test_ngram_matches_oracle(B, ld, vocab, n_min, n_max, K):
    sv = _sv()
    rng = np.random.default_rng(B + ld + vocab)
    ctx, lens = _contexts(rng, B, ld, vocab)
    g = sv.ngram_draft(torch.tensor(ctx, device=DEV), torch.tensor(lens, device=DEV), n_min, n_max, K)
    torch.cuda.synchronize()
    toks, dl = oracle.ngram_draft(ctx, lens, n_min, n_max, K)
    np.testing.assert_array_equal(g["draft_tokens"].cpu().numpy(), toks)
    np.testing.assert_array_equal(g["draft_len"].cpu().numpy(), dl)


@pytest.mark.parametrize("mode", ["fly", "greedy"])
def test_prompt_lookup_drafts_verified(mode):
    """One decoding step of FLy with prompt-lookup drafts: the GPU pipeline
    (spec_ngram_draft, then spec_verify_ragged) against the oracle pipeline
    on the same seeded contexts and target logits."""
    sv = _sv()
    w = workloads.FLY
    w = type(w)(**{**w.__dict__, "B": 32, "V": 32000})
    inp = workloads.make_inputs(w, 5150, DEV)
    rng = np.random.default_rng(7)
    ctx, lens = _contexts(rng, w.B, 1024, w.V)
    lens[:] = np.maximum(lens, 16)
    d = sv.ngram_draft(torch.tensor(ctx, device=DEV), torch.tensor(lens, device=DEV), 1, 4, w.K)
    kw = dict(fly_theta=w.fly_theta, fly_window=w.fly_window) if mode == "fly" else {}
    g = hv.verify(inp["zt"], None, d["draft_tokens"], None, mode=mode, want_pos_stats=True,
                  draft_len=d["draft_len"], **kw)
    torch.cuda.synchronize()
    toks, dl = oracle.ngram_draft(ctx, lens, 1, 4, w.K)
    assert dl.sum() > 0
    om = oracle.FLY if mode == "fly" else oracle.GREEDY
    r = oracle.verify(workloads.to_numpy_logits(inp["zt"]), None, toks, None, mode=om, draft_len=dl, **kw)
    compare(g, r, w.dtype)
