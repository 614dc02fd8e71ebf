"""Pins of the oracle's n-gram (prompt-lookup) drafting.

"Speculative Decoding: как черновая модель ускоряет генерацию LLM без потери
качества", section "N-gram (prompt lookup)": drafts are the tokens that
followed an earlier occurrence, in the prompt or the generated text, of the
context's last tokens. The readings (longest n first, most recent occurrence,
up to K tokens) are pinned against hand cases and an independent search built
on Python's str.rfind over a delimited encoding of the tokens. CPU only.
"""
import numpy as np
import pytest

import oracle


def _rfind_draft(ctx, L, n_min, n_max, K):
    """Independent reference: for n = n_max..n_min, the last occurrence of the
    final n tokens inside ctx[:L-1] (so that it ends before the context does),
    found by str.rfind on ',t1,t2,...,' strings."""
    toks = [int(t) for t in ctx[:L]]
    for n in range(n_max, n_min - 1, -1):
        if n > L - 1:
            continue
        hay = "," + ",".join(map(str, toks[:L - 1])) + ","
        needle = "," + ",".join(map(str, toks[L - n:])) + ","
        pos = hay.rfind(needle)
        if pos < 0:
            continue
        start_tok = hay[:pos + 1].count(",") - 1          # index of the match's first token
        e = start_tok + n
        out = toks[e:e + K]
        return out + [-1] * (K - len(out)), len(out)
    return [-1] * K, 0


def test_hand_cases():
    ctx = np.array([[1, 2, 3, 1, 2, 0, 0],     # "1 2" occurred at 0: propose 3 1 2
                    [5, 5, 5, 5, 0, 0, 0],     # "5 5" last occurred ending at 3: propose the final 5
                    [7, 8, 9, 0, 0, 0, 0],     # no earlier "8 9" or "9": nothing
                    [4, 6, 4, 9, 4, 6, 0]],    # "4 6" at 0 beats "6" alone: propose 4 9 4
                   np.int32)
    toks, dl = oracle.ngram_draft(ctx, [5, 4, 3, 6], 1, 2, 3)
    np.testing.assert_array_equal(toks, [[3, 1, 2], [5, -1, -1], [-1, -1, -1], [4, 9, 4]])
    np.testing.assert_array_equal(dl, [3, 1, 0, 3])


def test_longest_match_wins_over_a_more_recent_shorter_one():
    # "1 2 3" occurs at 0 (follow-up 7); "3" alone occurs later, at 5 (follow-up 8)
    ctx = np.array([[1, 2, 3, 7, 0, 3, 8, 1, 2, 3]], np.int32)
    toks, dl = oracle.ngram_draft(ctx, [10], 1, 3, 2)
    np.testing.assert_array_equal(toks[0], [7, 0])
    toks, dl = oracle.ngram_draft(ctx, [10], 1, 1, 2)        # n = 1 only: the most recent "3"
    np.testing.assert_array_equal(toks[0], [8, 1])


@pytest.mark.parametrize("seed", range(6))
def test_against_an_independent_search(seed):
    rng = np.random.default_rng(seed)
    B, ld, K = 40, 300, 6
    vocab = int(rng.integers(3, 30))
    ctx = rng.integers(0, vocab, (B, ld)).astype(np.int32)
    # plant repeats so that long matches exist
    for b in range(0, B, 3):
        a = int(rng.integers(0, ld // 2))
        ctx[b, ld - 20:] = ctx[b, a:a + 20]
    lens = rng.integers(0, ld + 1, B).astype(np.int32)
    lens[:4] = [0, 1, 2, ld]
    n_min, n_max = int(rng.integers(1, 3)), int(rng.integers(3, 7))
    toks, dl = oracle.ngram_draft(ctx, lens, n_min, n_max, K)
    for b in range(B):
        ref, m = _rfind_draft(ctx[b], int(lens[b]), n_min, n_max, K)
        assert dl[b] == m and list(toks[b]) == ref, (b, lens[b])
