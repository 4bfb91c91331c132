"""Pins of the oracle's multi-token reading (CPU only).

Reading: a request's seq_len counts all next_n query tokens, and token j sees
its causal prefix of seq_len - (next_n - 1 - j) tokens.  The pins fix that rule
by a hand-worked case, by the prefix structure it implies when every token
carries the same query, and by the last token reducing to the single-token
indexer; a planted off-by-one in the causal shift must fail one of them.
"""
import numpy as np
import pytest

from sparse_attention_paged_dsa_gb300 import inputs as I


def _case(seqs, next_n, seed=3, max_context=2048, num_pages=40, dist="normal"):
    base = I.make_case(name="mtp", batch=len(seqs), max_context=max_context, seq_lens=seqs,
                       num_pages=num_pages, k=16, seed=seed, key_dist=dist)
    return base, I.with_next_n(base, next_n, dist=dist)


def test_live_counts_by_hand(oracle):
    """seq_len 5 with 2 tokens: token 0 sees 4 tokens (1 key), token 1 sees 5 (2 keys).
    seq_len 1 with 3 tokens: tokens 0 and 1 see nothing, token 2 sees 1 token (1 key)."""
    base, c = _case([5, 1, 8], 3)
    s = oracle.case_scores_mtp(c)
    live = np.isfinite(s).sum(axis=2)
    # seq 5: tokens see 3, 4, 5 tokens -> 1, 1, 2 keys; seq 1: 0, 0, 1; seq 8: 6, 7, 8 -> 2, 2, 2
    np.testing.assert_array_equal(live, [[1, 1, 2], [0, 0, 1], [2, 2, 2]])


def test_last_token_is_the_single_token_indexer(oracle):
    base, c = _case([2048, 700, 3, 0], 4)
    s = oracle.case_scores_mtp(c)
    np.testing.assert_array_equal(s[:, -1], oracle.case_scores(base))


def test_same_query_for_every_token_gives_nested_prefixes(oracle):
    base, c = _case([2048, 1001, 1000, 999, 998, 17], 4, seed=5)
    q = np.repeat(base.q[:, None], 4, axis=1)
    w = np.repeat(base.w[:, None], 4, axis=1)
    s = oracle.scores_mtp(q, w, base.key_pool, base.page_table, base.seq_lens, base.max_context)
    full = oracle.case_scores(base)
    for j in range(4):
        n_j = np.array([I_live(L - (3 - j)) for L in base.seq_lens])
        for b in range(base.batch):
            np.testing.assert_array_equal(s[b, j, :n_j[b]], full[b, :n_j[b]])
            assert np.all(np.isneginf(s[b, j, n_j[b]:]))


def I_live(L):
    return (L + 3) // 4 if L > 0 else 0


def test_topk_per_token_uses_its_own_length(oracle):
    base, c = _case([2048, 64, 30], 2, seed=7)
    s = oracle.case_scores_mtp(c)
    t = oracle.topk_mtp(s, c.seq_lens, c.max_context, 16)
    for b, L in enumerate(c.seq_lens):
        for j in range(2):
            n = I_live(L - (1 - j))
            expect = np.sort(np.lexsort((np.arange(n), -s[b, j, :n]))[:min(16, n)])
            got = t[b, j]
            np.testing.assert_array_equal(got[:len(expect)], expect)
            assert np.all(got[len(expect):] == -1)


def test_planted_causal_shift_slip_fails_a_pin(oracle, monkeypatch):
    """Shift every token's prefix by one token too many; the hand-worked counts must catch it."""
    from oracle import oracle as o
    real = o.scores

    def slipped(q, w, key_pool, page_table, seq_lens, max_context):
        return real(q, w, key_pool, page_table, np.maximum(np.asarray(seq_lens) - 1, 0).astype(np.int32),
                    max_context)
    monkeypatch.setattr(o, "scores", slipped)
    with pytest.raises(AssertionError):
        test_live_counts_by_hand(o)
