"""Pins for the oracle's draft-tree construction (oracle/ddtree.py).

DDTree builds a best-first tree of at most `budget` nodes over the top-K
tokens of each draft position, after seeding the rank-0 chain, optionally
pruned by a cumulative log-probability margin tau ("Luce DFlash" README,
"How it works"; SpecLA PR, options table).  The pins tie it to a library
log-sum-exp, to a plain sort for the top-K, and -- the main pin -- to brute
force: because a node's score (the sum of log-probabilities on its root
path) never exceeds its parent's, best-first from the chain selects exactly
the highest-scoring admissible nodes, which enumeration over every rank path
finds without any frontier logic.
"""
import itertools

import numpy as np
import pytest
from scipy.special import logsumexp

import oracle


def _logits(rng, B, D, V, boost=True):
    x = rng.standard_normal((B, D, V)).astype(np.float32) * 2.0
    if boost:  # a few confident tokens per position, like a trained draft
        for b in range(B):
            for d in range(D):
                hot = rng.choice(V, size=3, replace=False)
                x[b, d, hot] += rng.uniform(3.0, 9.0, size=3).astype(np.float32)
    return x


def test_log_probs_match_library_logsumexp():
    rng = np.random.default_rng(0)
    x = _logits(rng, 2, 3, 1000)
    tok, logp, lse = oracle.draft_topk(x, 4)
    np.testing.assert_allclose(lse, logsumexp(x.astype(np.float64), axis=-1), rtol=1e-13)
    for b in range(2):
        for d in range(3):
            np.testing.assert_allclose(logp[b, d], x[b, d, tok[b, d]].astype(np.float64) - lse[b, d], rtol=1e-13)
    # probabilities of the whole vocabulary sum to one
    np.testing.assert_allclose(np.exp(x.astype(np.float64) - lse[..., None]).sum(-1), 1.0, rtol=1e-12)


def test_topk_order_and_ties():
    x = np.zeros((1, 1, 12), np.float32)
    x[0, 0, [9, 3, 7, 1]] = [5.0, 5.0, 4.0, 5.0]   # a three-way tie at the top
    tok, logp, _ = oracle.draft_topk(x, 5)
    assert list(tok[0, 0]) == [1, 3, 9, 7, 0]      # ties go to the lower id
    assert np.all(np.diff(logp[0, 0]) <= 0)
    rng = np.random.default_rng(1)
    x = rng.standard_normal((1, 2, 500)).astype(np.float32)
    tok, _, _ = oracle.draft_topk(x, 6)
    for d in range(2):
        assert list(tok[0, d]) == sorted(range(500), key=lambda v: (-x[0, d, v], v))[:6]


def _bruteforce(tok, logp, budget, tau):
    """Chain + the best admissible non-chain nodes by score, by enumeration
    of every rank path (tiny D and K only).  Returns the tree as a list of
    rank paths in insertion order."""
    D, K = logp.shape
    chain_score = np.concatenate([[0.0], np.cumsum(logp[:, 0])])
    n_chain = min(D, budget - 1)
    chain = [(0,) * d for d in range(1, n_chain + 1)]
    others = []
    for d in range(1, D + 1):
        for path in itertools.product(range(K), repeat=d):
            if all(r == 0 for r in path) and d <= n_chain:
                continue
            # admissible: every node on the path passes its depth's margin
            scores = np.cumsum([logp[e, r] for e, r in enumerate(path)])
            if tau is not None and any(scores[e] < chain_score[e + 1] - tau for e in range(d)):
                continue
            # a path through a missing chain node cannot be reached
            if all(r == 0 for r in path[:-1]) and d - 1 > n_chain:
                continue
            others.append((scores[-1], path))
    others.sort(key=lambda t: -t[0])
    return [()] + chain + [p for _, p in others[: budget - 1 - n_chain]]


def _rank_paths(t, b):
    n = int(t["n_nodes"][b])
    paths = []
    for i in range(n):
        p, path = i, []
        while p > 0:
            path.append(int(t["rank"][b, p]))
            p = int(t["parent"][b, p])
        paths.append(tuple(reversed(path)))
    return paths


@pytest.mark.parametrize("D,K,budget,tau", [(3, 3, 9, None), (4, 2, 12, None), (4, 3, 22, None), (3, 4, 30, None),
                                            (4, 3, 22, 2.0), (4, 3, 22, 0.5), (5, 2, 16, 1.5)])
def test_tree_equals_bruteforce_selection(D, K, budget, tau):
    rng = np.random.default_rng(100 + D * 10 + K)
    for trial in range(4):
        x = _logits(rng, 1, D, 64)
        tok, logp, _ = oracle.draft_topk(x, K)
        t = oracle.build_ddtree(tok, logp, [5], budget, tau)
        want = _bruteforce(tok[0], logp[0], budget, tau)
        got = _rank_paths(t, 0)
        assert got == want, (trial, got, want)
        n = int(t["n_nodes"][0])
        # structure: parents precede children, tokens follow their rank and depth
        for i in range(1, n):
            p = int(t["parent"][0, i])
            assert 0 <= p < i and t["depth"][0, i] == t["depth"][0, p] + 1
            assert t["tokens"][0, i] == tok[0, t["depth"][0, i] - 1, t["rank"][0, i]]
        assert t["tokens"][0, 0] == 5


def test_width_one_is_the_chain():
    rng = np.random.default_rng(3)
    x = _logits(rng, 1, 10, 100)
    tok, logp, _ = oracle.draft_topk(x, 1)
    for budget in (1, 4, 11, 22):
        t = oracle.build_ddtree(tok, logp, [0], budget, None)
        n = min(10, budget - 1) + 1
        assert t["n_nodes"][0] == n
        assert list(t["parent"][0, :n]) == list(range(-1, n - 1))
        assert list(t["tokens"][0, 1:n]) == [int(np.argmax(x[0, d])) for d in range(n - 1)]


def test_single_position_gives_a_star_in_rank_order():
    rng = np.random.default_rng(4)
    x = _logits(rng, 1, 1, 100)
    tok, logp, _ = oracle.draft_topk(x, 4)
    t = oracle.build_ddtree(tok, logp, [0], 22, None)
    assert t["n_nodes"][0] == 5
    assert list(t["parent"][0, :5]) == [-1, 0, 0, 0, 0]
    assert list(t["tokens"][0, 1:5]) == list(tok[0, 0])


def test_zero_margin_keeps_only_the_chain_and_large_margin_prunes_nothing():
    rng = np.random.default_rng(5)
    x = _logits(rng, 2, 8, 300)
    tok, logp, _ = oracle.draft_topk(x, 4)
    t0 = oracle.build_ddtree(tok, logp, [1, 2], 22, 0.0)
    assert list(t0["n_nodes"]) == [9, 9]      # root + 8 chain nodes: every other node scores below the chain
    free = oracle.build_ddtree(tok, logp, [1, 2], 22, None)
    wide = oracle.build_ddtree(tok, logp, [1, 2], 22, 1e9)
    for k in ("parent", "tokens", "n_nodes"):
        np.testing.assert_array_equal(free[k], wide[k])
    assert list(free["n_nodes"]) == [22, 22]


def test_scores_decrease_along_paths_and_best_first_order():
    rng = np.random.default_rng(6)
    x = _logits(rng, 3, 12, 2000)
    tok, logp, _ = oracle.draft_topk(x, 4)
    t = oracle.build_ddtree(tok, logp, [0, 0, 0], 22, 6.0)
    for b in range(3):
        n = int(t["n_nodes"][b])
        n_chain = min(12, 21)
        s = t["score"][b, :n]
        for i in range(1, n):
            assert s[i] <= s[t["parent"][b, i]]
        # non-chain nodes enter in non-increasing score order
        assert np.all(np.diff(s[n_chain + 1:]) <= 0)
