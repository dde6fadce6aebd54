"""Pins for the oracle's greedy acceptance, KV commit and the step as a whole.

Greedy acceptance: the verify skeleton stays argmax and AL counts committed
tokens per draft/verify step (Luce DFlash README, "Scope and limits" and
"Results").  Commit/rollback: after accept the state equals the committed
prefix ("How it works", per-step rollback; SpecLA PR: a chain is a
degenerate tree).
"""
import itertools

import numpy as np
import pytest

import synth


def _accept(orc, logits, tokens, parents):
    N = logits.shape[1]
    parent, n_nodes = synth.batch_trees(parents, N)
    return orc.accept_greedy(logits, tokens, parent, n_nodes)




def test_hand_made_walk(orc):
    # 0 -> {1, 2}; 1 -> 3; 2 -> 4.  Target argmax: root -> token of node 2,
    # node 2 -> token of node 4, node 4 -> 7 (no child) => path 0, 2, 4.
    V = 10
    par = np.array([-1, 0, 0, 1, 2], np.int32)
    tokens = np.array([[9, 3, 5, 6, 1]], np.int32)
    logits = np.zeros((1, 5, V), np.float32)
    logits[0, 0, 5] = 2.0
    logits[0, 2, 1] = 1.0
    logits[0, 4, 7] = 3.0
    logits[0, 1, 6] = 1.0      # node 1 would continue to 3, but is not taken
    path, L, nxt, best = _accept(orc, logits, tokens, [par])
    assert L[0] == 3 and list(path[0, :3]) == [0, 2, 4] and nxt[0] == 7
    assert list(best[0]) == [5, 6, 1, 0, 7]


def test_root_without_matching_child(orc):
    rng = np.random.default_rng(1)
    V = 16
    par = np.array([-1, 0, 0], np.int32)
    tokens = np.array([[0, 3, 4]], np.int32)
    logits = rng.standard_normal((1, 3, V)).astype(np.float32)
    logits[0, 0, 3:5] = -10.0
    path, L, nxt, best = _accept(orc, logits, tokens, [par])
    assert L[0] == 1 and path[0, 0] == 0 and nxt[0] == int(np.argmax(logits[0, 0]))


def test_ties_go_to_lowest_vocab_index_and_lowest_node(orc):
    V = 8
    par = np.array([-1, 0, 0, 1, 2], np.int32)
    tokens = np.array([[0, 2, 2, 6, 6]], np.int32)   # nodes 1 and 2 carry the same token
    logits = np.zeros((1, 5, V), np.float32)
    logits[0, 0, [2, 5]] = 4.0                       # tie -> 2
    logits[0, 1, [6, 7]] = 1.0                       # tie -> 6 -> node 3
    logits[0, 2, 6] = 1.0
    path, L, nxt, best = _accept(orc, logits, tokens, [par])
    assert best[0, 0] == 2 and best[0, 1] == 6
    assert L[0] == 3 and list(path[0, :3]) == [0, 1, 3]   # node 1 (not 2) is taken
    assert nxt[0] == 0


def test_nan_logits_count_as_minus_infinity(orc):
    # A NaN logit never wins unless nothing else can: row 0 has a NaN first
    # and its maximum later, row 1 is all NaN (index 0), row 2 mixes NaN and
    # -inf only (index 0, the lowest of the equal -inf values), row 3 has a
    # NaN after its maximum.  Compared with numpy's argmax after the same
    # substitution, which is an independent statement of the rule.
    V = 9
    par = np.array([-1, 0, 1, 2], np.int32)
    tokens = np.array([[0, 99, 99, 99]], np.int32)
    logits = np.zeros((1, 4, V), np.float32)
    logits[0, 0] = [np.nan, 1.0, 3.0, np.nan, 2.0, 3.0, -1.0, 0.0, np.nan]
    logits[0, 1] = np.nan
    logits[0, 2] = [np.nan, -np.inf, np.nan, -np.inf, np.nan, np.nan, -np.inf, np.nan, np.nan]
    logits[0, 3] = [0.5, 4.0, np.nan, 1.0, 2.0, np.nan, 0.0, 0.0, 0.0]
    _, L, nxt, best = _accept(orc, logits, tokens, [par])
    want = np.argmax(np.where(np.isnan(logits[0]), -np.inf, logits[0]), axis=1)
    assert list(want) == [2, 0, 0, 1]
    assert list(best[0]) == list(want) and L[0] == 1 and nxt[0] == 2


@pytest.mark.parametrize("seed", range(6))
def test_against_bruteforce_over_all_paths(orc, seed):
    # DDTree siblings carry distinct tokens, so at most one child can match
    # and the accepted path is the longest root path whose every step is the
    # target's argmax (np.argmax: first maximum).
    rng = np.random.default_rng(seed)
    V, B = 50, 3
    parents, toks = [], []
    for b in range(B):
        p, t = synth.ddtree(rng, int(rng.integers(1, 23)), V)
        parents.append(p)
        toks.append(t)
    N = max(len(p) for p in parents)
    tokens = np.zeros((B, N), np.int32)
    for b in range(B):
        tokens[b, : len(toks[b])] = toks[b]
    logits = synth.random_logits(rng, B, N, V)
    for b in range(B):
        synth.plant_path(logits, tokens, synth.deepest_path(parents[b])[: int(rng.integers(1, 6))], b)
    path, L, nxt, best = _accept(orc, logits, tokens, parents)
    for b in range(B):
        par, n = parents[b], len(parents[b])
        am = np.argmax(logits[b, :n], axis=1)
        np.testing.assert_array_equal(best[b, :n], am)
        longest = [0]
        for e in range(n):
            chain, c = [], e
            while c >= 0:
                chain.append(c)
                c = par[c]
            chain = chain[::-1]
            if all(tokens[b, chain[m + 1]] == am[chain[m]] for m in range(len(chain) - 1)):
                if len(chain) > len(longest):
                    longest = chain
        assert L[b] == len(longest) and list(path[b, : L[b]]) == longest
        assert nxt[b] == am[longest[-1]]


def test_planted_path_gives_known_length(orc):
    rng = np.random.default_rng(7)
    par, tok = synth.ddtree(rng, 22, 1000)
    planted = synth.deepest_path(par)
    logits = synth.random_logits(rng, 1, 22, 1000)
    synth.plant_path(logits, tok[None], planted)
    path, L, nxt, _ = _accept(orc, logits, tok[None], [par])
    assert L[0] >= len(planted) and list(path[0, : len(planted)]) == planted


# ---------------------------------------------------------------- KV commit
@pytest.mark.parametrize("kv_type", [synth.KV_Q8_0, synth.KV_Q4_0, synth.KV_F32, synth.KV_Q8_0_Q4_0,
                                     synth.KV_Q4_0_Q8_0])
def test_kv_compaction_moves_bytes_including_aliasing(orc, kv_type):
    rng = np.random.default_rng(10 + kv_type)
    B, Hkv, cap, D, P = 2, 3, 24, 64, 9
    cache = synth.kv_cache(rng, B, Hkv, cap, D, kv_type)
    before = synth.copy_cache(cache)
    path = np.full((B, 6), -1, np.int32)
    path[0, :3] = [0, 2, 3]          # dest 2 is also a source (of m = 1)
    path[1, :4] = [0, 1, 4, 5]
    L = np.array([3, 4], np.int32)
    n_past = np.array([P, P + 3], np.int32)
    orc.kv_commit(cache, kv_type, path, L, n_past)
    for key in ("kq", "vq", "ks", "vs"):
        if cache[key] is None:
            continue
        for b in range(B):
            Pb = n_past[b]
            for m in range(L[b]):
                assert np.array_equal(cache[key][b, :, Pb + m], before[key][b, :, Pb + path[b, m]])
            # untouched outside [P, P + L)
            assert np.array_equal(cache[key][b, :, :Pb], before[key][b, :, :Pb])
            assert np.array_equal(cache[key][b, :, Pb + 6:], before[key][b, :, Pb + 6:])


# ---------------------------------------------------------------- whole step
def test_second_step_after_commit_equals_decode_from_scratch(orc):
    """verify -> accept -> commit -> verify again == one verify of the
    accepted chain with the second tree hung below it, from the original
    state and cache (for the second tree's nodes)."""
    rng = np.random.default_rng(11)
    Hk, Hv, dk, dv = 2, 4, 16, 16
    Hq, Hkv, D = 4, 2, 64
    V, P, cap, W = 40, 14, 64, 0
    n1, n2 = 9, 6
    par1, tok1 = synth.ddtree(rng, n1, V)
    par2 = synth.uniform_tree(rng, n2)
    g1 = synth.gdn_inputs(rng, 1, n1, Hk, Hv, dk, dv, state_std=0.3)
    g2 = synth.gdn_inputs(rng, 1, n2, Hk, Hv, dk, dv, state=False)
    a1 = synth.attn_inputs(rng, 1, n1, Hq, Hkv, D)
    a2 = synth.attn_inputs(rng, 1, n2, Hq, Hkv, D)
    cache0 = synth.kv_cache(rng, 1, Hkv, cap, D, synth.KV_Q8_0)
    logits = synth.random_logits(rng, 1, n1, V)
    synth.plant_path(logits, tok1[None], synth.deepest_path(par1))
    p1, nn1 = synth.batch_trees([par1], n1)
    p2, nn2 = synth.batch_trees([par2], n2)

    # step 1
    cache = synth.copy_cache(cache0)
    orc.tree_gdn_verify(p1, nn1, g1["q"], g1["k"], g1["v"], g1["beta"], g1["log_alpha"], g1["state"])
    orc.tree_attn_verify(p1, nn1, np.array([P], np.int32), a1["q"], a1["k_new"], a1["v_new"], cache, W,
                         synth.KV_Q8_0)
    path, L, _, _ = orc.accept_greedy(logits, tok1[None], p1, nn1)
    assert L[0] >= 2
    st = orc.gdn_commit(g1["q"], g1["k"], g1["v"], g1["beta"], g1["log_alpha"], path, L, g1["state"])
    orc.kv_commit(cache, synth.KV_Q8_0, path, L, np.array([P], np.int32))
    P2 = P + int(L[0])
    # step 2 from the committed state
    og = orc.tree_gdn_verify(p2, nn2, g2["q"], g2["k"], g2["v"], g2["beta"], g2["log_alpha"], st)
    oa = orc.tree_attn_verify(p2, nn2, np.array([P2], np.int32), a2["q"], a2["k_new"], a2["v_new"],
                              cache, W, synth.KV_Q8_0)

    # from scratch: accepted chain + tree 2, one verify
    acc = list(path[0, : L[0]])
    Lc = len(acc)
    par_c = np.concatenate([synth.chain_tree(Lc), np.where(par2 < 0, Lc - 1, par2 + Lc)]).astype(np.int32)
    gc = {k: np.concatenate([g1[k][:, acc], g2[k]], axis=1) for k in ("q", "k", "v", "beta", "log_alpha")}
    ac = {k: np.concatenate([a1[k][:, acc], a2[k]], axis=1) for k in ("q", "k_new", "v_new")}
    pc, nc = synth.batch_trees([par_c], Lc + n2)
    og_c = orc.tree_gdn_verify(pc, nc, gc["q"], gc["k"], gc["v"], gc["beta"], gc["log_alpha"], g1["state"])
    oa_c = orc.tree_attn_verify(pc, nc, np.array([P], np.int32), ac["q"], ac["k_new"], ac["v_new"],
                                synth.copy_cache(cache0), W, synth.KV_Q8_0)
    # the committed state is stored in fp32 between steps: agreement to fp32 rounding
    np.testing.assert_allclose(og[0], og_c[0, Lc:], rtol=1e-5, atol=1e-6)
    # attention reads identical bytes in identical order: bitwise
    assert np.array_equal(oa[0], oa_c[0, Lc:])
