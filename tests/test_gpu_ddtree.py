"""GPU parity: draft-tree construction (libdflv) against the CPU oracle.

The top-K token ids are bit-exact (decided on the fp32 logits on both
sides); log-probabilities within the float tolerance of tests/gpu_util.py
(plus an absolute 1e-5: the kernel's log-sum-exp is fp32).  The tree (parent
array, tokens, node count) is bit-exact whenever every best-first decision of
the oracle is separated from the runner-up by more than 1e-4 in score; at a
closer decision the kernel's fp32 sums may pick the other candidate, and the
test then checks that its tree is a valid best-first tree under the oracle's
scores with that slack.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import dev, host, zeros_status

pytestmark = pytest.mark.gpu

TIE = 1e-4


@pytest.fixture(scope="module")
def dflv():
    import speculative_decoding_tree_layer_gb300 as pkg

    pkg.build()
    pkg.load()
    return pkg


def gpu_build(dflv, logits, root, K, budget, tau):
    B, D, V = logits.shape
    lg, rt = dev(logits), dev(np.asarray(root, np.int32))
    tt = torch.full((B, D, K), -7, dtype=torch.int32, device="cuda")
    tl = torch.full((B, D, K), float("nan"), dtype=torch.float32, device="cuda")
    par = torch.full((B, budget), -7, dtype=torch.int32, device="cuda")
    tok = torch.full((B, budget), -7, dtype=torch.int32, device="cuda")
    nn = torch.zeros(B, dtype=torch.int32, device="cuda")
    sc = torch.full((B, budget), float("nan"), dtype=torch.float32, device="cuda")
    st = zeros_status()
    desc = dflv.ddtree_desc(B, D, V, K, budget, -1.0 if tau is None else tau)
    dflv.check(dflv.dflv_ddtree_build(desc, lg, rt, tt, tl, par, tok, nn, sc, st), "dflv_ddtree_build")
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return dict(topk_tok=host(tt), topk_logp=host(tl), parent=host(par), tokens=host(tok), n_nodes=host(nn),
                score=host(sc))


def check_valid_best_first(g, b, tok, logp, budget, tau):
    """The kernel's tree is a best-first tree under the oracle's fp64 scores,
    choosing within TIE of the best candidate at every step."""
    D, K = logp.shape
    n = int(g["n_nodes"][b])
    chain = np.concatenate([[0.0], np.cumsum(logp[:, 0])])
    n_chain = min(D, budget - 1)
    assert list(g["parent"][b, : n_chain + 1]) == list(range(-1, n_chain))
    depth, rank, score = [0], [0], [0.0]
    for i in range(1, n_chain + 1):
        depth.append(i), rank.append(0), score.append(chain[i])
    nxt = [1] * (n_chain + 1)
    if n_chain < D:
        nxt[n_chain] = 0
    for i in range(n_chain + 1, n + 1):
        cands = []
        for p in range(i):
            dd, r = depth[p] + 1, nxt[p]
            if dd > D or r >= K:
                continue
            sv = score[p] + logp[dd - 1, r]
            if tau is not None and sv < chain[dd] - tau - TIE:
                continue
            cands.append((sv, p))
        if i == n:  # the kernel stopped: nothing clearly admissible may be left
            assert n == budget or all(tau is not None and sv < chain[depth[p] + 1] - tau + TIE for sv, p in cands)
            break
        p = int(g["parent"][b, i])
        best = max(c[0] for c in cands)
        mine = [c for c in cands if c[1] == p]
        assert mine and mine[0][0] >= best - TIE, (i, p)
        dd, r = depth[p] + 1, nxt[p]
        assert g["tokens"][b, i] == tok[dd - 1, r]
        depth.append(dd), rank.append(r), score.append(mine[0][0])
        nxt[p] = r + 1
        nxt.append(0)


CASES = [
    # (B, D, V, K, budget, tau)
    (1, 16, 151936, 4, 22, 6.0),     # the benchmark's draft: block 16, vocab 151,936, top-4, budget 22, tau 6
    (1, 16, 151936, 4, 22, None),
    (2, 16, 151936, 4, 64, None),    # the widest budget
    (3, 8, 32000, 8, 40, 3.0),
    (2, 5, 1000, 3, 64, None),       # budget above what the tree can hold (5 + 3 * ... nodes)
    (2, 12, 4096, 1, 22, None),      # width one: the chain
    (2, 1, 256, 4, 22, None),        # one position: a star
    (1, 16, 512, 2, 1, None),        # the root alone
    (8, 16, 151936, 4, 22, 6.0),     # a batch of 8 sequences
]


@pytest.mark.parametrize("case", CASES)
def test_ddtree_build_matches_oracle(dflv, orc, case):
    B, D, V, K, budget, tau = case
    rng = np.random.default_rng(2000 + CASES.index(case))
    logits = synth.draft_logits(rng, B, D, V)
    root = rng.integers(0, V, size=B).astype(np.int32)
    g = gpu_build(dflv, logits, root, K, budget, tau)
    tok, logp, _ = orc.draft_topk(logits, K)
    np.testing.assert_array_equal(g["topk_tok"], tok)
    np.testing.assert_allclose(g["topk_logp"], logp, rtol=2e-3, atol=1e-5)
    ref = orc.build_ddtree(tok, logp, root, budget, tau)
    for b in range(B):
        if ref["margin"][b] > TIE:
            n = int(ref["n_nodes"][b])
            assert int(g["n_nodes"][b]) == n
            np.testing.assert_array_equal(g["parent"][b], ref["parent"][b])
            np.testing.assert_array_equal(g["tokens"][b], ref["tokens"][b])
            np.testing.assert_allclose(g["score"][b, :n], ref["score"][b, :n], rtol=2e-3, atol=1e-4)
        else:
            check_valid_best_first(g, b, tok[b], logp[b], budget, tau)
        assert g["tokens"][b, 0] == root[b]


def test_ddtree_ties_go_to_the_lower_token_id(dflv, orc):
    # exact ties in the logits across CTA boundaries of the vocabulary split
    B, D, V, K = 1, 4, 151936, 4
    logits = np.zeros((B, D, V), np.float32)
    logits[0, :, [150000, 7, 90000, 40000, 3]] = 5.0
    logits[0, :, 120000] = 6.0
    g = gpu_build(dflv, logits, [1], K, 22, None)
    tok, _, _ = orc.draft_topk(logits, K)
    np.testing.assert_array_equal(g["topk_tok"], tok)
    assert list(g["topk_tok"][0, 0]) == [120000, 3, 7, 40000]


def test_tree_feeds_verify_and_accept(dflv, orc):
    # the built tree is a valid verify input: accept over it walks the chain
    # when the target agrees with the draft's rank-0 tokens
    rng = np.random.default_rng(77)
    B, D, V, K, budget = 1, 16, 4096, 4, 22
    logits = synth.draft_logits(rng, B, D, V)
    g = gpu_build(dflv, logits, [5], K, budget, 6.0)
    n = int(g["n_nodes"][0])
    n_chain = min(D, budget - 1)
    assert n >= n_chain + 1
    target = np.full((B, budget, V), -1.0, np.float32)
    for i in range(n_chain):  # after chain node i the target wants chain node i+1's token
        target[0, i, g["tokens"][0, i + 1]] = 1.0
    parent = dev(g["parent"])
    nn = dev(g["n_nodes"])
    path = torch.zeros((B, budget), dtype=torch.int32, device="cuda")
    plen = torch.zeros(B, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(B, dtype=torch.int32, device="cuda")
    best = torch.zeros((B, budget), dtype=torch.int32, device="cuda")
    st = zeros_status()
    dflv.check(dflv.dflv_accept_greedy(B, budget, V, dev(target), dev(g["tokens"]), parent, nn, path, plen, nxt,
                                       best, st))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    L = int(plen.item())
    assert L == n_chain + 1 and list(host(path)[0, :L]) == list(range(L))
