"""Oracle of the draft-tree construction -- TEST INFRASTRUCTURE ONLY (the
package rule of ``oracle/__init__.py`` applies).

What it computes, from the pages:
  * The draft proposes, for each of the D positions after the last committed
    token, a distribution over the vocabulary; a tree of at most ``budget``
    nodes spans the top-K candidates at each position, built best-first
    ("Luce DFlash" README, "How it works": DDTree tree verify, budget 22 over
    the top-K branches at each position; SpecLA PR, options table:
    --specla-top-k is the expansion width, default 4).
  * The rank-0 chain is placed first ("How it works": chain pre-seed,
    chain_seed=true).
  * --ddtree-tau is a cumulative log-probability pruning margin (SpecLA PR,
    options table; README server parameters: a confidence margin, off by
    default, 6 with SpecLA).

Readings where the pages are silent:
  * log-probabilities are the log-softmax of the draft's logits per
    position; a node's score is the sum of the log-probabilities of the
    tokens on its root path (the root scores 0);
  * the children of a node at depth d are the top-K tokens of position d+1
    (the draft's positions are predicted jointly, not conditioned on the
    branch), at most K per node, and depth <= D;
  * top-K order: log-probability descending, ties to the lower token id;
  * the chain seed places the rank-0 token of positions 1 .. min(D, budget-1)
    first, as nodes 1, 2, ...; best-first then adds, one at a time, the
    highest-scoring candidate child of any node in the tree, ties to the
    candidate whose parent has the lower node index, then the lower rank;
  * pruning: a candidate at depth d is admitted only if its score is at
    least the chain's score at depth d minus tau (the chain's node is the
    best possible at every depth); tau = None means no pruning; the tree
    may then have fewer than ``budget`` nodes;
  * node indices are insertion order, so parent[i] < i.
"""
from __future__ import annotations

import numpy as np


def draft_topk(logits, K):
    """logits [B][D][V] float32 -> (tok [B][D][K] int32, logp [B][D][K]
    float64, lse [B][D] float64): the K best tokens per position (ties to the
    lower id; decided on the fp32 logits themselves) and their
    log-probabilities logit - logsumexp(logits), in fp64."""
    x32 = np.asarray(logits, np.float32)
    B, D, V = x32.shape
    x = x32.astype(np.float64)
    m = x.max(axis=-1, keepdims=True)
    lse = (m + np.log(np.exp(x - m).sum(axis=-1, keepdims=True)))[..., 0]
    tok = np.zeros((B, D, K), np.int32)
    logp = np.zeros((B, D, K), np.float64)
    ids = np.arange(V)
    for b in range(B):
        for d in range(D):
            # primary key: value descending; secondary: id ascending
            order = np.lexsort((ids, -x32[b, d]))[:K]
            tok[b, d] = order
            logp[b, d] = x[b, d, order] - lse[b, d]
    return tok, logp, lse


def build_ddtree(tok, logp, root_token, budget, tau=None):
    """Best-first tree with chain seed for every sequence.

    tok, logp [B][D][K] (from draft_topk), root_token [B] ->
    dict(parent [B][budget] int32 (-1 padding), tokens [B][budget] int32
    (-1 padding), n_nodes [B] int32, score [B][budget] float64,
    depth [B][budget] int32, rank [B][budget] int32, margin [B] float64).
    ``margin`` is the smallest gap, over all best-first steps, between the
    chosen candidate's score and the best other candidate's (inf if a step
    had one candidate): a precision tie shows up as a tiny margin."""
    tok = np.asarray(tok)
    logp = np.asarray(logp, np.float64)
    B, D, K = tok.shape
    out = dict(parent=np.full((B, budget), -1, np.int32), tokens=np.full((B, budget), -1, np.int32),
               n_nodes=np.zeros(B, np.int32), score=np.zeros((B, budget)), depth=np.zeros((B, budget), np.int32),
               rank=np.zeros((B, budget), np.int32), margin=np.full(B, np.inf))
    for b in range(B):
        parent, tokens, score, depth, rank = [-1], [int(root_token[b])], [0.0], [0], [0]
        chain_score = np.concatenate([[0.0], np.cumsum(logp[b, :, 0])])  # the chain's score per depth
        # the chain seed
        for d in range(1, min(D, budget - 1) + 1):
            parent.append(d - 1)
            tokens.append(int(tok[b, d - 1, 0]))
            score.append(score[-1] + logp[b, d - 1, 0])
            depth.append(d)
            rank.append(0)
        # the next rank each node offers: a node's children enter in rank
        # order, since the top-K log-probabilities are sorted.  Every chain
        # node's rank-0 child is the next chain node; the last chain node's
        # is still open (it only matters when the chain stopped short of D).
        n_chain = len(parent) - 1
        next_rank = [1] * len(parent)
        if n_chain < D:
            next_rank[n_chain] = 0
        margin = np.inf
        while len(parent) < budget:
            cands = []
            for p in range(len(parent)):
                r = next_rank[p]
                d = depth[p] + 1
                if d > D or r >= K:
                    continue
                s = score[p] + logp[b, d - 1, r]
                if tau is not None and s < chain_score[d] - tau:
                    continue
                cands.append((s, p, r))
            if not cands:
                break
            # best score; ties: lower parent index, then lower rank
            cands.sort(key=lambda c: (-c[0], c[1], c[2]))
            s, p, r = cands[0]
            if len(cands) > 1:
                margin = min(margin, s - cands[1][0])
            parent.append(p)
            tokens.append(int(tok[b, depth[p], r]))
            score.append(s)
            depth.append(depth[p] + 1)
            rank.append(r)
            next_rank[p] = r + 1
            next_rank.append(0)
        n = len(parent)
        out["parent"][b, :n] = parent
        out["tokens"][b, :n] = tokens
        out["n_nodes"][b] = n
        out["score"][b, :n] = score
        out["depth"][b, :n] = depth
        out["rank"][b, :n] = rank
        out["margin"][b] = margin
    return out
