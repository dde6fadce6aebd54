"""Seeded synthetic inputs for the DDTree tree-verify step.

This module serves both the CUDA path's tests/benchmarks and the CPU oracle's
tests.  It holds none of the method's arithmetic: it only draws random
tensors with the shapes and distributions of the workloads below and lays
them out as the library's C ABI expects (bf16 and fp16 as uint16 bit
patterns).  Everything is numpy on the host; every generator takes a
``numpy.random.Generator`` so callers control the seed.

Workloads (the pages give the model geometry; the draws are synthetic):
  * gated-DeltaNet layer of a 27B-class hybrid target: 16 q/k heads, 48 v
    heads, dk = dv = 128 ("Luce DFlash" README, "Architecture note": 64
    layers, every 4th full attention, the rest Gated DeltaNet);
  * the short convolution over that layer's q/k/v channels (10240
    channels, width 4: a reading, the pages name the op but not its sizes);
  * full-attention layer: 24 query heads, 4 KV heads, head size 256 (same
    section), over a q8_0 / q4_0 KV cache ("Asymmetric K/V quantization");
  * draft trees built best-first over top-K branches with a rank-0 chain
    pre-seed (README "How it works", DDTree tree verify; SpecLA PR "CLI":
    budget 22, top-k 4).
"""
from __future__ import annotations

import heapq

import numpy as np

KV_Q8_0, KV_Q4_0, KV_F32, KV_Q8_0_Q4_0, KV_Q4_0_Q8_0, KV_TQ3_0 = 0, 1, 2, 3, 4, 5

GDN_27B = dict(Hk=16, Hv=48, dk=128, dv=128)
ATTN_27B = dict(Hq=24, Hkv=4, D=256)
# The short convolution in front of that gated-DeltaNet layer runs over its
# q, k and v channels together (2*16*128 + 48*128); the pages give neither
# the channel count nor the width, the width 4 is the common choice.
CONV_27B = dict(C=2 * 16 * 128 + 48 * 128, K=4)


# ------------------------------------------------------------------ encodings
def bf16_bits(x) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_to_f32(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def f16_bits(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


# ------------------------------------------------------------------ trees
def uniform_tree(rng, n: int) -> np.ndarray:
    """parent[0] = -1, parent[i] ~ U[0, i)."""
    parent = np.full(n, -1, np.int32)
    for i in range(1, n):
        parent[i] = rng.integers(0, i)
    return parent


def chain_tree(n: int) -> np.ndarray:
    parent = np.arange(-1, n - 1, dtype=np.int32)
    return parent


def ddtree(rng, n: int, vocab: int, top_k: int = 4, max_depth: int = 12):
    """Best-first draft tree of ``n`` nodes (root included).

    A random depth limit D ~ U{1..max_depth} is drawn (again until n nodes
    fit).  Each depth d has ``top_k`` distinct candidate tokens with
    descending log-probabilities.  The rank-0 chain is added first (chain
    pre-seed), then the remaining nodes best-first by cumulative
    log-probability, at most ``top_k`` children per node.  Node indices are
    insertion order, so parent[i] < i.  Returns (parent, tokens)."""
    assert n >= 1
    while True:
        D = int(rng.integers(1, max_depth + 1))
        if sum(top_k ** d for d in range(1, D + 1)) >= n - 1:
            break
    toks = np.stack([rng.choice(vocab, size=top_k, replace=False) for _ in range(D + 1)])
    lps = []
    for _ in range(D + 1):
        z = rng.normal(size=top_k + 4) * 2.0
        z = z - z.max()
        lp = z - np.log(np.exp(z).sum())
        lps.append(np.sort(lp)[::-1][:top_k])
    lps = np.stack(lps)

    parent = [-1]
    depth = [0]
    score = [0.0]
    tokens = [int(rng.integers(0, vocab))]
    present = set()

    def add(p, r):
        d = depth[p] + 1
        parent.append(p)
        depth.append(d)
        score.append(score[p] + float(lps[d][r]))
        tokens.append(int(toks[d][r]))
        present.add((p, r))
        return len(parent) - 1

    cur = 0
    for _ in range(D):
        if len(parent) >= n:
            break
        cur = add(cur, 0)
    heap = []
    counter = 0

    def push_children(u):
        nonlocal counter
        if depth[u] >= D:
            return
        for r in range(top_k):
            if (u, r) not in present:
                heapq.heappush(heap, (-(score[u] + float(lps[depth[u] + 1][r])), counter, u, r))
                counter += 1

    for u in range(len(parent)):
        push_children(u)
    while len(parent) < n:
        _, _, u, r = heapq.heappop(heap)
        if (u, r) in present:
            continue
        v = add(u, r)
        push_children(v)
    return np.asarray(parent, np.int32), np.asarray(tokens, np.int32)


def tree_depths(parent) -> np.ndarray:
    """Depth of every node (plain bookkeeping for input recipes)."""
    d = np.zeros(len(parent), np.int32)
    for i in range(1, len(parent)):
        d[i] = d[parent[i]] + 1
    return d


def deepest_path(parent) -> list:
    """Root-to-node path ending at the first deepest node."""
    d = tree_depths(parent)
    e = int(np.argmax(d))
    path = []
    while e >= 0:
        path.append(e)
        e = int(parent[e])
    return path[::-1]


def batch_trees(parents, n_max: int):
    """Stack per-sequence parent arrays into [B][n_max] (padding -1) plus n_nodes."""
    B = len(parents)
    out = np.full((B, n_max), -1, np.int32)
    n_nodes = np.zeros(B, np.int32)
    for b, p in enumerate(parents):
        out[b, : len(p)] = p
        n_nodes[b] = len(p)
    return out, n_nodes


# ------------------------------------------------------------------ GDN layer
def _l2n(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def gdn_inputs(rng, B, N, Hk, Hv, dk, dv, state_std=0.02, state=True):
    """One gated-DeltaNet layer's verify inputs.

    q, k ~ N(0,1) L2-normalised per head, then bf16; v ~ N(0,1) bf16;
    beta = sigmoid(N(0,1)); log_alpha = -softplus(N(0,1)); committed state
    ~ N(0, state_std) fp32."""
    q = bf16_bits(_l2n(rng.standard_normal((B, N, Hk, dk), dtype=np.float32)))
    k = bf16_bits(_l2n(rng.standard_normal((B, N, Hk, dk), dtype=np.float32)))
    v = bf16_bits(rng.standard_normal((B, N, Hv, dv), dtype=np.float32))
    z = rng.standard_normal((B, N, Hv)).astype(np.float64)
    beta = (1.0 / (1.0 + np.exp(-z))).astype(np.float32)
    z = rng.standard_normal((B, N, Hv)).astype(np.float64)
    log_alpha = (-np.logaddexp(0.0, z)).astype(np.float32)
    out = dict(q=q, k=k, v=v, beta=beta, log_alpha=log_alpha)
    if state:
        out["state"] = (rng.standard_normal((B, Hv, dv, dk), dtype=np.float32) * state_std).astype(np.float32)
    return out


# ------------------------------------------------------------------ short convolution
def conv_inputs(rng, B, N, C, K, w_std=0.5):
    """Tree-conv inputs: x [B][N][C] and the conv state [B][K-1][C] as bf16
    ~ N(0, 1), weights [C][K] fp32 ~ N(0, w_std)."""
    return dict(
        x=bf16_bits(rng.standard_normal((B, N, C), dtype=np.float32)),
        state=bf16_bits(rng.standard_normal((B, K - 1, C), dtype=np.float32)),
        w=(rng.standard_normal((C, K), dtype=np.float32) * w_std).astype(np.float32),
    )


# ------------------------------------------------------------------ draft logits
def draft_logits(rng, B, D, V, std=2.0, n_hot=3, boost=(3.0, 9.0)):
    """Draft logits [B][D][V] fp32: N(0, std) plus, at every position,
    n_hot random tokens raised by U(boost) -- a confident head over a flat
    tail, as a trained draft gives."""
    x = (rng.standard_normal((B, D, V), dtype=np.float32) * std).astype(np.float32)
    for b in range(B):
        for d in range(D):
            hot = rng.choice(V, size=n_hot, replace=False)
            x[b, d, hot] += rng.uniform(boost[0], boost[1], size=n_hot).astype(np.float32)
    return x


# ------------------------------------------------------------------ attention layer
def attn_inputs(rng, B, N, Hq, Hkv, D):
    """Tree queries and the tree's new keys/values, bf16 ~ N(0,1)."""
    return dict(
        q=bf16_bits(rng.standard_normal((B, N, Hq, D), dtype=np.float32)),
        k_new=bf16_bits(rng.standard_normal((B, N, Hkv, D), dtype=np.float32)),
        v_new=bf16_bits(rng.standard_normal((B, N, Hkv, D), dtype=np.float32)),
    )


def kv_cache(rng, B, Hkv, cap, D, kv_type, scale_std=0.02):
    """A filled KV cache in the library's plane layout.

    q8_0: int8 codes ~ U[-127, 127], fp16 scales ~ |N(0, scale_std)|;
    q4_0: 4-bit codes ~ U[0, 15] (two per byte), same scales;
    TQ3_0: 3-bit codes ~ U[0, 7] (any byte pattern is 32 valid codes per 12
          bytes), same scales;
    f32:  values ~ N(0, 1), no scale planes;
    the asymmetric types draw each plane in its own format."""
    if kv_type == KV_F32:
        return dict(kq=rng.standard_normal((B, Hkv, cap, D), dtype=np.float32),
                    vq=rng.standard_normal((B, Hkv, cap, D), dtype=np.float32), ks=None, vs=None)
    nb = D // 32

    def scales():
        return f16_bits(np.abs(rng.standard_normal((B, Hkv, cap, nb), dtype=np.float32)) * scale_std)

    def plane(t):
        if t == KV_Q8_0:
            return rng.integers(-127, 128, size=(B, Hkv, cap, D), dtype=np.int8)
        if t == KV_TQ3_0:
            return rng.integers(0, 256, size=(B, Hkv, cap, D // 32 * 12), dtype=np.uint8)
        return rng.integers(0, 256, size=(B, Hkv, cap, D // 2), dtype=np.uint8)

    planes = {KV_Q8_0: (KV_Q8_0, KV_Q8_0), KV_Q4_0: (KV_Q4_0, KV_Q4_0), KV_Q8_0_Q4_0: (KV_Q8_0, KV_Q4_0),
              KV_Q4_0_Q8_0: (KV_Q4_0, KV_Q8_0), KV_TQ3_0: (KV_TQ3_0, KV_TQ3_0)}
    if kv_type not in planes:
        raise ValueError(kv_type)
    kt, vt = planes[kv_type]
    kq = plane(kt)
    vq = plane(vt)
    return dict(kq=kq, vq=vq, ks=scales(), vs=scales())


def copy_cache(c):
    return {k: (None if v is None else v.copy()) for k, v in c.items()}


# ------------------------------------------------------------------ acceptance
def random_logits(rng, B, N, V):
    return rng.standard_normal((B, N, V), dtype=np.float32)


def plant_path(logits, tokens, path, b=0):
    """Make the target's argmax at path[m] equal the token of path[m+1], so a
    greedy walk accepts exactly ``path`` (when siblings carry distinct
    tokens).  Modifies ``logits`` in place."""
    for m in range(len(path) - 1):
        row = logits[b, path[m]]
        row[int(tokens[b, path[m + 1]])] = row.max() + 1.0
    return logits
