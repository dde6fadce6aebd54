"""The seeded input generators keep the recipe they state (CPU only).

Trees: topological parent arrays; the DDTree-shaped generator seeds the
rank-0 chain, gives a node at most top_k children with distinct tokens and
stays within its depth limit.  Layer inputs: q and k unit-norm per head up to
bf16 rounding, beta in (0, 1), log alpha < 0, quantised caches inside their
code ranges with positive finite fp16 scales.  The same seed gives the same
inputs.
"""
import numpy as np
import pytest

import synth


def _check_topological(parent):
    assert parent[0] == -1
    for i in range(1, len(parent)):
        assert 0 <= parent[i] < i


@pytest.mark.parametrize("n", [1, 2, 7, 22, 48, 64])
def test_ddtree_shape(n):
    rng = np.random.default_rng(n)
    for _ in range(5):
        parent, tokens = synth.ddtree(rng, n, 1000)
        assert len(parent) == n and len(tokens) == n
        _check_topological(parent)
        depth = synth.tree_depths(parent)
        assert depth.max(initial=0) <= 12
        kids = {}
        for i in range(1, n):
            kids.setdefault(int(parent[i]), []).append(i)
        for p, cs in kids.items():
            assert len(cs) <= 4
            assert len({int(tokens[c]) for c in cs}) == len(cs)   # distinct top-K candidates
        if n > 1:
            # chain seed: nodes 1, 2, ... continue the chain from the root
            # down to the deepest level the tree reaches
            c = 1
            while c < n and parent[c] == c - 1:
                c += 1
            assert c - 1 == depth.max()
        assert np.all((tokens >= 0) & (tokens < 1000))


def test_other_trees_and_batching():
    rng = np.random.default_rng(3)
    u = synth.uniform_tree(rng, 30)
    _check_topological(u)
    ch = synth.chain_tree(9)
    assert list(ch) == list(range(-1, 8))
    assert synth.deepest_path(ch) == list(range(9))
    p = synth.ddtree(rng, 22, 100)[0]
    dp = synth.deepest_path(p)
    d = synth.tree_depths(p)
    assert dp[0] == 0 and d[dp[-1]] == d.max() and len(dp) == d.max() + 1
    for a, b in zip(dp, dp[1:]):
        assert p[b] == a
    par, nn = synth.batch_trees([u, ch], 32)
    assert par.shape == (2, 32) and list(nn) == [30, 9]
    assert np.all(par[0, 30:] == -1) and np.all(par[1, 9:] == -1)


def test_gdn_inputs_recipe():
    rng = np.random.default_rng(4)
    g = synth.gdn_inputs(rng, 2, 22, 4, 12, 128, 64)
    for k in ("q", "k"):
        x = synth.bf16_to_f32(g[k]).astype(np.float64)
        assert x.shape == (2, 22, 4, 128)
        np.testing.assert_allclose(np.linalg.norm(x, axis=-1), 1.0, atol=4e-3)
    assert g["v"].shape == (2, 22, 12, 64) and g["v"].dtype == np.uint16
    assert np.all((g["beta"] > 0) & (g["beta"] < 1))
    assert np.all(g["log_alpha"] < 0)
    assert g["state"].shape == (2, 12, 64, 128) and g["state"].dtype == np.float32
    assert 0.015 < float(g["state"].std()) < 0.025


@pytest.mark.parametrize("kv_type", [synth.KV_Q8_0, synth.KV_Q4_0, synth.KV_Q8_0_Q4_0, synth.KV_Q4_0_Q8_0,
                                     synth.KV_TQ3_0])
def test_kv_cache_recipe(kv_type):
    rng = np.random.default_rng(5)
    D = 128
    c = synth.kv_cache(rng, 2, 3, 40, D, kv_type)
    widths = {synth.KV_Q8_0: (D, D), synth.KV_Q4_0: (D // 2, D // 2), synth.KV_Q8_0_Q4_0: (D, D // 2),
              synth.KV_Q4_0_Q8_0: (D // 2, D), synth.KV_TQ3_0: (D // 32 * 12, D // 32 * 12)}[kv_type]
    for plane, w in zip(("kq", "vq"), widths):
        a = c[plane]
        assert a.shape == (2, 3, 40, w)
        if w == D:
            assert a.dtype == np.int8 and a.min() >= -127
        else:
            assert a.dtype == np.uint8
    for plane in ("ks", "vs"):
        s = c[plane].view(np.float16).astype(np.float64)
        assert s.shape == (2, 3, 40, D // 32)
        assert np.all(np.isfinite(s)) and np.all(s >= 0)


def test_same_seed_same_inputs():
    a = synth.gdn_inputs(np.random.default_rng(9), 1, 7, 2, 2, 16, 16)
    b = synth.gdn_inputs(np.random.default_rng(9), 1, 7, 2, 2, 16, 16)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])
    x = synth.draft_logits(np.random.default_rng(10), 1, 4, 300)
    y = synth.draft_logits(np.random.default_rng(10), 1, 4, 300)
    np.testing.assert_array_equal(x, y)
    assert x.shape == (1, 4, 300) and x.dtype == np.float32
