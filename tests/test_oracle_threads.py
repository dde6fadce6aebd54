"""The oracle's parallel loops change nothing but the time.

The C oracle runs the independent (sequence, head) pairs of the GDN verify
and commit, and the output rows of attention, on several threads; each unit
is computed in the same order as on one thread, so every result must be
bit-identical to the single-thread one.  (Without OpenMP both runs are the
same serial code and the test holds trivially.)
"""
import os

import numpy as np
import pytest

import synth


@pytest.fixture
def threads(orc):
    many = orc.set_threads(max(4, os.cpu_count() or 1))
    yield many
    orc.set_threads(os.cpu_count() or 1)


def _both(orc, fn):
    orc.set_threads(1)
    one = fn()
    orc.set_threads(max(4, os.cpu_count() or 1))
    many = fn()
    return one, many


def test_gdn_verify_and_commit_do_not_depend_on_threads(orc, threads):
    rng = np.random.default_rng(7)
    B, N, Hk, Hv, dk, dv = 3, 13, 2, 4, 16, 8
    parents = [synth.uniform_tree(rng, 13), synth.chain_tree(5), synth.uniform_tree(rng, 9)]
    parent, n_nodes = synth.batch_trees(parents, N)
    d = synth.gdn_inputs(rng, B, N, Hk, Hv, dk, dv)
    args = (parent, n_nodes, d["q"], d["k"], d["v"], d["beta"], d["log_alpha"], d["state"])
    (o1, s1), (o2, s2) = _both(orc, lambda: orc.tree_gdn_verify(*args, want_states=True))
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(s1, s2)
    path = np.zeros((B, N), np.int32)
    lens = []
    for b, p in enumerate(parents):
        dp = synth.deepest_path(p)
        path[b, : len(dp)] = dp
        lens.append(len(dp))
    c1, c2 = _both(orc, lambda: orc.gdn_commit(d["q"], d["k"], d["v"], d["beta"], d["log_alpha"], path,
                                               np.array(lens, np.int32), d["state"]))
    np.testing.assert_array_equal(c1, c2)


@pytest.mark.parametrize("kv_type", [synth.KV_Q8_0, synth.KV_Q4_0])
def test_attention_does_not_depend_on_threads(orc, threads, kv_type):
    rng = np.random.default_rng(8)
    B, Hq, Hkv, D, P, cap = 2, 4, 2, 64, 70, 96
    parents = [synth.uniform_tree(rng, 11), synth.chain_tree(6)]
    parent, n_nodes = synth.batch_trees(parents, 11)
    inp = synth.attn_inputs(rng, B, 11, Hq, Hkv, D)
    cache = synth.kv_cache(rng, B, Hkv, cap, D, kv_type, scale_std=0.05)
    n_past = np.full(B, P, np.int32)

    def run():
        c = synth.copy_cache(cache)
        out = orc.tree_attn_verify(parent, n_nodes, n_past, inp["q"], inp["k_new"], inp["v_new"], c, 32, kv_type)
        return out, c

    (o1, c1), (o2, c2) = _both(orc, run)
    np.testing.assert_array_equal(o1, o2)
    for k in ("kq", "vq", "ks", "vs"):
        np.testing.assert_array_equal(c1[k], c2[k])
