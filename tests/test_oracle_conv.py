"""Pins for the oracle's tree-aware short convolution and its commit.

The op ("Luce DFlash" README, "How it works": ggml_ssm_conv_tree) is the
depthwise causal convolution in front of a gated-DeltaNet layer, evaluated on
a tree: every node reads its K-1 predecessors along its parent chain, and
positions before the root come from the committed conv state.  The pins tie
it to a library convolution (a chain is an ordinary sequence), to a
per-node replay of the root-to-node path, to shifted copies for one-hot
weights, and to sequential decoding across a commit.
"""
import numpy as np
import pytest

import synth


def _conv_seq(seq, w):
    """Causal depthwise conv of a [T][C] sequence with weights [C][K]: output
    t uses seq[t-K+1 .. t], tap K-1 on seq[t]; computed with numpy's
    convolve (full mode), one channel at a time, for t >= K-1."""
    T, C = seq.shape
    K = w.shape[1]
    out = np.zeros((T - K + 1, C))
    for c in range(C):
        # convolve flips its second operand: flip the taps so that tap K-1
        # meets the newest sample
        full = np.convolve(seq[:, c], w[c, ::-1].astype(np.float64), mode="full")
        out[:, c] = full[K - 1:T]
    return out


def _case(rng, parents, C, K):
    N = max(len(p) for p in parents)
    parent, n_nodes = synth.batch_trees(parents, N)
    d = synth.conv_inputs(rng, len(parents), N, C, K)
    return parent, n_nodes, d


@pytest.mark.parametrize("K", [2, 4, 5])
def test_chain_equals_library_convolution(orc, K):
    rng = np.random.default_rng(10 + K)
    n, C = 13, 7
    parent, n_nodes, d = _case(rng, [synth.chain_tree(n)], C, K)
    out = orc.tree_conv_verify(parent, n_nodes, d["x"], d["state"], d["w"])
    seq = np.concatenate([synth.bf16_to_f32(d["state"][0]), synth.bf16_to_f32(d["x"][0])]).astype(np.float64)
    ref = _conv_seq(seq, d["w"])
    np.testing.assert_allclose(out[0], ref, rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tree_equals_per_node_path_replay(orc, seed):
    rng = np.random.default_rng(100 + seed)
    C, K = 5, 4
    parents = [synth.ddtree(rng, 22, 50)[0], synth.uniform_tree(rng, 17), synth.chain_tree(3)]
    parent, n_nodes, d = _case(rng, parents, C, K)
    out = orc.tree_conv_verify(parent, n_nodes, d["x"], d["state"], d["w"])
    for b, par in enumerate(parents):
        st = synth.bf16_to_f32(d["state"][b]).astype(np.float64)
        xb = synth.bf16_to_f32(d["x"][b]).astype(np.float64)
        for i in range(len(par)):
            path = []
            j = i
            while j >= 0:
                path.append(j)
                j = int(par[j])
            seq = np.concatenate([st, xb[path[::-1]]])
            ref = _conv_seq(seq, d["w"])[-1]
            np.testing.assert_allclose(out[b, i], ref, rtol=1e-6, atol=1e-6)


def test_one_hot_taps_give_the_ancestor_at_that_distance(orc):
    # w[c][K-1-dist] = 1: the output is the input `dist` steps up the
    # parent chain, or the conv state once the chain has passed the root.
    rng = np.random.default_rng(7)
    K, C = 4, 3
    par = np.array([-1, 0, 0, 1, 3, 2, 4], np.int32)
    parent, n_nodes, d = _case(rng, [par], C, K)
    xb, st = d["x"][0], d["state"][0]
    for dist in range(K):
        w = np.zeros((C, K), np.float32)
        w[:, K - 1 - dist] = 1.0
        out = orc.tree_conv_verify(parent, n_nodes, d["x"], d["state"], w)
        for i in range(len(par)):
            j, up = i, 0
            while up < dist and j >= 0:
                j, up = int(par[j]), up + 1
            if j >= 0:
                want = synth.bf16_to_f32(xb[j])
            else:
                # up == dist - (depth(i) + 1) steps taken past the root
                depth = int(synth.tree_depths(par)[i])
                want = synth.bf16_to_f32(st[K - 1 - (dist - depth)])
            np.testing.assert_array_equal(out[0, i], want)


def test_padding_nodes_are_untouched(orc):
    rng = np.random.default_rng(3)
    parents = [synth.chain_tree(2), synth.uniform_tree(rng, 9)]
    parent, n_nodes, d = _case(rng, parents, 4, 4)
    out = orc.tree_conv_verify(parent, n_nodes, d["x"], d["state"], d["w"])
    assert np.all(out[0, 2:] == 0.0)


@pytest.mark.parametrize("L", [0, 1, 2, 3, 6])
def test_commit_is_the_tail_of_the_accepted_sequence(orc, L):
    rng = np.random.default_rng(20 + L)
    K, C, n = 4, 6, 9
    d = synth.conv_inputs(rng, 1, n, C, K)
    # the accepted nodes in path order, at scattered node ids
    ids = rng.permutation(n)[:L]
    path = np.zeros((1, n), np.int32)
    path[0, :L] = ids
    st = orc.conv_commit(d["x"], path, np.array([L], np.int32), d["state"])
    seq = np.concatenate([d["state"][0], d["x"][0, ids]])
    np.testing.assert_array_equal(st[0], seq[-(K - 1):])


def test_commit_then_verify_equals_one_long_chain(orc):
    # Decode-order consistency: verifying a chain, committing its first L
    # nodes, then verifying the next nodes from the new state gives what one
    # chain over all the nodes gives at those positions.
    rng = np.random.default_rng(5)
    K, C, n1, n2, L = 4, 8, 10, 6, 7
    d = synth.conv_inputs(rng, 1, n1 + n2, C, K)
    x_all = d["x"]
    parent, n_nodes = synth.batch_trees([synth.chain_tree(n1 + n2)], n1 + n2)
    ref = orc.tree_conv_verify(parent, n_nodes, x_all, d["state"], d["w"])
    # the first L inputs sit at scattered node ids of the first batch
    rng2 = np.random.default_rng(6)
    perm = np.concatenate([[0], 1 + rng2.permutation(n1 - 1)])
    x1 = np.zeros((1, n1, C), np.uint16)
    x1[0, perm] = x_all[0, :n1]
    path = np.zeros((1, n1), np.int32)
    path[0, :L] = perm[:L]
    st = orc.conv_commit(x1, path, np.array([L], np.int32), d["state"])
    x2 = x_all[:, L:L + n2]
    p2, nn2 = synth.batch_trees([synth.chain_tree(n2)], n2)
    out2 = orc.tree_conv_verify(p2, nn2, x2, st, d["w"])
    np.testing.assert_allclose(out2[0], ref[0, L:L + n2], rtol=1e-6, atol=1e-6)


def test_bad_topology_is_rejected(orc):
    rng = np.random.default_rng(0)
    d = synth.conv_inputs(rng, 1, 3, 2, 4)
    parent = np.array([[-1, 2, 1]], np.int32)
    with pytest.raises(orc.OracleError):
        orc.tree_conv_verify(parent, np.array([3], np.int32), d["x"], d["state"], d["w"])
