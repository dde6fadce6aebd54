"""GPU parity: the tree-aware short convolution and its commit (libdflv)
against the CPU oracle.

Outputs within the float tolerance of tests/gpu_util.py, over several CTAs
of channels with a ragged tail and at the 27B layer's full width; the
committed conv state bit-exact (it is a gather of bf16 values); malformed
trees and paths reported through the device status word.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import assert_close, dev, host, zeros_status

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dflv():
    import speculative_decoding_tree_layer_gb300 as pkg

    pkg.build()
    pkg.load()
    return pkg


def _trees(rng, ns, kind):
    if kind == "chain":
        return [synth.chain_tree(n) for n in ns]
    if kind == "ddtree":
        return [synth.ddtree(rng, n, 64)[0] if n > 1 else np.array([-1], np.int32) for n in ns]
    return [synth.uniform_tree(rng, n) for n in ns]


def gpu_conv(dflv, parent, n_nodes, d, flags=0, expect_status=0):
    B, N = parent.shape
    C, K = d["w"].shape
    out = torch.full((B, N, C), float("nan"), dtype=torch.float32, device="cuda")
    st = zeros_status()
    keep = dict(parent=dev(parent), n_nodes=dev(n_nodes), x=dev(d["x"]), state=dev(d["state"]), w=dev(d["w"]))
    rc = dflv.dflv_tree_conv_verify(dflv.conv_desc(B, N, C, K, flags), keep["parent"], keep["n_nodes"], keep["x"],
                                    keep["state"], keep["w"], out, st)
    dflv.check(rc, "dflv_tree_conv_verify")
    torch.cuda.synchronize()
    assert int(st.item()) == expect_status
    return host(out)


CASES = [
    # (B, n list, C, K, tree kind)
    (1, [7], 16, 4, "uniform"),
    (2, [22, 9], 600, 4, "ddtree"),          # 2 full CTAs of channels + a ragged one
    (2, [1, 2], 260, 2, "uniform"),          # a lone root; 4 channels in the last CTA
    (1, [64], 1028, 8, "chain"),             # depth 63, widest window
    (3, [13, 64, 40], 516, 5, "uniform"),
    (1, [22], 10240, 4, "ddtree"),           # the 27B layer's q/k/v channels
    (8, [64] * 8, 10240, 4, "ddtree"),       # widest trees, batch 8
]


@pytest.mark.parametrize("case", CASES)
def test_tree_conv_matches_oracle(dflv, orc, case):
    B, ns, C, K, kind = case
    rng = np.random.default_rng(1000 + CASES.index(case))
    N = max(ns)
    parent, n_nodes = synth.batch_trees(_trees(rng, ns, kind), N)
    d = synth.conv_inputs(rng, B, N, C, K)
    got = gpu_conv(dflv, parent, n_nodes, d)
    ref = orc.tree_conv_verify(parent, n_nodes, d["x"], d["state"], d["w"])
    for b in range(B):
        assert_close(got[b, : n_nodes[b]], ref[b, : n_nodes[b]], what=f"conv out[b={b}]")


def test_tree_conv_early_prefetch_back_to_back(dflv, orc):
    # Several layers' convolutions back to back with the early-prefetch flag:
    # each reads its own taps and state before its dependency wait.
    rng = np.random.default_rng(41)
    B, N, C, K, n_layers = 2, 22, 10240, 4, 4
    parent, n_nodes = synth.batch_trees([synth.ddtree(rng, N, 64)[0], synth.uniform_tree(rng, 15)], N)
    layers = [synth.conv_inputs(rng, B, N, C, K) for _ in range(n_layers)]
    par_d, nn_d = dev(parent), dev(n_nodes)
    keep = [{k: dev(v) for k, v in d.items()} for d in layers]
    outs = [torch.full((B, N, C), float("nan"), dtype=torch.float32, device="cuda") for _ in layers]
    st = zeros_status()
    for li, kd in enumerate(keep):
        flags = 0 if li == 0 else dflv.DFLV_FLAG_EARLY_PREFETCH
        dflv.check(dflv.dflv_tree_conv_verify(dflv.conv_desc(B, N, C, K, flags), par_d, nn_d, kd["x"], kd["state"],
                                              kd["w"], outs[li], st))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for li, d in enumerate(layers):
        ref = orc.tree_conv_verify(parent, n_nodes, d["x"], d["state"], d["w"])
        got = host(outs[li])
        for b in range(B):
            assert_close(got[b, : n_nodes[b]], ref[b, : n_nodes[b]], what=f"layer {li} b={b}")


def test_tree_conv_bad_topology_sets_status(dflv):
    rng = np.random.default_rng(3)
    parent = np.array([[-1, 0, 2, 1], [-1, 0, 1, 2]], np.int32)  # node 2 of sequence 0 is its own parent
    n_nodes = np.array([4, 4], np.int32)
    d = synth.conv_inputs(rng, 2, 4, 256, 4)
    got = gpu_conv(dflv, parent, n_nodes, d, expect_status=dflv.DFLV_DEV_TOPOLOGY)
    assert np.all(np.isnan(got[0]))     # sequence 0 wrote nothing
    assert np.all(np.isfinite(got[1]))  # sequence 1 is unaffected


@pytest.mark.parametrize("K", [2, 4, 8])
def test_conv_commit_matches_oracle(dflv, orc, K):
    rng = np.random.default_rng(50 + K)
    B, N, C, n_layers = 4, 22, 10240 + 4 * K, 3
    parents = [synth.ddtree(rng, N, 64)[0] for _ in range(B)]
    parent, n_nodes = synth.batch_trees(parents, N)
    # accepted paths of lengths 0, 1, a few, the deepest
    lens = [0, 1, min(3, K), len(synth.deepest_path(parents[3]))]
    path = np.zeros((B, N), np.int32)
    for b in range(B):
        dp = synth.deepest_path(parents[b])[: lens[b]]
        path[b, : len(dp)] = dp
        lens[b] = len(dp)
    path_len = np.array(lens, np.int32)
    layers = [synth.conv_inputs(rng, B, N, C, K) for _ in range(n_layers)]
    states = [dev(d["state"]) for d in layers]
    xs = [dev(d["x"]) for d in layers]
    st = zeros_status()
    dflv.check(dflv.dflv_conv_commit(dflv.conv_desc(B, N, C, K), n_layers, states, xs, dev(path), dev(path_len), st))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for li, d in enumerate(layers):
        ref = orc.conv_commit(d["x"], path, path_len, d["state"])
        np.testing.assert_array_equal(host(states[li], np.uint16), ref)


def test_conv_commit_then_verify_continues_the_sequence(dflv, orc):
    # verify -> accept a path -> commit -> verify a chain from the new state
    # equals one oracle chain over [accepted inputs ; next inputs].
    rng = np.random.default_rng(61)
    N, C, K = 22, 1024, 4
    par = synth.ddtree(rng, N, 64)[0]
    parent, n_nodes = synth.batch_trees([par], N)
    d = synth.conv_inputs(rng, 1, N, C, K)
    dp = synth.deepest_path(par)
    path = np.zeros((1, N), np.int32)
    path[0, : len(dp)] = dp
    state = dev(d["state"])
    st = zeros_status()
    dflv.check(dflv.dflv_conv_commit(dflv.conv_desc(1, N, C, K), 1, [state], [dev(d["x"])], dev(path),
                                     dev(np.array([len(dp)], np.int32)), st))
    n2 = 9
    d2 = synth.conv_inputs(rng, 1, n2, C, K)
    p2, nn2 = synth.batch_trees([synth.chain_tree(n2)], n2)
    d2["state"] = host(state, np.uint16)
    got = gpu_conv(dflv, p2, nn2, d2)
    # the same as one chain over the accepted inputs and the new ones
    x_all = np.concatenate([d["x"][:, dp], d2["x"]], axis=1)
    pc, nc = synth.batch_trees([synth.chain_tree(x_all.shape[1])], x_all.shape[1])
    ref = orc.tree_conv_verify(pc, nc, x_all, d["state"], d2["w"])[:, len(dp):]
    assert int(st.item()) == 0
    assert_close(got[0], ref[0], what="continued chain")


def test_conv_commit_bad_path_sets_status(dflv):
    rng = np.random.default_rng(7)
    B, N, C, K = 2, 8, 256, 4
    d = synth.conv_inputs(rng, B, N, C, K)
    path = np.zeros((B, N), np.int32)
    path[0, :3] = [0, 1, 9]          # node 9 is outside [0, N)
    path[1, :2] = [0, 1]
    state = dev(d["state"])
    st = zeros_status()
    dflv.check(dflv.dflv_conv_commit(dflv.conv_desc(B, N, C, K), 1, [state], [dev(d["x"])], dev(path),
                                     dev(np.array([3, 2], np.int32)), st))
    torch.cuda.synchronize()
    assert int(st.item()) == dflv.DFLV_DEV_PATH
    got = host(state, np.uint16)
    np.testing.assert_array_equal(got[0], d["state"][0])   # left unchanged
    assert not np.array_equal(got[1], d["state"][1])       # the valid sequence committed
