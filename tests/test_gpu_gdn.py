"""GPU parity: gated-DeltaNet tree verify (libdflv) against the CPU oracle.

Outputs within the float tolerance of tests/gpu_util.py; the captured
factors checked against their definitions (u_i = beta_i (v_i - alpha_i
S_parent k_i), g_i = sum of log alpha over ancestors-or-self, k copied
bitwise); malformed trees reported through the device status word.
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


def gpu_gdn(dflv, parent, n_nodes, inp, Hk, Hv, dk, dv, expect_status=0, flags=0):
    B, N = parent.shape
    keep = {k: dev(v) for k, v in inp.items()}
    keep["parent"], keep["n_nodes"] = dev(parent), dev(n_nodes)
    out = torch.full((B, N, Hv, dv), float("nan"), dtype=torch.float32, device="cuda")
    u = torch.full((B, N, Hv, dv), float("nan"), dtype=torch.float32, device="cuda")
    g = torch.full((B, N, Hv), float("nan"), dtype=torch.float32, device="cuda")
    kc = torch.zeros((B, N, Hk, dk), dtype=torch.int16, device="cuda")
    st = zeros_status()
    rc = dflv.dflv_tree_gdn_verify(dflv.gdn_desc(B, N, Hk, Hv, dk, dv, flags), keep["parent"], keep["n_nodes"],
                                   keep["q"], keep["k"], keep["v"], keep["beta"], keep["log_alpha"],
                                   keep["state"], out, dflv.gdn_factors(u, g, kc), st)
    dflv.check(rc, "dflv_tree_gdn_verify")
    torch.cuda.synchronize()
    assert int(st.item()) == expect_status
    return host(out), host(u), host(g), host(kc, np.uint16)


def oracle_gdn(orc, parent, n_nodes, inp, want_states=False):
    return orc.tree_gdn_verify(parent, n_nodes, inp["q"], inp["k"], inp["v"], inp["beta"], inp["log_alpha"],
                               inp["state"], want_states=want_states)


def compare_valid(got, ref, n_nodes, what):
    e = 0.0
    for b in range(len(n_nodes)):
        e = max(e, assert_close(got[b, : n_nodes[b]], ref[b, : n_nodes[b]], what=f"{what}[b={b}]"))
    return e


CASES = [
    # (B, n list, Hk, Hv, dk, dv, tree kind)
    (1, [7], 2, 2, 16, 16, "uniform"),          # the tiny case's geometry
    (2, [22, 9], 2, 6, 64, 32, "ddtree"),
    (2, [1, 2], 1, 3, 32, 16, "uniform"),
    (1, [64], 4, 8, 128, 64, "ddtree"),
    (1, [64], 1, 2, 128, 128, "chain"),        # depth 63
    (3, [13, 64, 40], 2, 4, 128, 128, "uniform"),
    (2, [22, 31], 2, 4, 128, 128, "ddtree"),    # up to 32 nodes: 64-row blocks
    (1, [32], 1, 2, 64, 64, "chain"),           # one 64-row block per head
    (2, [40, 33], 2, 4, 64, 96, "uniform"),     # over 32 nodes, dv 96: 32-row blocks
    (1, [48], 1, 2, 32, 48, "ddtree"),          # over 32 nodes, dv 48: 16-row blocks
]


@pytest.mark.parametrize("case", CASES)
def test_gdn_tree_verify_matches_oracle(dflv, orc, case):
    B, ns, Hk, Hv, dk, dv, kind = case
    rng = np.random.default_rng(sum(ns) * 7 + dk)
    parents = []
    for n in ns:
        if kind == "chain":
            parents.append(synth.chain_tree(n))
        elif kind == "ddtree":
            parents.append(synth.ddtree(rng, n, 1000)[0])
        else:
            parents.append(synth.uniform_tree(rng, n))
    N = max(ns)
    parent, n_nodes = synth.batch_trees(parents, N)
    inp = synth.gdn_inputs(rng, B, N, Hk, Hv, dk, dv, state_std=0.3)
    out, u, g, kc = gpu_gdn(dflv, parent, n_nodes, inp, Hk, Hv, dk, dv)
    ref, states = oracle_gdn(orc, parent, n_nodes, inp, want_states=True)
    compare_valid(out, ref, n_nodes, "o")
    # factors: g, k copy, u
    f = synth.bf16_to_f32
    for b in range(B):
        n = n_nodes[b]
        par = parent[b]
        la = inp["log_alpha"][b].astype(np.float64)
        gref = np.zeros((n, Hv))
        for i in range(n):
            c = i
            while c >= 0:
                gref[i] += la[c]
                c = par[c]
        np.testing.assert_allclose(g[b, :n], gref, rtol=1e-5, atol=1e-5)
        assert np.array_equal(kc[b, :n], inp["k"][b, :n])
        uref = np.zeros((n, Hv, dv))
        for i in range(n):
            for h in range(Hv):
                hk = h // (Hv // Hk)
                Sp = inp["state"][b, h].astype(np.float64) if par[i] < 0 else states[b, par[i], h]
                kk = f(inp["k"][b, i, hk]).astype(np.float64)
                vv = f(inp["v"][b, i, h]).astype(np.float64)
                uref[i, h] = inp["beta"][b, i, h] * (vv - np.exp(np.float64(la[i, h])) * (Sp @ kk))
        assert_close(u[b, :n], uref, what=f"u[b={b}]")


def test_gdn_full_size_27b_layer(dflv, orc):
    # one gated-DeltaNet layer of a 27B-class hybrid target: 16 q/k heads,
    # 48 v heads, dk = dv = 128, a 22-node DDTree, state ~ N(0, 0.02)
    rng = np.random.default_rng(1235)
    par, _ = synth.ddtree(rng, 22, 151936)
    parent, n_nodes = synth.batch_trees([par], 22)
    inp = synth.gdn_inputs(rng, 1, 22, **synth.GDN_27B)
    out, _, _, _ = gpu_gdn(dflv, parent, n_nodes, inp, **synth.GDN_27B)
    ref = oracle_gdn(orc, parent, n_nodes, inp)
    e = compare_valid(out, ref, n_nodes, "o")
    print(f"full-size GDN max rel err {e:.2e}")


def test_gdn_wide_batch(dflv, orc):
    # batch of 8 sequences with 64-node trees (long-context stress shapes)
    rng = np.random.default_rng(1238)
    parents = [synth.ddtree(rng, 64, 151936)[0] for _ in range(8)]
    parent, n_nodes = synth.batch_trees(parents, 64)
    inp = synth.gdn_inputs(rng, 8, 64, **synth.GDN_27B)
    out, _, _, _ = gpu_gdn(dflv, parent, n_nodes, inp, **synth.GDN_27B)
    ref = oracle_gdn(orc, parent, n_nodes, inp)
    compare_valid(out, ref, n_nodes, "o")


def test_gdn_bad_topology_sets_status(dflv):
    rng = np.random.default_rng(5)
    inp = synth.gdn_inputs(rng, 2, 4, 1, 2, 16, 16)
    parent = np.array([[-1, 0, 2, 1], [0, 0, 1, 2]], np.int32)   # seq 0: parent[2] = 2; seq 1: root != -1
    n_nodes = np.array([4, 4], np.int32)
    gpu_gdn(dflv, parent, n_nodes, inp, 1, 2, 16, 16, expect_status=dflv.DFLV_DEV_TOPOLOGY)
    n_bad = np.array([0, 5], np.int32)
    gpu_gdn(dflv, synth.batch_trees([synth.chain_tree(4)] * 2, 4)[0], n_bad, inp, 1, 2, 16, 16,
            expect_status=dflv.DFLV_DEV_TOPOLOGY)
    # the same with the tree read before the dependency wait
    gpu_gdn(dflv, parent, n_nodes, inp, 1, 2, 16, 16, expect_status=dflv.DFLV_DEV_TOPOLOGY,
            flags=dflv.DFLV_FLAG_EARLY_PREFETCH)


def test_gdn_layers_back_to_back_with_early_prefetch(dflv, orc):
    # four layers launched back to back on one stream, every layer after the
    # first with the state and tree read before the dependency wait; each
    # layer's inputs are written by an elementwise kernel queued just before
    # it, so a kernel that read them before its dependency wait could still
    # see the zeros they held
    rng = np.random.default_rng(1240)
    par, _ = synth.ddtree(rng, 22, 151936)
    parent, n_nodes = synth.batch_trees([par], 22)
    dp, dn = dev(parent), dev(n_nodes)
    G = synth.GDN_27B
    st = zeros_status()
    layers = []
    for li in range(4):
        inp = synth.gdn_inputs(rng, 1, 22, **G)
        src = {k: dev(v) for k, v in inp.items()}
        dst = {k: torch.zeros_like(v) for k, v in src.items()}
        out = torch.full((1, 22, G["Hv"], G["dv"]), float("nan"), device="cuda")
        u = torch.empty_like(out)
        g = torch.empty((1, 22, G["Hv"]), device="cuda")
        kc = torch.empty((1, 22, G["Hk"], G["dk"]), dtype=torch.int16, device="cuda")
        layers.append((inp, src, dst, out, u, g, kc))
    for inp, src, dst, out, u, g, kc in layers:
        dst["state"].copy_(src["state"])   # the committed state: not produced inside the step
    torch.cuda.synchronize()
    for li, (inp, src, dst, out, u, g, kc) in enumerate(layers):
        for k in ("q", "k", "v", "beta", "log_alpha"):
            torch.mul(src[k], 1, out=dst[k])   # an elementwise kernel produces this layer's inputs
        flags = 0 if li == 0 else dflv.DFLV_FLAG_EARLY_PREFETCH
        dflv.check(dflv.dflv_tree_gdn_verify(dflv.gdn_desc(1, 22, G["Hk"], G["Hv"], G["dk"], G["dv"], flags), dp, dn,
                                             dst["q"], dst["k"], dst["v"], dst["beta"], dst["log_alpha"],
                                             dst["state"], out, dflv.gdn_factors(u, g, kc), st))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for inp, src, dst, out, u, g, kc in layers:
        ref = oracle_gdn(orc, parent, n_nodes, inp)
        compare_valid(host(out), ref, n_nodes, "o")


def test_gdn_state_is_read_only(dflv):
    rng = np.random.default_rng(6)
    par, _ = synth.ddtree(rng, 22, 1000)
    parent, n_nodes = synth.batch_trees([par], 22)
    inp = synth.gdn_inputs(rng, 1, 22, 2, 4, 128, 64)
    state = dev(inp["state"])
    before = state.clone()
    keep = {k: dev(v) for k, v in inp.items() if k != "state"}
    out = torch.empty((1, 22, 4, 64), device="cuda")
    u = torch.empty_like(out)
    g = torch.empty((1, 22, 4), device="cuda")
    kc = torch.empty((1, 22, 2, 128), dtype=torch.int16, device="cuda")
    st = zeros_status()
    dflv.check(dflv.dflv_tree_gdn_verify(dflv.gdn_desc(1, 22, 2, 4, 128, 64), dev(parent), dev(n_nodes),
                                         keep["q"], keep["k"], keep["v"], keep["beta"], keep["log_alpha"],
                                         state, out, dflv.gdn_factors(u, g, kc), st))
    torch.cuda.synchronize()
    assert torch.equal(state, before)
