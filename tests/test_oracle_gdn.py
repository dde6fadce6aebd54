"""Pins for the oracle's gated delta-rule tree verify (CPU only).

The pages name the op (Luce DFlash README, "Architecture note":
ggml_gated_delta_net and its _tree variant) and the tree rule (README "How it
works": one forward verifies the whole tree through a mask derived from the
parent pointers); the recurrence is the standard gated delta rule
S' = alpha S (I - beta k k^T) + beta v k^T, o = S' q.  Each test below would
fail for a plausible slip in the oracle: a dropped term, a sign, a transposed
operand, the pre-update state in the output, or a wrong parent in the tree.
"""
import numpy as np
import pytest

import synth

pytestmark = []


def _rand_state(rng, dv, dk):
    return rng.standard_normal((dv, dk))


def _unit(rng, d):
    x = rng.standard_normal(d)
    return x / np.linalg.norm(x)


# ---------------------------------------------------------------- one step
def test_step_beta_zero_is_pure_decay(orc):
    rng = np.random.default_rng(1)
    dv, dk = 6, 5
    S = _rand_state(rng, dv, dk)
    q, k, v = rng.standard_normal(dk), rng.standard_normal(dk), rng.standard_normal(dv)
    S1, o = orc.gdn_step(S, q, k, v, beta=0.0, alpha=0.37)
    np.testing.assert_allclose(S1, 0.37 * S, rtol=0, atol=1e-15)
    np.testing.assert_allclose(o, (0.37 * S) @ q, rtol=1e-13, atol=1e-13)


def test_step_delta_rule_overwrites_along_k(orc):
    # alpha = 1, beta = 1, |k| = 1: the new state maps k exactly onto v.
    rng = np.random.default_rng(2)
    dv, dk = 7, 9
    S = _rand_state(rng, dv, dk)
    k = _unit(rng, dk)
    v = rng.standard_normal(dv)
    S1, _ = orc.gdn_step(S, rng.standard_normal(dk), k, v, beta=1.0, alpha=1.0)
    np.testing.assert_allclose(S1 @ k, v, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", [3, 4, 5])
def test_step_action_on_k_and_its_complement(orc, seed):
    # For any x orthogonal to k: S' x = alpha S x.  Along k:
    # S' k = alpha (1 - beta |k|^2) S k + beta |k|^2 v.  Together these fix
    # S' on every vector, so they determine the step completely; S is not
    # symmetric, so a transposed S or k k^T on the wrong side fails here.
    rng = np.random.default_rng(seed)
    dv, dk = 5, 8
    S = _rand_state(rng, dv, dk)
    k = rng.standard_normal(dk) * 0.7
    v = rng.standard_normal(dv)
    alpha, beta = 0.81, 0.43
    S1, _ = orc.gdn_step(S, rng.standard_normal(dk), k, v, beta=beta, alpha=alpha)
    kk = k @ k
    np.testing.assert_allclose(S1 @ k, alpha * (1 - beta * kk) * (S @ k) + beta * kk * v,
                               rtol=1e-12, atol=1e-12)
    for _ in range(4):
        x = rng.standard_normal(dk)
        x -= (x @ k) / kk * k
        np.testing.assert_allclose(S1 @ x, alpha * (S @ x), rtol=1e-11, atol=1e-12)


def test_step_output_reads_updated_state(orc):
    # S = 0: the only content is the write, so o = beta (k . q) v (the
    # pre-update state would give 0).
    rng = np.random.default_rng(6)
    dv, dk = 4, 6
    q, k, v = rng.standard_normal(dk), rng.standard_normal(dk), rng.standard_normal(dv)
    _, o = orc.gdn_step(np.zeros((dv, dk)), q, k, v, beta=0.6, alpha=0.9)
    np.testing.assert_allclose(o, 0.6 * (k @ q) * v, rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- tree verify
def _gdn_case(rng, B, N, Hk, Hv, dk, dv, parents):
    inp = synth.gdn_inputs(rng, B, N, Hk, Hv, dk, dv, state_std=0.5)
    parent, n_nodes = synth.batch_trees(parents, N)
    return parent, n_nodes, inp


def _verify(orc, parent, n_nodes, inp, **kw):
    return orc.tree_gdn_verify(parent, n_nodes, inp["q"], inp["k"], inp["v"], inp["beta"],
                               inp["log_alpha"], inp["state"], **kw)


@pytest.mark.parametrize("n", [1, 2, 7, 13])
def test_tree_equals_per_path_bruteforce(orc, n):
    rng = np.random.default_rng(10 + n)
    parents = [synth.uniform_tree(rng, n), synth.uniform_tree(rng, max(1, n - 1))]
    parent, n_nodes, inp = _gdn_case(rng, 2, n, 2, 4, 8, 6, parents)
    a = _verify(orc, parent, n_nodes, inp)
    b = orc.tree_gdn_verify_bruteforce(parent, n_nodes, inp["q"], inp["k"], inp["v"], inp["beta"],
                                       inp["log_alpha"], inp["state"])
    for bb in range(2):
        m = n_nodes[bb]
        assert np.array_equal(a[bb, :m], b[bb, :m])  # same operations, same order: bitwise


def test_chain_tree_equals_sequential_decode(orc):
    # A chain is a degenerate tree (SpecLA PR, "Paper mapping"); verifying it
    # must equal decoding its tokens one step at a time.
    rng = np.random.default_rng(20)
    n, Hk, Hv, dk, dv = 6, 1, 2, 8, 5
    parent, n_nodes, inp = _gdn_case(rng, 1, n, Hk, Hv, dk, dv, [synth.chain_tree(n)])
    out = _verify(orc, parent, n_nodes, inp)
    f = synth.bf16_to_f32
    for h in range(Hv):
        S = inp["state"][0, h].astype(np.float64)
        for i in range(n):
            S, o = orc.gdn_step(S, f(inp["q"][0, i, 0]), f(inp["k"][0, i, 0]), f(inp["v"][0, i, h]),
                                inp["beta"][0, i, h], np.exp(np.float64(inp["log_alpha"][0, i, h])))
            np.testing.assert_array_equal(out[0, i, h], o.astype(np.float32))


def test_single_node_is_one_decode_step(orc):
    rng = np.random.default_rng(21)
    parent, n_nodes, inp = _gdn_case(rng, 1, 1, 2, 2, 8, 8, [synth.chain_tree(1)])
    out = _verify(orc, parent, n_nodes, inp)
    f = synth.bf16_to_f32
    for h in range(2):
        _, o = orc.gdn_step(inp["state"][0, h].astype(np.float64), f(inp["q"][0, 0, h]),
                            f(inp["k"][0, 0, h]), f(inp["v"][0, 0, h]), inp["beta"][0, 0, h],
                            np.exp(np.float64(inp["log_alpha"][0, 0, h])))
        np.testing.assert_array_equal(out[0, 0, h], o.astype(np.float32))


def test_relabelling_siblings_permutes_outputs(orc):
    # Any topological relabelling describes the same tree; outputs follow the
    # nodes.  Tree: 0 -> {1, 2}, 1 -> 3, 2 -> 4; swap the two subtrees.
    rng = np.random.default_rng(22)
    par_a = np.array([-1, 0, 0, 1, 2], np.int32)
    perm = np.array([0, 2, 1, 4, 3])          # new index j holds old node perm[j]
    inv = np.argsort(perm)
    par_b = np.array([-1 if par_a[perm[j]] < 0 else inv[par_a[perm[j]]] for j in range(5)], np.int32)
    parent, n_nodes, inp = _gdn_case(rng, 1, 5, 2, 4, 8, 4, [par_a])
    out_a = _verify(orc, parent, n_nodes, inp)
    inp_b = dict(inp)
    for key in ("q", "k", "v", "beta", "log_alpha"):
        inp_b[key] = inp[key][:, perm].copy()
    out_b = _verify(orc, par_b[None], n_nodes, inp_b)
    np.testing.assert_array_equal(out_b[0], out_a[0, perm])


def test_wy_form_agrees_with_sequential_oracle(orc):
    # An independent algorithm: the WY/UT representation never builds a
    # node's state.  With u_i = beta_i (v_i - alpha_i S_parent k_i) and
    # g_i = sum of log alpha over i's ancestors-or-self,
    #   S_i = e^{g_i} S_0 + sum_{l in anc*(i)} e^{g_i - g_l} u_l k_l^T,
    #   o_i = e^{g_i} S_0 q_i + sum_{l in anc*(i)} e^{g_i - g_l} (k_l . q_i) u_l.
    rng = np.random.default_rng(23)
    n, Hk, Hv, dk, dv = 17, 2, 6, 16, 12
    parents = [synth.uniform_tree(rng, n)]
    parent, n_nodes, inp = _gdn_case(rng, 1, n, Hk, Hv, dk, dv, parents)
    out = _verify(orc, parent, n_nodes, inp)
    par = parent[0]
    anc = []
    for i in range(n):
        a, c = [], i
        while c >= 0:
            a.append(c)
            c = par[c]
        anc.append(sorted(a))
    f = synth.bf16_to_f32
    for h in range(Hv):
        hk = h // (Hv // Hk)
        S0 = inp["state"][0, h].astype(np.float64)
        K = f(inp["k"][0, :, hk]).astype(np.float64)
        Q = f(inp["q"][0, :, hk]).astype(np.float64)
        V = f(inp["v"][0, :, h]).astype(np.float64)
        be = inp["beta"][0, :, h].astype(np.float64)
        la = inp["log_alpha"][0, :, h].astype(np.float64)
        g = np.array([la[a].sum() for a in anc])
        U = np.zeros((n, dv))
        for i in range(n):
            p = par[i]
            if p < 0:
                Sk = S0 @ K[i]
                gp = 0.0
            else:
                gp = g[p]
                Sk = np.exp(gp) * (S0 @ K[i]) + sum(np.exp(gp - g[l]) * (K[l] @ K[i]) * U[l] for l in anc[p])
            U[i] = be[i] * (V[i] - np.exp(la[i]) * Sk)
        for i in range(n):
            o = np.exp(g[i]) * (S0 @ Q[i]) + sum(np.exp(g[i] - g[l]) * (K[l] @ Q[i]) * U[l] for l in anc[i])
            np.testing.assert_allclose(out[0, i, h], o, rtol=2e-6, atol=1e-6)


def test_topology_errors_are_reported(orc):
    rng = np.random.default_rng(24)
    for bad in ([0, 0, 1], [-1, 1, 0], [-1, 0, 3], [-1, -1, 0]):
        parent, n_nodes, inp = _gdn_case(rng, 1, 3, 1, 1, 4, 4, [np.array(bad, np.int32)])
        with pytest.raises(orc.OracleError) as e:
            _verify(orc, parent, n_nodes, inp)
        assert e.value.code == orc.ERR_TOPOLOGY


def test_commit_equals_decoding_the_accepted_tokens(orc):
    # Commit leaves the state of decoding only the accepted path ("How it
    # works", per-step rollback): bit-identical to the fp32 state of a chain
    # verify over exactly those tokens.
    rng = np.random.default_rng(25)
    n, Hk, Hv, dk, dv = 9, 2, 4, 8, 8
    par = np.array([-1, 0, 0, 1, 1, 3, 2, 5, 5], np.int32)
    parent, n_nodes, inp = _gdn_case(rng, 1, n, Hk, Hv, dk, dv, [par])
    path = np.full((1, n), -1, np.int32)
    acc = [0, 1, 3, 5, 8]
    path[0, :5] = acc
    committed = orc.gdn_commit(inp["q"], inp["k"], inp["v"], inp["beta"], inp["log_alpha"], path,
                               np.array([5], np.int32), inp["state"])
    # chain over the accepted tokens only
    chain_inp = {k: inp[k][:, acc].copy() for k in ("q", "k", "v", "beta", "log_alpha")}
    chain_inp["state"] = inp["state"]
    cpar, cn = synth.batch_trees([synth.chain_tree(5)], 5)
    _, states = _verify(orc, cpar, cn, chain_inp, want_states=True)
    assert np.array_equal(committed, states[:, 4].astype(np.float32))
    # and equal to the end node's state inside the full tree verify
    _, tree_states = _verify(orc, parent, n_nodes, inp, want_states=True)
    assert np.array_equal(committed, tree_states[:, 8].astype(np.float32))
