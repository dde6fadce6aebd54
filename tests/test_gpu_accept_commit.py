"""GPU parity: greedy acceptance (bit-exact), commit/rollback (state within
tolerance, KV compaction bit-exact) and whole verify steps against the CPU
oracle."""
import numpy as np
import pytest
import torch

import synth
from gpu_util import assert_close, dev, host, zeros_status
from test_gpu_attn import gpu_attn
from test_gpu_gdn import gpu_gdn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dflv():
    import speculative_decoding_tree_layer_gb300 as pkg

    pkg.build()
    pkg.load()
    return pkg


def gpu_accept(dflv, logits, tokens, parent, n_nodes, expect_status=0):
    B, N, V = logits.shape
    keep = dict(logits=dev(logits), tokens=dev(tokens), parent=dev(parent), n_nodes=dev(n_nodes))
    path = torch.full((B, N), -1, dtype=torch.int32, device="cuda")
    plen = torch.zeros(B, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(B, dtype=torch.int32, device="cuda")
    best = torch.full((B, N), -1, dtype=torch.int32, device="cuda")
    st = zeros_status()
    dflv.check(dflv.dflv_accept_greedy(B, N, V, keep["logits"], keep["tokens"], keep["parent"], keep["n_nodes"],
                                       path, plen, nxt, best, st), "dflv_accept_greedy")
    torch.cuda.synchronize()
    assert int(st.item()) == expect_status
    return host(path), host(plen), host(nxt), host(best)


def _trees(rng, ns, V, kind="ddtree"):
    parents, toks = [], []
    for n in ns:
        if kind == "ddtree":
            p, t = synth.ddtree(rng, n, V)
        else:
            p = synth.uniform_tree(rng, n)
            t = rng.integers(0, V, n).astype(np.int32)
        parents.append(p)
        toks.append(t)
    N = max(ns)
    parent, n_nodes = synth.batch_trees(parents, N)
    tokens = np.zeros((len(ns), N), np.int32)
    for b, t in enumerate(toks):
        tokens[b, : len(t)] = t
    return parent, n_nodes, tokens, parents


ACCEPT = [
    ([22], 151936, "ddtree", True),
    ([22], 151936, "ddtree", False),
    ([64, 5, 22], 1001, "ddtree", True),          # vocab not a multiple of 4
    ([7, 7], 32, "uniform", True),                # tiny vocab: duplicate sibling tokens
    ([1], 50, "uniform", False),
]


@pytest.mark.parametrize("case", ACCEPT)
def test_accept_bit_exact(dflv, orc, case):
    ns, V, kind, plant = case
    rng = np.random.default_rng(V + sum(ns))
    parent, n_nodes, tokens, parents = _trees(rng, ns, V, kind)
    logits = synth.random_logits(rng, len(ns), parent.shape[1], V)
    if plant:
        for b, p in enumerate(parents):
            synth.plant_path(logits, tokens, synth.deepest_path(p), b)
    path, plen, nxt, best = gpu_accept(dflv, logits, tokens, parent, n_nodes)
    rp, rl, rn, rb = orc.accept_greedy(logits, tokens, parent, n_nodes)
    for b in range(len(ns)):
        assert plen[b] == rl[b]
        assert np.array_equal(path[b, : rl[b]], rp[b, : rl[b]])
        assert np.array_equal(best[b, : n_nodes[b]], rb[b, : n_nodes[b]])
        assert nxt[b] == rn[b]


def test_accept_ties(dflv, orc):
    V = 4096
    parent = np.array([[-1, 0, 0, 1, 2]], np.int32)
    tokens = np.array([[0, 7, 7, 9, 9]], np.int32)      # two children with the same token
    logits = np.zeros((1, 5, V), np.float32)
    logits[0, :, [7, 2000, 4000]] = 3.0                 # three-way tie in every row -> 7
    logits[0, 1, 9] = 5.0
    path, plen, nxt, best = gpu_accept(dflv, logits, tokens, parent, np.array([5], np.int32))
    rp, rl, rn, rb = orc.accept_greedy(logits, tokens, parent, np.array([5], np.int32))
    assert plen[0] == rl[0] == 3 and list(path[0, :3]) == list(rp[0, :3]) == [0, 1, 3]
    assert np.array_equal(best, rb) and nxt[0] == rn[0] == 7


def test_accept_ties_across_ctas(dflv, orc):
    """Equal maxima in different CTAs' shares of one row: the lowest index
    wins wherever the split falls (a 22-node tree over 151,936 splits every
    row 16 ways, 9,496 entries each); plus a row whose only maximum is the
    last vocabulary entry."""
    V, N = 151936, 22
    rng = np.random.default_rng(17)
    parent = np.array([[-1] + list(range(N - 1))], np.int32)
    tokens = np.zeros((1, N), np.int32)
    logits = synth.random_logits(rng, 1, N, V)
    top = float(logits.max()) + 1.0
    logits[0, 0, [9495, 9496, V - 1]] = top
    logits[0, 1, [9496 * 5, 9496 * 5 - 1, 9496 * 11]] = top
    logits[0, 2, [V - 1]] = top
    logits[0, 3, [0, V - 1]] = top
    logits[0, 4, [9496 * 15, V - 4]] = top
    path, plen, nxt, best = gpu_accept(dflv, logits, tokens, parent, np.array([N], np.int32))
    rp, rl, rn, rb = orc.accept_greedy(logits, tokens, parent, np.array([N], np.int32))
    assert list(rb[0, :5]) == [9495, 9496 * 5 - 1, V - 1, 0, 9496 * 15]
    assert np.array_equal(best, rb) and plen[0] == rl[0] and nxt[0] == rn[0]


def test_accept_batch8_n64(dflv, orc):
    """Eight 64-node trees over the full vocabulary: one CTA per row, several
    load batches per thread; paths planted in every sequence."""
    V, B = 151936, 8
    rng = np.random.default_rng(64)
    parent, n_nodes, tokens, parents = _trees(rng, [64, 64, 63, 64, 40, 64, 64, 1], V)
    logits = synth.random_logits(rng, B, parent.shape[1], V)
    for b, p in enumerate(parents):
        synth.plant_path(logits, tokens, synth.deepest_path(p), b)
    path, plen, nxt, best = gpu_accept(dflv, logits, tokens, parent, n_nodes)
    rp, rl, rn, rb = orc.accept_greedy(logits, tokens, parent, n_nodes)
    for b in range(B):
        assert plen[b] == rl[b] and nxt[b] == rn[b]
        assert np.array_equal(path[b, : rl[b]], rp[b, : rl[b]])
        assert np.array_equal(best[b, : n_nodes[b]], rb[b, : n_nodes[b]])


def test_accept_bad_topology_sets_status(dflv):
    """A parent that does not precede its child, and a node count past N_max,
    raise the topology bit; those sequences get path_len 0, the valid one is
    walked."""
    V, N = 4096, 6
    rng = np.random.default_rng(5)
    parent = np.array([[-1, 0, 0, 1, 2, 3], [-1, 0, 3, 1, 2, 3], [-1, 0, 1, 2, 3, 4]], np.int32)
    n_nodes = np.array([6, 6, 7], np.int32)
    tokens = np.zeros((3, N), np.int32)
    logits = synth.random_logits(rng, 3, N, V)
    path, plen, nxt, best = gpu_accept(dflv, logits, tokens, parent, n_nodes, expect_status=dflv.DFLV_DEV_TOPOLOGY)
    assert plen[0] >= 1 and plen[1] == 0 and plen[2] == 0


def test_accept_nan_logits(dflv, orc):
    """A NaN logit counts as -inf on both sides: rows with NaN before, after
    and instead of the maximum, an all-NaN row and a NaN/-inf row, at a
    vocabulary that several CTAs of a row split."""
    V = 151936
    rng = np.random.default_rng(91)
    parent = np.array([[-1, 0, 1, 2, 3, 4]], np.int32)
    logits = synth.random_logits(rng, 1, 6, V)
    logits[0, 0, rng.integers(0, V, 500)] = np.nan
    logits[0, 0, 0] = np.nan
    logits[0, 1] = np.nan
    logits[0, 2] = -np.inf
    logits[0, 2, ::3] = np.nan
    logits[0, 3, : V // 2] = np.nan
    logits[0, 4, V // 2:] = np.nan
    tokens = np.zeros((1, 6), np.int32)
    path, plen, nxt, best = gpu_accept(dflv, logits, tokens, parent, np.array([6], np.int32))
    rp, rl, rn, rb = orc.accept_greedy(logits, tokens, parent, np.array([6], np.int32))
    assert np.array_equal(best, rb) and plen[0] == rl[0] and nxt[0] == rn[0]
    assert np.array_equal(path[0, : rl[0]], rp[0, : rl[0]])
    assert rb[0, 1] == 0 and rb[0, 2] == 0


def gpu_commit(dflv, gdn_layers, attn_layers, path, path_len, n_past, dims, expect_status=0):
    """gdn_layers: list of dicts with device tensors state/u/g/kc; attn_layers:
    list of dicts with device planes."""
    B, N = path.shape
    st = zeros_status()
    keep = dict(path=dev(path), plen=dev(path_len), n_past=dev(n_past))
    gd = dflv.gdn_desc(B, N, *dims["gdn"]) if gdn_layers else None
    ad = dflv.attn_desc(B, N, *dims["attn"]) if attn_layers else None
    rc = dflv.dflv_commit_rollback(
        gd, len(gdn_layers), [l["state"] for l in gdn_layers],
        [dflv.gdn_factors(l["u"], l["g"], l["kc"]) for l in gdn_layers], ad, len(attn_layers),
        [dflv.kv_layer(l["kq"], l["vq"], l.get("ks"), l.get("vs")) for l in attn_layers],
        keep["path"], keep["plen"], keep["n_past"], st)
    dflv.check(rc, "dflv_commit_rollback")
    torch.cuda.synchronize()
    assert int(st.item()) == expect_status
    return host(keep["n_past"])


@pytest.mark.parametrize("kv_type", [synth.KV_Q8_0, synth.KV_Q4_0, synth.KV_F32, synth.KV_Q8_0_Q4_0,
                                     synth.KV_Q4_0_Q8_0, synth.KV_TQ3_0])
def test_commit_gdn_and_kv(dflv, orc, kv_type):
    rng = np.random.default_rng(40 + kv_type)
    Hk, Hv, dk, dv = 2, 6, 128, 64
    Hq, Hkv, D = 4, 2, {synth.KV_F32: 16, synth.KV_Q8_0_Q4_0: 128, synth.KV_Q4_0_Q8_0: 128,
                        synth.KV_TQ3_0: 128}.get(kv_type, 64)
    B, N = 3, 9
    parents = [np.array([-1, 0, 0, 2, 3, 1, 4, 6, 6], np.int32),  # accepted path 0, 2, 3 aliases
               synth.chain_tree(9), np.array([-1, 0, 1, 1], np.int32)]
    parent, n_nodes = synth.batch_trees(parents, N)
    path = np.full((B, N), -1, np.int32)
    path[0, :5] = [0, 2, 3, 4, 6]
    path[1, :9] = np.arange(9)
    path[2, :1] = [0]
    path_len = np.array([5, 9, 1], np.int32)
    # GDN: verify on the GPU (factors), commit on the GPU; oracle decodes the path
    ginp = synth.gdn_inputs(rng, B, N, Hk, Hv, dk, dv, state_std=0.3)
    keep = {k: dev(v) for k, v in ginp.items()}
    u = torch.empty((B, N, Hv, dv), device="cuda")
    g = torch.empty((B, N, Hv), device="cuda")
    kc = torch.empty((B, N, Hk, dk), dtype=torch.int16, device="cuda")
    out = torch.empty((B, N, Hv, dv), device="cuda")
    st = zeros_status()
    dflv.check(dflv.dflv_tree_gdn_verify(dflv.gdn_desc(B, N, Hk, Hv, dk, dv), dev(parent), dev(n_nodes), keep["q"],
                                         keep["k"], keep["v"], keep["beta"], keep["log_alpha"], keep["state"], out,
                                         dflv.gdn_factors(u, g, kc), st))
    # KV: a cache the tree has been written into
    P = np.array([40, 17, 3], np.int32)
    cap = 64
    cache = synth.kv_cache(rng, B, Hkv, cap, D, kv_type)
    dc = {k: (None if v is None else dev(v)) for k, v in cache.items()}
    before = {k: (None if v is None else v.copy()) for k, v in cache.items()}
    new_P = gpu_commit(dflv, [dict(state=keep["state"], u=u, g=g, kc=kc)],
                       [dict(kq=dc["kq"], vq=dc["vq"], ks=dc["ks"], vs=dc["vs"])], path, path_len, P,
                       dict(gdn=(Hk, Hv, dk, dv), attn=(Hq, Hkv, D, cap, 0, kv_type, 0.125)))
    assert np.array_equal(new_P, P + path_len)
    ref_state = orc.gdn_commit(ginp["q"], ginp["k"], ginp["v"], ginp["beta"], ginp["log_alpha"], path, path_len,
                               ginp["state"])
    assert_close(host(keep["state"]), ref_state, what="committed state")
    orc.kv_commit(before, kv_type, path, path_len, P)
    for key in ("kq", "vq", "ks", "vs"):
        if before[key] is None:
            continue
        got = host(dc[key], before[key].dtype)
        for b in range(B):
            # slots below P + L are fully specified; [P + L, P + N) are not
            hi = P[b] + path_len[b]
            assert np.array_equal(got[b, :, :hi], before[key][b, :, :hi]), key
            assert np.array_equal(got[b, :, P[b] + N:], before[key][b, :, P[b] + N:]), key


def test_commit_bad_path_sets_status(dflv):
    rng = np.random.default_rng(3)
    B, N, Hkv, D, cap = 1, 4, 1, 64, 16
    cache = synth.kv_cache(rng, B, Hkv, cap, D, synth.KV_Q8_0)
    dc = {k: dev(v) for k, v in cache.items()}
    path = np.array([[0, 1, 2, 3]], np.int32)
    new_P = gpu_commit(dflv, [], [dict(kq=dc["kq"], vq=dc["vq"], ks=dc["ks"], vs=dc["vs"])], path,
                       np.array([0], np.int32), np.array([2], np.int32),
                       dict(attn=(2, Hkv, D, cap, 0, synth.KV_Q8_0, 0.125)), expect_status=dflv.DFLV_DEV_PATH)
    assert new_P[0] == 2


def test_tiny_case_full_step_twice(dflv, orc):
    """The tiny end-to-end case, all on the GPU: an 8-token prefix decoded as a
    chain from zero state and committed, then two tree verify -> accept ->
    commit steps (7-node trees, parent[i] ~ U[0, i)), against the oracle."""
    rng = np.random.default_rng(1234)
    Hk = Hv = 2
    dk = dv = 16
    Hq = Hkv = 1
    D, V, P0, cap = 16, 32, 64, 128
    gdims = (Hk, Hv, dk, dv)
    adims = (Hq, Hkv, D, cap, 0, synth.KV_F32, 0.25)
    # ---- prefix: 8-token chain from the zero state
    pre = synth.gdn_inputs(rng, 1, 8, Hk, Hv, dk, dv)
    pre["state"] = np.zeros((1, Hv, dv, dk), np.float32)
    cpar, cn = synth.batch_trees([synth.chain_tree(8)], 8)
    _, u, g, kc = gpu_gdn(dflv, cpar, cn, pre, Hk, Hv, dk, dv)
    state = dev(pre["state"])
    fac = dict(state=state, u=dev(u), g=dev(g), kc=dev(kc.view(np.uint16)))
    full = np.arange(8, dtype=np.int32)[None]
    gpu_commit(dflv, [fac], [], full, np.array([8], np.int32), np.array([0], np.int32), dict(gdn=gdims))
    ref_state = orc.gdn_commit(pre["q"], pre["k"], pre["v"], pre["beta"], pre["log_alpha"], full,
                               np.array([8], np.int32), pre["state"])
    assert_close(host(state), ref_state, what="prefix state")
    cache = synth.kv_cache(rng, 1, Hkv, cap, D, synth.KV_F32)
    ref_cache = synth.copy_cache(cache)
    dcache = {k: (None if v is None else dev(v)) for k, v in cache.items()}
    n_past = dev(np.array([P0], np.int32))
    ref_P = P0
    gstate_ref = ref_state
    for step in range(2):
        par = synth.uniform_tree(rng, 7)
        parent, n_nodes = synth.batch_trees([par], 7)
        tokens = rng.integers(0, V, (1, 7)).astype(np.int32)
        gi = synth.gdn_inputs(rng, 1, 7, Hk, Hv, dk, dv, state=False)
        ai = synth.attn_inputs(rng, 1, 7, Hq, Hkv, D)
        logits = synth.random_logits(rng, 1, 7, V)
        synth.plant_path(logits, tokens, synth.deepest_path(par))
        # GPU step
        gk = {k: dev(v) for k, v in gi.items()}
        ak = {k: dev(v) for k, v in ai.items()}
        kp, kn = dev(parent), dev(n_nodes)
        go = torch.empty((1, 7, Hv, dv), device="cuda")
        u = torch.empty_like(go)
        g = torch.empty((1, 7, Hv), device="cuda")
        kc = torch.empty((1, 7, Hk, dk), dtype=torch.int16, device="cuda")
        ao = torch.empty((1, 7, Hq, D), device="cuda")
        st = zeros_status()
        dflv.check(dflv.dflv_tree_gdn_verify(dflv.gdn_desc(1, 7, *gdims), kp, kn, gk["q"], gk["k"], gk["v"],
                                             gk["beta"], gk["log_alpha"], state, go, dflv.gdn_factors(u, g, kc), st))
        dflv.check(dflv.dflv_tree_attn_verify(dflv.attn_desc(1, 7, *adims), kp, kn, n_past, ak["q"], ak["k_new"],
                                              ak["v_new"], dflv.kv_layer(dcache["kq"], dcache["vq"]), ao, st))
        lg, tk = dev(logits), dev(tokens)
        path = torch.empty((1, 7), dtype=torch.int32, device="cuda")
        plen = torch.empty(1, dtype=torch.int32, device="cuda")
        nxt = torch.empty(1, dtype=torch.int32, device="cuda")
        best = torch.empty((1, 7), dtype=torch.int32, device="cuda")
        dflv.check(dflv.dflv_accept_greedy(1, 7, V, lg, tk, kp, kn, path, plen, nxt, best, st))
        dflv.check(dflv.dflv_commit_rollback(dflv.gdn_desc(1, 7, *gdims), 1, [state], [dflv.gdn_factors(u, g, kc)],
                                             dflv.attn_desc(1, 7, *adims), 1,
                                             [dflv.kv_layer(dcache["kq"], dcache["vq"])], path, plen, n_past, st))
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        # oracle step
        gi_ref = dict(gi, state=gstate_ref)
        ref_go = orc.tree_gdn_verify(parent, n_nodes, gi["q"], gi["k"], gi["v"], gi["beta"], gi["log_alpha"],
                                     gstate_ref)
        ref_ao = orc.tree_attn_verify(parent, n_nodes, np.array([ref_P], np.int32), ai["q"], ai["k_new"],
                                      ai["v_new"], ref_cache, 0, synth.KV_F32)
        rp, rl, rn, _ = orc.accept_greedy(logits, tokens, parent, n_nodes)
        gstate_ref = orc.gdn_commit(gi["q"], gi["k"], gi["v"], gi["beta"], gi["log_alpha"], rp, rl, gstate_ref)
        orc.kv_commit(ref_cache, synth.KV_F32, rp, rl, np.array([ref_P], np.int32))
        ref_P += int(rl[0])
        assert_close(host(go), ref_go, what=f"step {step} gdn out")
        assert_close(host(ao), ref_ao, what=f"step {step} attn out")
        L = int(host(plen)[0])
        assert L == rl[0] and np.array_equal(host(path)[0, :L], rp[0, :L]) and int(host(nxt)[0]) == rn[0]
        assert int(host(n_past)[0]) == ref_P
        assert_close(host(state), gstate_ref, what=f"step {step} state")
        hc = host(dcache["kq"])
        assert np.array_equal(hc[:, :, :ref_P], ref_cache["kq"][:, :, :ref_P])


@pytest.mark.parametrize("N", [22, 48])
def test_deferred_commit_matches_eager(dflv, orc, N):
    """Deferred commit: each verify applies the previous step's accepted path
    to the state it streams (and writes it back), so a step commits only the
    KV caches.  Three steps on two sequences (one with an empty pending
    path), outputs and states against the oracle's eager commit; trees of up
    to 32 nodes and over 32 take different launch forms."""
    rng = np.random.default_rng(77 + N)
    Hk, Hv, dk, dv, B = 2, 6, 128, 64, 2
    state0 = (rng.standard_normal((B, Hv, dv, dk)) * 0.3).astype(np.float32)
    state = dev(state0)
    ref_state = state0.copy()
    fac = [dict(u=torch.empty((B, N, Hv, dv), device="cuda"), g=torch.empty((B, N, Hv), device="cuda"),
                kc=torch.empty((B, N, Hk, dk), dtype=torch.int16, device="cuda")) for _ in range(2)]
    prev = None
    for step in range(3):
        parents = [synth.ddtree(rng, N, 1000)[0] for _ in range(B)]
        parent, n_nodes = synth.batch_trees(parents, N)
        gi = synth.gdn_inputs(rng, B, N, Hk, Hv, dk, dv, state=False)
        keep = {k: dev(v) for k, v in gi.items()}
        out = torch.full((B, N, Hv, dv), float("nan"), device="cuda")
        f = fac[step % 2]
        st = zeros_status()
        args = (dflv.gdn_desc(B, N, Hk, Hv, dk, dv), dev(parent), dev(n_nodes), keep["q"], keep["k"], keep["v"],
                keep["beta"], keep["log_alpha"], state)
        if prev is None:
            dflv.check(dflv.dflv_tree_gdn_verify(*args, out, dflv.gdn_factors(f["u"], f["g"], f["kc"]), st))
        else:
            pf, ppath, plen = prev
            dflv.check(dflv.dflv_tree_gdn_verify_pending(*args, dflv.gdn_factors(pf["u"], pf["g"], pf["kc"]),
                                                         dev(ppath), dev(plen), out,
                                                         dflv.gdn_factors(f["u"], f["g"], f["kc"]), st))
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        ref_out = orc.tree_gdn_verify(parent, n_nodes, gi["q"], gi["k"], gi["v"], gi["beta"], gi["log_alpha"],
                                      ref_state)
        for b in range(B):
            assert_close(host(out)[b], ref_out[b], what=f"step {step} out b={b}")
        if prev is not None:
            assert_close(host(state), ref_state, what=f"state written by step {step}")
        # this step's accepted paths: a prefix of the deepest path (empty for b = 1 at step 1)
        path = np.full((B, N), -1, np.int32)
        plen = np.zeros(B, np.int32)
        for b in range(B):
            dp = synth.deepest_path(parents[b])
            L = 0 if (b == 1 and step == 1) else int(rng.integers(1, len(dp) + 1))
            path[b, :L] = dp[:L]
            plen[b] = L
        ref_state = np.stack([
            orc.gdn_commit(gi["q"][b:b + 1], gi["k"][b:b + 1], gi["v"][b:b + 1], gi["beta"][b:b + 1],
                           gi["log_alpha"][b:b + 1], path[b:b + 1], plen[b:b + 1], ref_state[b:b + 1])[0]
            if plen[b] > 0 else ref_state[b] for b in range(B)])
        prev = (f, path, plen)


def test_deferred_commit_bad_path_sets_status(dflv):
    rng = np.random.default_rng(78)
    Hk, Hv, dk, dv, B, N = 1, 2, 64, 32, 1, 6
    par = synth.uniform_tree(rng, N)
    parent, n_nodes = synth.batch_trees([par], N)
    gi = synth.gdn_inputs(rng, B, N, Hk, Hv, dk, dv)
    keep = {k: dev(v) for k, v in gi.items()}
    fa = [dict(u=torch.zeros((B, N, Hv, dv), device="cuda"), g=torch.zeros((B, N, Hv), device="cuda"),
               kc=torch.zeros((B, N, Hk, dk), dtype=torch.int16, device="cuda")) for _ in range(2)]
    out = torch.empty((B, N, Hv, dv), device="cuda")
    before = keep["state"].clone()
    st = zeros_status()
    dflv.check(dflv.dflv_tree_gdn_verify_pending(
        dflv.gdn_desc(B, N, Hk, Hv, dk, dv), dev(parent), dev(n_nodes), keep["q"], keep["k"], keep["v"],
        keep["beta"], keep["log_alpha"], keep["state"], dflv.gdn_factors(fa[0]["u"], fa[0]["g"], fa[0]["kc"]),
        dev(np.arange(N, dtype=np.int32)[None]), dev(np.array([N + 1], np.int32)), out,
        dflv.gdn_factors(fa[1]["u"], fa[1]["g"], fa[1]["kc"]), st))
    torch.cuda.synchronize()
    assert int(st.item()) == dflv.DFLV_DEV_PATH
    assert torch.equal(keep["state"], before)
