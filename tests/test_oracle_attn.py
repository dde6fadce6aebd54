"""Pins for the oracle's attention tree verify (CPU only).

Tree queries attend to the cached prefix and to their own ancestors-or-self
(Luce DFlash README, "How it works": a causal mask derived from parent
pointers), optionally inside a sliding window ("--fa-window N", 0 = full),
over a q8_0 / q4_0 KV cache ("Asymmetric K/V quantization").  The tree's own
keys and values are written into cache slots P.. first and attended in their
quantised form, as a sequential decode would read them.
"""
import numpy as np
import pytest
import torch

import synth

TYPES = [synth.KV_Q8_0, synth.KV_Q4_0, synth.KV_F32]
# keys and values in different formats ("Asymmetric K/V quantization")
ASYM = [synth.KV_Q8_0_Q4_0, synth.KV_Q4_0_Q8_0]


def _plane_type(kv_type, which):
    if kv_type == synth.KV_Q8_0_Q4_0:
        return synth.KV_Q4_0 if which else synth.KV_Q8_0
    if kv_type == synth.KV_Q4_0_Q8_0:
        return synth.KV_Q8_0 if which else synth.KV_Q4_0
    return kv_type


def _case(rng, kv_type, parents, P, cap, Hq=4, Hkv=2, D=64):
    N = max(len(p) for p in parents)
    B = len(parents)
    parent, n_nodes = synth.batch_trees(parents, N)
    inp = synth.attn_inputs(rng, B, N, Hq, Hkv, D)
    cache = synth.kv_cache(rng, B, Hkv, cap, D, kv_type, scale_std=0.05)
    n_past = np.full(B, P, np.int32)
    return parent, n_nodes, n_past, inp, cache


def _run(orc, parent, n_nodes, n_past, inp, cache, window, kv_type):
    c = synth.copy_cache(cache)
    out = orc.tree_attn_verify(parent, n_nodes, n_past, inp["q"], inp["k_new"], inp["v_new"], c,
                               window, kv_type)
    return out, c


def _dequant_rows(cache, which, kv_type, b, h, D):
    """numpy dequantisation of every slot of one (sequence, kv head)."""
    q = cache["kq" if which == 0 else "vq"][b, h]
    kv_type = _plane_type(kv_type, which)
    if kv_type == synth.KV_F32:
        return q.astype(np.float64)
    s = cache["ks" if which == 0 else "vs"][b, h].view(np.float16).astype(np.float64)
    if kv_type == synth.KV_Q8_0:
        codes = q.astype(np.float64).reshape(q.shape[0], D // 32, 32)
    else:
        lo = (q & 0x0F).astype(np.float64) - 8
        hi = (q >> 4).astype(np.float64) - 8
        codes = np.concatenate([lo.reshape(q.shape[0], D // 32, 16), hi.reshape(q.shape[0], D // 32, 16)], axis=2)
    return (codes * s[:, :, None]).reshape(q.shape[0], D)


def _ancestors(par, i):
    a = []
    while i >= 0:
        a.append(i)
        i = par[i]
    return set(a)


@pytest.mark.parametrize("kv_type", TYPES + ASYM)
@pytest.mark.parametrize("window", [0, 5, 13])
def test_matches_torch_sdpa_with_explicit_mask(orc, kv_type, window):
    # Library cross-check: fp64 scaled_dot_product_attention over the
    # dequantised cache with a boolean mask built from the parent pointers.
    rng = np.random.default_rng(100 + kv_type * 10 + window)
    par = synth.uniform_tree(rng, 9)
    P, cap, Hq, Hkv, D = 21, 40, 4, 2, 64
    parent, n_nodes, n_past, inp, cache = _case(rng, kv_type, [par], P, cap, Hq, Hkv, D)
    out, c = _run(orc, parent, n_nodes, n_past, inp, cache, window, kv_type)
    depth = synth.tree_depths(par)
    n = len(par)
    slots = P + n
    mask = np.zeros((n, slots), bool)
    for i in range(n):
        ipos = P + depth[i]
        anc = _ancestors(par, i)
        for s in range(slots):
            jpos = s if s < P else P + depth[s - P]
            if s >= P and (s - P) not in anc:
                continue
            if window and not jpos > ipos - window:
                continue
            mask[i, s] = True
    G = Hq // Hkv
    for h in range(Hq):
        K = torch.from_numpy(_dequant_rows(c, 0, kv_type, 0, h // G, D)[:slots])
        V = torch.from_numpy(_dequant_rows(c, 1, kv_type, 0, h // G, D)[:slots])
        Q = torch.from_numpy(synth.bf16_to_f32(inp["q"][0, :n, h]).astype(np.float64))
        ref = torch.nn.functional.scaled_dot_product_attention(
            Q[None, None], K[None, None], V[None, None], attn_mask=torch.from_numpy(mask)[None, None])
        np.testing.assert_allclose(out[0, :n, h], ref[0, 0].numpy(), rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("kv_type", TYPES)
def test_window_zero_equals_window_covering_everything(orc, kv_type):
    rng = np.random.default_rng(200 + kv_type)
    par = synth.uniform_tree(rng, 8)
    P, cap = 17, 30
    args = _case(rng, kv_type, [par], P, cap)
    a, ca = _run(orc, *args, window=0, kv_type=kv_type)
    b, cb = _run(orc, *args, window=P + 8, kv_type=kv_type)
    assert np.array_equal(a, b)
    for key in ("kq", "vq", "ks", "vs"):
        if ca[key] is not None:
            assert np.array_equal(ca[key], cb[key])


@pytest.mark.parametrize("kv_type", TYPES)
def test_single_visible_key_returns_its_value(orc, kv_type):
    # Empty prefix and a root-only tree: the softmax has one term.
    rng = np.random.default_rng(300 + kv_type)
    args = _case(rng, kv_type, [synth.chain_tree(1)], 0, 4)
    out, c = _run(orc, *args, window=0, kv_type=kv_type)
    D = out.shape[-1]
    for h in range(out.shape[2]):
        v = _dequant_rows(c, 1, kv_type, 0, h // 2, D)[0]
        np.testing.assert_array_equal(out[0, 0, h], v.astype(np.float32))


@pytest.mark.parametrize("kv_type", [synth.KV_Q8_0, synth.KV_Q4_0])
def test_identical_keys_average_the_values(orc, kv_type):
    rng = np.random.default_rng(400 + kv_type)
    P, cap, window = 12, 20, 6
    args = _case(rng, kv_type, [synth.chain_tree(1)], P, cap)
    _, c = _run(orc, *args, window=0, kv_type=kv_type)
    cache = args[4]
    for key in ("kq", "ks"):                 # every cached key := the root's quantised key
        cache[key][:, :, :P] = c[key][:, :, P:P + 1]
    out, c2 = _run(orc, *args, window=window, kv_type=kv_type)
    D = out.shape[-1]
    for h in range(out.shape[2]):
        V = _dequant_rows(c2, 1, kv_type, 0, h // 2, D)
        want = V[P - window + 1:P + 1].mean(axis=0)   # window keeps the last W positions
        np.testing.assert_allclose(out[0, 0, h], want, rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("kv_type", TYPES)
def test_non_ancestors_do_not_leak(orc, kv_type):
    rng = np.random.default_rng(500 + kv_type)
    par = np.array([-1, 0, 0, 1, 2, 3, 4], np.int32)   # two branches
    P, cap = 10, 20
    parent, n_nodes, n_past, inp, cache = _case(rng, kv_type, [par], P, cap)
    a, _ = _run(orc, parent, n_nodes, n_past, inp, cache, 0, kv_type)
    inp2 = {k: v.copy() for k, v in inp.items()}
    # perturb branch {2, 4, 6}; branch {1, 3, 5} must not see it
    inp2["k_new"][0, [2, 4, 6]] = synth.bf16_bits(rng.standard_normal((3,) + inp["k_new"].shape[2:]))
    inp2["v_new"][0, [2, 4, 6]] = synth.bf16_bits(rng.standard_normal((3,) + inp["v_new"].shape[2:]))
    b, _ = _run(orc, parent, n_nodes, n_past, inp2, cache, 0, kv_type)
    for i in (0, 1, 3, 5):
        assert np.array_equal(a[0, i], b[0, i])
    assert not np.array_equal(a[0, 6], b[0, 6])


@pytest.mark.parametrize("kv_type", TYPES)
@pytest.mark.parametrize("window", [0, 4])
def test_chain_equals_sequential_decode(orc, kv_type, window):
    # Chain verify == decoding the same tokens one at a time with a growing
    # cache (README "Correctness": bit-identical to autoregressive decode).
    rng = np.random.default_rng(600 + kv_type + window)
    n, P, cap = 6, 9, 24
    parent, n_nodes, n_past, inp, cache = _case(rng, kv_type, [synth.chain_tree(n)], P, cap)
    chain_out, _ = _run(orc, parent, n_nodes, n_past, inp, cache, window, kv_type)
    c = synth.copy_cache(cache)
    root = synth.batch_trees([synth.chain_tree(1)], 1)
    for i in range(n):
        step = {k: v[:, i:i + 1].copy() for k, v in inp.items()}
        o = orc.tree_attn_verify(root[0], root[1], np.array([P + i], np.int32), step["q"],
                                 step["k_new"], step["v_new"], c, window, kv_type)
        assert np.array_equal(o[0, 0], chain_out[0, i])


def test_capacity_and_topology_errors(orc):
    rng = np.random.default_rng(700)
    parent, n_nodes, n_past, inp, cache = _case(rng, synth.KV_Q8_0, [synth.chain_tree(5)], 8, 12)
    with pytest.raises(orc.OracleError) as e:
        orc.tree_attn_verify(parent, n_nodes, n_past, inp["q"], inp["k_new"], inp["v_new"],
                             synth.copy_cache(cache), 0, synth.KV_Q8_0)
    assert e.value.code == orc.ERR_CAPACITY
    bad = parent.copy()
    bad[0, 3] = 3
    with pytest.raises(orc.OracleError) as e:
        orc.tree_attn_verify(bad, n_nodes, np.array([2], np.int32), inp["q"], inp["k_new"],
                             inp["v_new"], synth.copy_cache(cache), 0, synth.KV_Q8_0)
    assert e.value.code == orc.ERR_TOPOLOGY


def test_row_selection_matches_full_computation(orc):
    rng = np.random.default_rng(800)
    pars = [synth.uniform_tree(rng, 6), synth.uniform_tree(rng, 4)]
    parent, n_nodes, n_past, inp, cache = _case(rng, synth.KV_Q8_0, pars, 7, 16)
    full, _ = _run(orc, parent, n_nodes, n_past, inp, cache, 3, synth.KV_Q8_0)
    rows = np.array([(0 * 6 + 5) * 4 + 2, (1 * 6 + 3) * 4 + 0, 1], np.int32)
    part = orc.tree_attn_verify(parent, n_nodes, n_past, inp["q"], inp["k_new"], inp["v_new"],
                                synth.copy_cache(cache), 3, synth.KV_Q8_0, rows=rows)
    flat_full = full.reshape(-1, full.shape[-1])
    flat_part = part.reshape(-1, part.shape[-1])
    for r in rows:
        assert np.array_equal(flat_full[r], flat_part[r])


@pytest.mark.parametrize("kv_type", ASYM)
def test_asymmetric_planes_match_their_symmetric_formats(orc, kv_type):
    # An asymmetric cache writes the tree's keys exactly as the symmetric
    # cache of the key format does and its values as the cache of the value
    # format (compared byte for byte), and reads each plane in its own format
    # (the output equals fp64 attention over the per-plane dequantised rows).
    rng = np.random.default_rng(300 + kv_type)
    par = synth.ddtree(rng, 11, 50)[0]
    P, cap, Hq, Hkv, D = 17, 32, 4, 2, 64
    parent, n_nodes, n_past, inp, cache = _case(rng, kv_type, [par], P, cap, Hq, Hkv, D)
    out, c = _run(orc, parent, n_nodes, n_past, inp, cache, 0, kv_type)
    kt, vt = _plane_type(kv_type, 0), _plane_type(kv_type, 1)
    _, ck = _run(orc, parent, n_nodes, n_past, inp, synth.kv_cache(rng, 1, Hkv, cap, D, kt), 0, kt)
    _, cv = _run(orc, parent, n_nodes, n_past, inp, synth.kv_cache(rng, 1, Hkv, cap, D, vt), 0, vt)
    n = len(par)
    for key, src in (("kq", ck), ("ks", ck), ("vq", cv), ("vs", cv)):
        np.testing.assert_array_equal(c[key][:, :, P:P + n], src[key][:, :, P:P + n])
    G = Hq // Hkv
    mask = np.zeros((n, P + n), bool)
    for i in range(n):
        mask[i, :P] = True
        for l in _ancestors(par, i):
            mask[i, P + l] = True
    for h in range(Hq):
        K = torch.from_numpy(_dequant_rows(c, 0, kv_type, 0, h // G, D)[:P + n])
        V = torch.from_numpy(_dequant_rows(c, 1, kv_type, 0, h // G, D)[:P + n])
        Q = torch.from_numpy(synth.bf16_to_f32(inp["q"][0, :n, h]).astype(np.float64))
        ref = torch.nn.functional.scaled_dot_product_attention(
            Q[None, None], K[None, None], V[None, None], attn_mask=torch.from_numpy(mask)[None, None])
        np.testing.assert_allclose(out[0, :n, h], ref[0, 0].numpy(), rtol=1e-6, atol=1e-6)
