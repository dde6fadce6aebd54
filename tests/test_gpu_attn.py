"""GPU parity: attention tree verify (libdflv) against the CPU oracle.

Outputs within the float tolerance of tests/gpu_util.py; the tree's
quantised keys/values written into cache slots [P, P + n) bit-identical to
the oracle's quantiser, every other slot untouched; sampled rows at the full
long-context size; capacity/topology errors through the status word.
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


def _plane_np_dtype(key, kv_type):
    if key in ("ks", "vs"):
        return np.uint16
    if kv_type == synth.KV_Q8_0_Q4_0:
        kv_type = synth.KV_Q8_0 if key == "kq" else synth.KV_Q4_0
    elif kv_type == synth.KV_Q4_0_Q8_0:
        kv_type = synth.KV_Q4_0 if key == "kq" else synth.KV_Q8_0
    return {synth.KV_Q8_0: np.int8, synth.KV_Q4_0: np.uint8, synth.KV_F32: np.float32,
            synth.KV_TQ3_0: np.uint8}[kv_type]


def gpu_attn(dflv, parent, n_nodes, n_past, inp, cache, window, kv_type, Hq, Hkv, D, expect_status=0,
             rows_only=None, ws=False):
    """ws: merge the key splits through a workspace of the queried size
    (else through the cluster's shared memory)."""
    B, N = parent.shape
    cap = cache["kq"].shape[2]
    keep = {k: dev(v) for k, v in inp.items()}
    dc = {k: (None if v is None else dev(v)) for k, v in cache.items()}
    keep.update(parent=dev(parent), n_nodes=dev(n_nodes), n_past=dev(n_past))
    out = torch.full((B, N, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    st = zeros_status()
    desc = dflv.attn_desc(B, N, Hq, Hkv, D, cap, window, kv_type, 1.0 / np.sqrt(D))
    wsb = dflv.dflv_attn_workspace_size(desc) if ws else 0
    if ws:
        assert wsb > 0 or D not in (128, 256) or kv_type == synth.KV_F32
    # stale contents must not matter: the workspace starts as NaN bytes
    wst = torch.full((max(wsb, 16) // 4,), float("nan"), device="cuda") if ws else None
    rc = dflv.dflv_tree_attn_verify(desc, keep["parent"], keep["n_nodes"], keep["n_past"], keep["q"],
                                    keep["k_new"], keep["v_new"], dflv.kv_layer(dc["kq"], dc["vq"], dc["ks"], dc["vs"]),
                                    out, st, wst, wsb)
    dflv.check(rc, "dflv_tree_attn_verify")
    torch.cuda.synchronize()
    assert int(st.item()) == expect_status
    planes = {k: (None if v is None else host(v, _plane_np_dtype(k, kv_type))) for k, v in dc.items()}
    return host(out), planes


def make_case(rng, kv_type, ns, P, cap, Hq, Hkv, D, tree="ddtree", scale_std=0.02):
    parents = []
    for n in ns:
        if tree == "ddtree":
            parents.append(synth.ddtree(rng, n, 1000)[0])
        elif tree == "chain":
            parents.append(synth.chain_tree(n))
        else:
            parents.append(synth.uniform_tree(rng, n))
    N = max(ns)
    parent, n_nodes = synth.batch_trees(parents, N)
    inp = synth.attn_inputs(rng, len(ns), N, Hq, Hkv, D)
    cache = synth.kv_cache(rng, len(ns), Hkv, cap, D, kv_type, scale_std=scale_std)
    n_past = np.asarray(P, np.int32) if np.ndim(P) else np.full(len(ns), P, np.int32)
    return parent, n_nodes, n_past, inp, cache


def check_against_oracle(dflv, orc, parent, n_nodes, n_past, inp, cache, window, kv_type, Hq, Hkv, D, ws=False):
    out, planes = gpu_attn(dflv, parent, n_nodes, n_past, inp, cache, window, kv_type, Hq, Hkv, D, ws=ws)
    ref_cache = synth.copy_cache(cache)
    ref = orc.tree_attn_verify(parent, n_nodes, n_past, inp["q"], inp["k_new"], inp["v_new"], ref_cache,
                               window, kv_type)
    e = 0.0
    for b in range(parent.shape[0]):
        e = max(e, assert_close(out[b, : n_nodes[b]], ref[b, : n_nodes[b]], what=f"o[b={b}]"))
    for key in ("kq", "vq", "ks", "vs"):
        if ref_cache[key] is None:
            continue
        assert np.array_equal(planes[key], ref_cache[key]), f"cache plane {key} differs"
    return e


SMALL = [
    # kv_type, ns, P, cap, Hq, Hkv, D, window, tree
    (synth.KV_Q8_0, [7], 100, 128, 4, 2, 256, 0, "uniform"),
    (synth.KV_Q8_0, [22, 9], [300, 57], 400, 6, 1, 256, 64, "ddtree"),
    (synth.KV_Q4_0, [22, 9], [300, 57], 400, 6, 1, 256, 64, "ddtree"),
    (synth.KV_Q8_0, [5], 0, 16, 2, 2, 128, 0, "uniform"),          # empty prefix
    (synth.KV_Q4_0, [13], 200, 256, 8, 2, 64, 1, "uniform"),       # window 1: only itself
    (synth.KV_Q8_0, [64], 513, 600, 6, 1, 256, 20, "chain"),       # window shorter than the chain
    (synth.KV_Q4_0, [64, 3], [1000, 5], 1100, 12, 2, 128, 0, "ddtree"),
    (synth.KV_Q8_0, [1], 77, 80, 24, 4, 256, 2048, "uniform"),     # window covering everything
    # asymmetric caches: keys and values in different formats
    (synth.KV_Q8_0_Q4_0, [22, 9], [300, 57], 400, 6, 1, 256, 64, "ddtree"),
    (synth.KV_Q4_0_Q8_0, [22, 9], [300, 57], 400, 6, 1, 256, 64, "ddtree"),
    (synth.KV_Q8_0_Q4_0, [64, 3], [1000, 5], 1100, 12, 2, 128, 0, "ddtree"),
    (synth.KV_Q4_0_Q8_0, [22], 4096, 4200, 24, 4, 256, 2048, "ddtree"),
    # TQ3_0: rotated 3.5-bit cache (query rotated in, output rotated back)
    (synth.KV_TQ3_0, [22, 9], [300, 57], 400, 6, 1, 256, 64, "ddtree"),
    (synth.KV_TQ3_0, [13], 200, 256, 8, 2, 128, 0, "uniform"),
    (synth.KV_TQ3_0, [64], 513, 600, 6, 1, 256, 20, "chain"),
    (synth.KV_TQ3_0, [64, 3], [1000, 5], 1100, 12, 2, 128, 0, "ddtree"),
]


@pytest.mark.parametrize("ws", [False, True], ids=["cluster_merge", "workspace_merge"])
@pytest.mark.parametrize("case", SMALL)
def test_attn_tree_verify_matches_oracle(dflv, orc, case, ws):
    kv_type, ns, P, cap, Hq, Hkv, D, window, tree = case
    rng = np.random.default_rng(len(ns) * 1000 + cap + D + window)
    args = make_case(rng, kv_type, ns, P, cap, Hq, Hkv, D, tree)
    check_against_oracle(dflv, orc, *args, window, kv_type, Hq, Hkv, D, ws=ws)


def test_attn_f32_cache_tiny_case(dflv, orc):
    # 1 attention head, head size 16, fp32 cache of 64 tokens, full attention
    rng = np.random.default_rng(1234)
    args = make_case(rng, synth.KV_F32, [7], 64, 80, 1, 1, 16, "uniform")
    check_against_oracle(dflv, orc, *args, 0, synth.KV_F32, 1, 1, 16)


@pytest.mark.parametrize("ws", [False, True], ids=["cluster_merge", "workspace_merge"])
def test_attn_full_size_32k_q8_window(dflv, orc, ws):
    # full-attention layer of a 27B-class target: 24 query heads, 4 KV heads,
    # head size 256, q8_0 cache of 32,768 tokens, window 2048, 22-node tree
    rng = np.random.default_rng(1236)
    args = make_case(rng, synth.KV_Q8_0, [22], 32768, 32768 + 64, 24, 4, 256, "ddtree")
    e = check_against_oracle(dflv, orc, *args, 2048, synth.KV_Q8_0, 24, 4, 256, ws=ws)
    print(f"full-size attention max rel err {e:.2e} ({'workspace' if ws else 'cluster'} merge)")


@pytest.mark.parametrize("ws", [False, True], ids=["cluster_merge", "workspace_merge"])
def test_attn_full_size_32k_tq3_window(dflv, orc, ws):
    # the same layer over a TQ3_0 cache (the pages' default KV type)
    rng = np.random.default_rng(1237)
    args = make_case(rng, synth.KV_TQ3_0, [22], 32768, 32768 + 64, 24, 4, 256, "ddtree")
    e = check_against_oracle(dflv, orc, *args, 2048, synth.KV_TQ3_0, 24, 4, 256, ws=ws)
    print(f"full-size TQ3_0 attention max rel err {e:.2e} ({'workspace' if ws else 'cluster'} merge)")


def test_attn_long_context_tq3_full_attention(dflv, orc):
    # 2 sequences over a 131,072-token TQ3_0 cache, full attention: every
    # row of one whole sequence against the oracle, and the tree slots of both
    rng = np.random.default_rng(1301)
    B, n, P, Hq, Hkv, D = 2, 22, 131072, 24, 4, 256
    parents = [synth.ddtree(rng, n, 151936)[0] for _ in range(B)]
    parent, n_nodes = synth.batch_trees(parents, n)
    inp = synth.attn_inputs(rng, B, n, Hq, Hkv, D)
    cache = synth.kv_cache(rng, B, Hkv, P + 64, D, synth.KV_TQ3_0)
    n_past = np.full(B, P, np.int32)
    out, planes = gpu_attn(dflv, parent, n_nodes, n_past, inp, cache, 0, synth.KV_TQ3_0, Hq, Hkv, D, ws=True)
    rows = np.arange(1 * n * Hq, 2 * n * Hq, dtype=np.int32)
    ref_cache = synth.copy_cache(cache)
    ref = orc.tree_attn_verify(parent, n_nodes, n_past, inp["q"], inp["k_new"], inp["v_new"], ref_cache, 0,
                               synth.KV_TQ3_0, rows=rows)
    e = assert_close(out[1], ref[1], what="every row of sequence 1")
    print(f"131K TQ3_0 full attention max rel err {e:.2e}")
    for key in ("kq", "vq", "ks", "vs"):
        sl = np.s_[:, :, P:P + n]
        assert np.array_equal(planes[key][sl], ref_cache[key][sl]), key


@pytest.mark.parametrize("n", [8, 22, 64])
def test_attn_long_context_q4_full_attention(dflv, orc, n):
    # 8 sequences, 131,072-token q4_0 cache, full attention: one whole
    # sequence and sampled rows of others
    rng = np.random.default_rng(1239 + n)
    B, P, Hq, Hkv, D = 8, 131072, 24, 4, 256
    parents = [synth.ddtree(rng, n, 151936)[0] for _ in range(B)]
    parent, n_nodes = synth.batch_trees(parents, n)
    inp = synth.attn_inputs(rng, B, n, Hq, Hkv, D)
    cache = synth.kv_cache(rng, B, Hkv, P + 64, D, synth.KV_Q4_0)
    n_past = np.full(B, P, np.int32)
    out, planes = gpu_attn(dflv, parent, n_nodes, n_past, inp, cache, 0, synth.KV_Q4_0, Hq, Hkv, D, ws=n != 8)
    # every row of one whole sequence (all nodes x all query heads: every row
    # tile, KV head and key split of that sequence's launch blocks), plus
    # sampled rows of three other sequences
    full_b = {8: 5, 22: 2, 64: 6}[n]
    rows = list(range(full_b * n * Hq, (full_b + 1) * n * Hq))
    sampled = []
    for b in (0, 3, 7):
        for i in (0, n - 1, int(rng.integers(0, n))):
            sampled.append((b * n + i) * Hq + int(rng.integers(0, Hq)))
    sampled = np.unique(np.asarray(sampled, np.int32))
    rows = np.unique(np.concatenate([np.asarray(rows, np.int32), sampled]))
    ref_cache = synth.copy_cache(cache)
    ref = orc.tree_attn_verify(parent, n_nodes, n_past, inp["q"], inp["k_new"], inp["v_new"], ref_cache, 0,
                               synth.KV_Q4_0, rows=rows)
    flat_o, flat_r = out.reshape(-1, D), ref.reshape(-1, D)
    assert_close(out[full_b], ref[full_b], what=f"every row of sequence {full_b}")
    # the tolerance's rms is taken over the sampled rows
    assert_close(flat_o[sampled], flat_r[sampled], what="sampled rows")
    for key in ("kq", "vq", "ks", "vs"):
        sl = np.s_[:, :, P:P + n]
        assert np.array_equal(planes[key][sl], ref_cache[key][sl]), key


def test_attn_errors_set_status(dflv):
    rng = np.random.default_rng(9)
    # capacity: P + n > cap
    parent, n_nodes, n_past, inp, cache = make_case(rng, synth.KV_Q8_0, [5], 30, 32, 2, 1, 64, "uniform")
    gpu_attn(dflv, parent, n_nodes, n_past, inp, cache, 0, synth.KV_Q8_0, 2, 1, 64,
             expect_status=dflv.DFLV_DEV_CAPACITY)
    # topology
    parent, n_nodes, n_past, inp, cache = make_case(rng, synth.KV_Q8_0, [5], 10, 32, 2, 1, 64, "uniform")
    parent[0, 3] = 4
    out, planes = gpu_attn(dflv, parent, n_nodes, n_past, inp, cache, 0, synth.KV_Q8_0, 2, 1, 64,
                           expect_status=dflv.DFLV_DEV_TOPOLOGY)


def test_attn_layers_back_to_back_with_early_prefetch(dflv, orc):
    # three attention layers launched back to back on one stream, every
    # layer after the first reading its tree and cache prefix before the
    # dependency wait; q, k_new and v_new of each layer are written by an
    # elementwise kernel queued just before it, so a kernel that read them
    # before its wait could still see the zeros they held
    rng = np.random.default_rng(1250)
    Hq, Hkv, D, P, W = 24, 4, 256, 3000, 2048
    par, _ = synth.ddtree(rng, 22, 151936)
    parent, n_nodes = synth.batch_trees([par], 22)
    n_past = np.array([P], np.int32)
    dp, dn, dP = dev(parent), dev(n_nodes), dev(n_past)
    st = zeros_status()
    layers = []
    for li in range(3):
        inp = synth.attn_inputs(rng, 1, 22, Hq, Hkv, D)
        cache = synth.kv_cache(rng, 1, Hkv, P + 64, D, synth.KV_Q8_0)
        src = {k: dev(v) for k, v in inp.items()}
        dst = {k: torch.zeros_like(v) for k, v in src.items()}
        dc = {k: dev(v) for k, v in cache.items()}
        out = torch.full((1, 22, Hq, D), float("nan"), device="cuda")
        layers.append((inp, cache, src, dst, dc, out))
    torch.cuda.synchronize()
    for li, (inp, cache, src, dst, dc, out) in enumerate(layers):
        for k in ("q", "k_new", "v_new"):
            torch.mul(src[k], 1, out=dst[k])
        flags = 0 if li == 0 else dflv.DFLV_FLAG_EARLY_PREFETCH
        desc = dflv.attn_desc(1, 22, Hq, Hkv, D, P + 64, W, synth.KV_Q8_0, 1.0 / np.sqrt(D), flags)
        if li == 0:  # one workspace shared by the three calls on the stream
            wsb = dflv.dflv_attn_workspace_size(desc)
            wst = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        dflv.check(dflv.dflv_tree_attn_verify(desc, dp, dn, dP, dst["q"], dst["k_new"], dst["v_new"],
                                              dflv.kv_layer(dc["kq"], dc["vq"], dc["ks"], dc["vs"]), out, st, wst,
                                              wsb))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for inp, cache, src, dst, dc, out in layers:
        ref_cache = synth.copy_cache(cache)
        ref = orc.tree_attn_verify(parent, n_nodes, n_past, inp["q"], inp["k_new"], inp["v_new"], ref_cache, W,
                                   synth.KV_Q8_0)
        assert_close(host(out)[0, :22], ref[0, :22], what="o")
        for key in ("kq", "vq", "ks", "vs"):
            got = host(dc[key], _plane_np_dtype(key, synth.KV_Q8_0))
            assert np.array_equal(got, ref_cache[key]), key
