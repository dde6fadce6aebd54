"""Pins for the oracle's TQ3_0 cache (CPU only).

The pages ("Luce DFlash" README, "Asymmetric K/V quantization" and the
KV-cache note under "Results") fix the bit rate, 3.5 bits per value, and that
an FWHT rotation is applied to the query and undone on the attention output
when the keys are TQ3_0.  The block layout, the codebook and the rotation
size are readings (oracle/oracle.h).  The pins:
  * hand-worked examples (tests/golden/tq3_examples.json): decoding a known
    byte pattern, quantising a block whose halves separate round-half-away
    from ties-to-even, and a 4-point transform;
  * the bit rate against the pages' 3.5;
  * the rotation against scipy's Hadamard matrix (a library routine), and its
    being its own inverse;
  * the quantiser's round-trip error bound;
  * attention: fp64 scaled_dot_product_attention on the rotated query over
    the dequantised (rotated) cache, rotated back with the library Hadamard
    matrix, equals the oracle's output; the tree's keys and values are stored
    rotated; a chain equals sequential decode; compaction moves the bytes.
"""
import json
import os

import numpy as np
import pytest
import torch
from scipy.linalg import hadamard

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tq3_examples.json")
TQ3 = synth.KV_TQ3_0


@pytest.fixture(scope="module")
def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _unpack(codes_row, D):
    """3-bit codes of one cache row (bytes [D/32 * 12]) -> [D] ints, by a
    library bit unpacking (little-endian bit order)."""
    blocks = codes_row.reshape(D // 32, 12)
    bits = np.unpackbits(blocks, axis=1, bitorder="little").reshape(D // 32, 32, 3)
    return (bits[..., 0] + 2 * bits[..., 1] + 4 * bits[..., 2]).reshape(D).astype(np.int64)


def _dequant_rows(cache, which, b, h, D):
    q = cache["kq" if which == 0 else "vq"][b, h]
    s = cache["ks" if which == 0 else "vs"][b, h].view(np.float16).astype(np.float64)
    out = np.zeros((q.shape[0], D))
    for r in range(q.shape[0]):
        c = _unpack(q[r], D).reshape(D // 32, 32)
        out[r] = ((c - 4) * s[r][:, None]).reshape(D)
    return out


def test_worked_examples(orc, golden):
    ex = golden["dequant"]
    d16 = int(ex["d16"], 16)
    assert orc.half_to_float(d16) == ex["d"]
    x = orc.dequantize_tq3_0(np.array(ex["bytes"], np.uint8), d16)
    np.testing.assert_array_equal(x[:8], ex["x_first8"])
    np.testing.assert_array_equal(x[8:16], ex["x_first8"])
    ex = golden["quantize"]
    xin = np.zeros(32, np.float32)
    for j, v in ex["x_nonzero"].items():
        xin[int(j)] = v
    codes, d16 = orc.quantize_tq3_0(xin)
    assert d16 == int(ex["d16"], 16)
    assert list(codes) == ex["bytes"]
    np.testing.assert_array_equal(orc.dequantize_tq3_0(codes, d16)[:8], ex["x_back_first8"])
    ex = golden["fwht"]
    np.testing.assert_array_equal(orc.fwht(np.array(ex["x"], np.float32)), ex["y"])


def test_bits_per_value_is_the_pages_figure():
    D = 256
    c = synth.kv_cache(np.random.default_rng(0), 1, 1, 4, D, TQ3)
    bits = (c["kq"].shape[-1] + c["ks"].shape[-1] * 2) * 8 / D
    assert bits == 3.5


@pytest.mark.parametrize("n", [4, 32, 64, 128, 256])
def test_rotation_is_the_normalised_hadamard_transform(orc, n):
    rng = np.random.default_rng(n)
    x = rng.standard_normal((5, n)).astype(np.float32)
    y = orc.fwht(x)
    ref = x.astype(np.float64) @ hadamard(n).T / np.sqrt(n)
    np.testing.assert_allclose(y, ref, rtol=0, atol=2e-6 * np.abs(x).max() * np.log2(n))
    # its own inverse, and norm-preserving, up to fp32 rounding
    np.testing.assert_allclose(orc.fwht(y), x, rtol=0, atol=1e-5 * np.abs(x).max())
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-5)


def test_quantiser_round_trip_bound(orc):
    rng = np.random.default_rng(1)
    for _ in range(200):
        x = (rng.standard_normal(32) * rng.uniform(0.01, 10)).astype(np.float32)
        codes, d16 = orc.quantize_tq3_0(x)
        d = np.float32(np.abs(x).max()) / np.float32(3.0)
        dh = orc.half_to_float(d16)
        err = np.abs(orc.dequantize_tq3_0(codes, d16) - x.astype(np.float64))
        # half a step from the rounding (fp32 products) plus the scale's fp16 rounding on at most 4 steps
        assert np.all(err <= 0.5 * float(d) * (1 + 1e-6) + 4 * abs(float(d) - dh) + 1e-12)
    codes, d16 = orc.quantize_tq3_0(np.zeros(32, np.float32))
    assert d16 == 0 and np.all(orc.dequantize_tq3_0(codes, d16) == 0)


def _case(rng, parents, P, cap, Hq=4, Hkv=2, D=64):
    N = max(len(p) for p in parents)
    parent, n_nodes = synth.batch_trees(parents, N)
    inp = synth.attn_inputs(rng, len(parents), N, Hq, Hkv, D)
    cache = synth.kv_cache(rng, len(parents), Hkv, cap, D, TQ3, scale_std=0.05)
    return parent, n_nodes, np.full(len(parents), P, np.int32), inp, cache


@pytest.mark.parametrize("window", [0, 5, 13])
def test_attention_matches_library_in_the_rotated_basis(orc, window):
    rng = np.random.default_rng(700 + window)
    par = synth.uniform_tree(rng, 9)
    P, cap, Hq, Hkv, D = 21, 40, 4, 2, 64
    parent, n_nodes, n_past, inp, cache = _case(rng, [par], P, cap, Hq, Hkv, D)
    c = synth.copy_cache(cache)
    out = orc.tree_attn_verify(parent, n_nodes, n_past, inp["q"], inp["k_new"], inp["v_new"], c, window, TQ3)
    depth = synth.tree_depths(par)
    n = len(par)
    slots = P + n
    mask = np.zeros((n, slots), bool)
    for i in range(n):
        anc, a = set(), i
        while a >= 0:
            anc.add(a)
            a = par[a]
        ipos = P + depth[i]
        for s in range(slots):
            jpos = s if s < P else P + depth[s - P]
            if s >= P and (s - P) not in anc:
                continue
            if window and not jpos > ipos - window:
                continue
            mask[i, s] = True
    H = hadamard(D).astype(np.float64) / np.sqrt(D)
    G = Hq // Hkv
    for h in range(Hq):
        K = torch.from_numpy(_dequant_rows(c, 0, 0, h // G, D)[:slots])
        V = torch.from_numpy(_dequant_rows(c, 1, 0, h // G, D)[:slots])
        q = synth.bf16_to_f32(inp["q"][0, :n, h]).astype(np.float64)
        Q = torch.from_numpy(q @ H.T)                       # the query into the keys' basis
        o_rot = torch.nn.functional.scaled_dot_product_attention(
            Q[None, None], K[None, None], V[None, None], attn_mask=torch.from_numpy(mask)[None, None])
        ref = o_rot[0, 0].numpy() @ H.T                     # back from the values' basis
        np.testing.assert_allclose(out[0, :n, h], ref, rtol=1e-6, atol=1e-6)


def test_tree_keys_and_values_are_stored_rotated(orc):
    rng = np.random.default_rng(5)
    par = synth.uniform_tree(rng, 6)
    P, cap, D = 10, 20, 128
    parent, n_nodes, n_past, inp, cache = _case(rng, [par], P, cap, 2, 1, D)
    c = synth.copy_cache(cache)
    orc.tree_attn_verify(parent, n_nodes, n_past, inp["q"], inp["k_new"], inp["v_new"], c, 0, TQ3)
    for plane, scales, src in (("kq", "ks", "k_new"), ("vq", "vs", "v_new")):
        for i in range(len(par)):
            row = orc.fwht(synth.bf16_to_f32(inp[src][0, i, 0]))
            for blk in range(D // 32):
                codes, d16 = orc.quantize_tq3_0(row[32 * blk:32 * blk + 32])
                assert list(c[plane][0, 0, P + i, 12 * blk:12 * blk + 12]) == list(codes)
                assert int(c[scales][0, 0, P + i, blk]) == d16
        # the slots below P are untouched
        np.testing.assert_array_equal(c[plane][0, :, :P], cache[plane][0, :, :P])


@pytest.mark.parametrize("window", [0, 4])
def test_chain_equals_sequential_decode(orc, window):
    rng = np.random.default_rng(800 + window)
    n, P, cap = 6, 9, 24
    parent, n_nodes, n_past, inp, cache = _case(rng, [synth.chain_tree(n)], P, cap)
    c = synth.copy_cache(cache)
    chain_out = orc.tree_attn_verify(parent, n_nodes, n_past, inp["q"], inp["k_new"], inp["v_new"], c, window, TQ3)
    c = synth.copy_cache(cache)
    root = synth.batch_trees([synth.chain_tree(1)], 1)
    for i in range(n):
        step = {k: v[:, i:i + 1].copy() for k, v in inp.items()}
        o = orc.tree_attn_verify(root[0], root[1], np.array([P + i], np.int32), step["q"], step["k_new"],
                                 step["v_new"], c, window, TQ3)
        assert np.array_equal(o[0, 0], chain_out[0, i])


def test_compaction_moves_the_rows(orc):
    rng = np.random.default_rng(9)
    B, Hkv, cap, D, N, P = 1, 2, 30, 64, 6, 12
    cache = synth.kv_cache(rng, B, Hkv, cap, D, TQ3)
    before = synth.copy_cache(cache)
    path = np.array([[0, 2, 3, 0, 0, 0]], np.int32)       # 2 -> 1 and 3 -> 2: a destination is a source
    orc.kv_commit(cache, TQ3, path, np.array([3], np.int32), np.array([P], np.int32))
    for plane in ("kq", "vq", "ks", "vs"):
        for m, src in enumerate([0, 2, 3]):
            np.testing.assert_array_equal(cache[plane][0, :, P + m], before[plane][0, :, P + src])
        np.testing.assert_array_equal(cache[plane][0, :, :P], before[plane][0, :, :P])


def test_head_size_must_be_a_power_of_two(orc):
    rng = np.random.default_rng(11)
    parent, n_nodes, n_past, inp, cache = _case(rng, [synth.chain_tree(2)], 4, 8, 2, 1, 96)
    with pytest.raises(orc.OracleError):
        orc.tree_attn_verify(parent, n_nodes, n_past, inp["q"], inp["k_new"], inp["v_new"], cache, 0, TQ3)
