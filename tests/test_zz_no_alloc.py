"""The attention verify that allocates nothing (dflv_tree_attn_verify_noalloc).

Some callers cannot allocate device memory on the path that runs a step: a
serving runtime that gives each plugin a fixed pool, an allocator that must
not be entered while a CUDA graph is captured, or a loop that cannot take
cudaMalloc's implicit synchronisation.  This entry point takes no workspace:
it merges through one fixed scratch array in the library's own device memory.

Here it is called through the C ABI on two different layers in a row (the
second call finds the first call's partials in the shared scratch) and its
outputs and cache slots are compared with the regular entry point given a
workspace of its own, within the float tolerance of the other parity tests
(the two take the same path, so they agree to the bit in practice).  A shape
whose merge needs more than the fixed scratch is refused before any launch.
This file is collected last, and passes alone in a fresh process as well.
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


def _layer(rng, B, N, P, Hq, Hkv, D, kv_type):
    pars = [synth.ddtree(rng, N, 151936)[0] for _ in range(B)]
    parent, n_nodes = synth.batch_trees(pars, N)
    inp = synth.attn_inputs(rng, B, N, Hq, Hkv, D)
    cache = synth.kv_cache(rng, B, Hkv, P + 64, D, kv_type)
    return parent, n_nodes, inp, cache


def _run(dflv, fn, desc, parent, n_nodes, P, inp, cache, extra=()):
    B, N = parent.shape
    keep = {k: dev(v) for k, v in inp.items()}
    dc = {k: dev(v) for k, v in cache.items()}
    out = torch.full((B, N, desc.Hq, desc.D), float("nan"), device="cuda")
    st = zeros_status()
    rc = fn(desc, dev(parent), dev(n_nodes), dev(np.full(B, P, np.int32)), keep["q"], keep["k_new"], keep["v_new"],
            dflv.kv_layer(dc["kq"], dc["vq"], dc["ks"], dc["vs"]), out, st, *extra)
    dflv.check(rc, fn.__name__)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return host(out), {k: host(v) for k, v in dc.items()}


def test_noalloc_matches_the_workspace_entry_point_twice(dflv):
    rng = np.random.default_rng(2027)
    B, N, P, Hq, Hkv, D, W = 1, 22, 4096, 24, 4, 256, 2048
    desc = dflv.attn_desc(B, N, Hq, Hkv, D, P + 64, W, dflv.DFLV_KV_Q8_0, 1.0 / np.sqrt(D))
    need = dflv.dflv_attn_workspace_size(desc)
    assert 0 < need <= dflv.DFLV_NOALLOC_SCRATCH_BYTES
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    for call in range(2):   # two different layers, one after the other on one stream
        parent, n_nodes, inp, cache = _layer(rng, B, N, P, Hq, Hkv, D, synth.KV_Q8_0)
        ref, ref_planes = _run(dflv, dflv.dflv_tree_attn_verify, desc, parent, n_nodes, P, inp, cache, (ws, need))
        got, planes = _run(dflv, dflv.dflv_tree_attn_verify_noalloc, desc, parent, n_nodes, P, inp, cache)
        n = int(n_nodes[0])
        assert_close(got[0, :n], ref[0, :n], what=f"call {call} output")
        for key in ("kq", "vq", "ks", "vs"):
            assert np.array_equal(planes[key], ref_planes[key]), f"call {call} cache plane {key}"


def test_noalloc_refuses_a_shape_beyond_its_scratch(dflv):
    # 8 sequences of 64-node trees over a 131,072-token cache: the merge
    # needs more than the fixed scratch, so the call is refused on the host
    B, N, P, Hq, Hkv, D = 8, 64, 131072, 24, 4, 256
    desc = dflv.attn_desc(B, N, Hq, Hkv, D, P + 64, 0, dflv.DFLV_KV_Q4_0, 1.0 / np.sqrt(D))
    assert dflv.dflv_attn_workspace_size(desc) > dflv.DFLV_NOALLOC_SCRATCH_BYTES
    x = torch.zeros(16, dtype=torch.int32, device="cuda")
    st = zeros_status()
    rc = dflv.dflv_tree_attn_verify_noalloc(desc, x, x, x, x, x, x, dflv.kv_layer(x, x, x, x), x, st)
    assert rc == dflv.DFLV_ERR_CAPACITY
    torch.cuda.synchronize()
    assert int(st.item()) == 0
