"""The C-ABI library builds for sm_103a, loads, exports every symbol the
header declares, and rejects bad arguments on the host (CPU only: no call
here reaches a kernel)."""
import ctypes

import pytest

import speculative_decoding_tree_layer_gb300 as pkg
from speculative_decoding_tree_layer_gb300 import dflv


@pytest.fixture(scope="module")
def lib():
    pkg.build()
    return dflv.load()


def test_exports_every_declared_symbol(lib):
    names = dflv.header_symbols()
    assert set(names) >= {"dflv_tree_gdn_verify", "dflv_tree_attn_verify", "dflv_accept_greedy",
                          "dflv_commit_rollback", "dflv_gdn_workspace_size", "dflv_attn_workspace_size",
                          "dflv_status_string", "dflv_tree_conv_verify", "dflv_conv_commit", "dflv_ddtree_build"}
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(6):
        assert dflv.status_string(code)
    assert dflv.status_string(0) == "ok"


def _gdn_call(desc, **over):
    args = dict(parent=16, n_nodes=16, q=16, k=16, v=16, beta=16, log_alpha=16, state=16, out=16,
                factors=dflv.dflv_gdn_factors(16, 16, 16), status_dev=16)
    args.update(over)
    return dflv.dflv_tree_gdn_verify(desc, stream=0, **args)


def test_gdn_host_validation(lib):
    ok = dflv.gdn_desc(1, 22, 16, 48, 128, 128)
    assert _gdn_call(dflv.gdn_desc(1, 65, 16, 48, 128, 128)) == dflv.DFLV_ERR_UNSUPPORTED
    assert _gdn_call(dflv.gdn_desc(1, 22, 16, 48, 96, 128)) == dflv.DFLV_ERR_UNSUPPORTED
    assert _gdn_call(dflv.gdn_desc(1, 22, 16, 40, 128, 128)) == dflv.DFLV_ERR_INVALID_ARG
    assert _gdn_call(dflv.gdn_desc(0, 22, 16, 48, 128, 128)) == dflv.DFLV_ERR_INVALID_ARG
    # only DFLV_FLAG_EARLY_PREFETCH: the launchers keep higher bits for
    # themselves (the layer-input prefetch), so no caller can set them
    for flags in (2, 1 << 16, 1 | (1 << 16)):
        assert _gdn_call(dflv.gdn_desc(1, 22, 16, 48, 128, 128, flags)) == dflv.DFLV_ERR_INVALID_ARG
    assert _gdn_call(ok, q=None) == dflv.DFLV_ERR_INVALID_ARG
    assert _gdn_call(ok, state=24) == dflv.DFLV_ERR_INVALID_ARG          # misaligned
    assert _gdn_call(ok, factors=dflv.dflv_gdn_factors(16, None, 16)) == dflv.DFLV_ERR_INVALID_ARG
    assert dflv.dflv_gdn_workspace_size(ok) == 0


def test_attn_host_validation(lib):
    cache = dflv.dflv_kv_layer(16, 16, 16, 16)

    def call(desc, **over):
        args = dict(parent=16, n_nodes=16, n_past=16, q=16, k_new=16, v_new=16, cache=cache, out=16,
                    status_dev=16)
        args.update(over)
        return dflv.dflv_tree_attn_verify(desc, stream=0, **args)

    base = dict(B=1, N_max=22, Hq=24, Hkv=4, D=256, cap=40000, window=2048, kv_type=0, scale=0.0625)

    def d(**kw):
        x = dict(base)
        x.update(kw)
        return dflv.attn_desc(**x)

    assert call(d(N_max=65)) == dflv.DFLV_ERR_UNSUPPORTED
    assert call(d(D=96)) == dflv.DFLV_ERR_UNSUPPORTED
    assert call(d(window=-1)) == dflv.DFLV_ERR_INVALID_ARG
    assert call(d(Hq=25)) == dflv.DFLV_ERR_INVALID_ARG
    assert call(d(cap=10)) == dflv.DFLV_ERR_CAPACITY
    assert call(d(kv_type=7)) == dflv.DFLV_ERR_UNSUPPORTED
    # asymmetric caches run on the tensor-core kernel only (head sizes 128, 256)
    assert call(d(kv_type=dflv.DFLV_KV_Q8_0_Q4_0, D=64)) == dflv.DFLV_ERR_UNSUPPORTED
    assert call(d(kv_type=dflv.DFLV_KV_Q4_0_Q8_0, D=64)) == dflv.DFLV_ERR_UNSUPPORTED
    assert call(d(scale=float("nan"))) == dflv.DFLV_ERR_INVALID_ARG
    for flags in (2, 1 << 16, 1 | (1 << 16)):
        assert call(d(flags=flags)) == dflv.DFLV_ERR_INVALID_ARG
    assert call(d(), cache=dflv.dflv_kv_layer(16, 16, None, 16)) == dflv.DFLV_ERR_INVALID_ARG
    assert call(d(), cache=dflv.dflv_kv_layer(16, 16, 18, 16)) == dflv.DFLV_ERR_INVALID_ARG  # scale rows
    assert call(d(), q=None) == dflv.DFLV_ERR_INVALID_ARG
    assert call(d(), workspace=24, ws_bytes=1 << 20) == dflv.DFLV_ERR_INVALID_ARG  # misaligned workspace
    # the workspace size follows the device's launch plan (a GPU test checks
    # it is positive there); an invalid descriptor needs none
    assert dflv.dflv_attn_workspace_size(d(N_max=65)) == 0
    assert dflv.dflv_attn_workspace_size(d()) >= 0


def test_accept_and_commit_host_validation(lib):
    P = 16
    assert dflv.dflv_accept_greedy(1, 65, 100, P, P, P, P, P, P, P, P, P, stream=0) == dflv.DFLV_ERR_UNSUPPORTED
    assert dflv.dflv_accept_greedy(0, 22, 100, P, P, P, P, P, P, P, P, P, stream=0) == dflv.DFLV_ERR_INVALID_ARG
    assert dflv.dflv_accept_greedy(1, 22, 100, None, P, P, P, P, P, P, P, P, stream=0) == dflv.DFLV_ERR_INVALID_ARG
    assert dflv.dflv_accept_greedy(1, 22, 100, 20, P, P, P, P, P, P, P, P, stream=0) == dflv.DFLV_ERR_INVALID_ARG
    g = dflv.gdn_desc(1, 22, 16, 48, 128, 128)
    fac = dflv.dflv_gdn_factors(P, P, P)
    assert dflv.dflv_commit_rollback(g, 129, [P] * 129, [fac] * 129, None, 0, [], P, P, P, P,
                                     stream=0) == dflv.DFLV_ERR_UNSUPPORTED
    assert dflv.dflv_commit_rollback(g, 1, [None], [fac], None, 0, [], P, P, P, P,
                                     stream=0) == dflv.DFLV_ERR_INVALID_ARG
    a = dflv.attn_desc(2, 22, 24, 4, 256, 40000, 0, 0, 0.0625)
    assert dflv.dflv_commit_rollback(g, 1, [P], [fac], a, 1, [dflv.dflv_kv_layer(P, P, P, P)], P, P, P, P,
                                     stream=0) == dflv.DFLV_ERR_INVALID_ARG   # batch mismatch


def test_conv_host_validation(lib):
    P = 16

    def call(desc, **over):
        args = dict(parent=P, n_nodes=P, x=P, conv_state=P, weight=P, out=P, status_dev=P)
        args.update(over)
        return dflv.dflv_tree_conv_verify(desc, stream=0, **args)

    ok = dflv.conv_desc(1, 22, 10240, 4)
    assert call(dflv.conv_desc(1, 22, 10, 4)) == dflv.DFLV_ERR_UNSUPPORTED      # C not a multiple of 4
    assert call(dflv.conv_desc(1, 22, 16, 9)) == dflv.DFLV_ERR_UNSUPPORTED      # K > 8
    assert call(dflv.conv_desc(1, 22, 16, 1)) == dflv.DFLV_ERR_UNSUPPORTED      # K < 2
    assert call(dflv.conv_desc(1, 65, 16, 4)) == dflv.DFLV_ERR_UNSUPPORTED
    assert call(dflv.conv_desc(0, 22, 16, 4)) == dflv.DFLV_ERR_INVALID_ARG
    assert call(dflv.conv_desc(1, 22, 16, 4, 2)) == dflv.DFLV_ERR_INVALID_ARG   # unknown flag
    assert call(ok, x=None) == dflv.DFLV_ERR_INVALID_ARG
    assert call(ok, x=24) == dflv.DFLV_ERR_INVALID_ARG                          # misaligned
    assert call(ok, parent=18) == dflv.DFLV_ERR_INVALID_ARG
    assert dflv.dflv_conv_commit(ok, 0, [], [], P, P, P, stream=0) == dflv.DFLV_ERR_INVALID_ARG
    assert dflv.dflv_conv_commit(ok, 129, [P] * 129, [P] * 129, P, P, P, stream=0) == dflv.DFLV_ERR_INVALID_ARG
    assert dflv.dflv_conv_commit(ok, 2, [P, None], [P, P], P, P, P, stream=0) == dflv.DFLV_ERR_INVALID_ARG
    assert dflv.dflv_conv_commit(ok, 1, [P], [24], P, P, P, stream=0) == dflv.DFLV_ERR_INVALID_ARG


def test_ddtree_host_validation(lib):
    P = 16

    def call(desc, **over):
        args = dict(draft_logits=P, root_token=P, topk_tok=P, topk_logp=P, parent=P, tokens=P, n_nodes=P, score=P,
                    status_dev=P)
        args.update(over)
        return dflv.dflv_ddtree_build(desc, stream=0, **args)

    assert call(dflv.ddtree_desc(1, 16, 151936, 9, 22)) == dflv.DFLV_ERR_UNSUPPORTED      # K > 8
    assert call(dflv.ddtree_desc(1, 65, 151936, 4, 22)) == dflv.DFLV_ERR_UNSUPPORTED      # D > 64
    assert call(dflv.ddtree_desc(1, 16, 151936, 4, 65)) == dflv.DFLV_ERR_UNSUPPORTED      # budget > 64
    assert call(dflv.ddtree_desc(1, 16, 151937, 4, 22)) == dflv.DFLV_ERR_UNSUPPORTED      # V not a multiple of 4
    assert call(dflv.ddtree_desc(0, 16, 151936, 4, 22)) == dflv.DFLV_ERR_INVALID_ARG
    assert call(dflv.ddtree_desc(1, 16, 151936, 4, 22, float("nan"))) == dflv.DFLV_ERR_INVALID_ARG
    assert call(dflv.ddtree_desc(1, 16, 151936, 4, 22, 6.0, 1)) == dflv.DFLV_ERR_INVALID_ARG   # flags
    ok = dflv.ddtree_desc(1, 16, 151936, 4, 22, 6.0)
    assert call(ok, draft_logits=None) == dflv.DFLV_ERR_INVALID_ARG
    assert call(ok, draft_logits=24) == dflv.DFLV_ERR_INVALID_ARG                        # misaligned
    assert call(ok, parent=18) == dflv.DFLV_ERR_INVALID_ARG


def test_structs_keep_the_tensors_they_point_to():
    # A factor or cache struct made from temporaries must keep them alive:
    # the library stores only their addresses, and a freed tensor's memory
    # would be handed to the next allocation while kernels still write it.
    import gc
    import weakref

    import torch

    u = torch.empty(8)
    ref = weakref.ref(u)
    f = dflv.gdn_factors(u, torch.empty(4), torch.empty(4, dtype=torch.int16))
    addr = u.data_ptr()
    del u
    gc.collect()
    assert ref() is not None and f.u == addr
    kq = torch.empty(16, dtype=torch.uint8)
    kref = weakref.ref(kq)
    c = dflv.kv_layer(kq, torch.empty(16, dtype=torch.uint8))
    del kq
    gc.collect()
    assert kref() is not None and c.kq == kref().data_ptr()
    del f, c
    gc.collect()
    assert ref() is None and kref() is None


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    # The product path has no fallback: without libdflv.so every entry point
    # raises instead of computing anything.
    monkeypatch.setattr(dflv, "_lib", None)
    monkeypatch.setattr(dflv, "LIB_PATH", str(tmp_path / "libdflv.so"))
    with pytest.raises(RuntimeError, match="not built"):
        dflv.load()
    with pytest.raises(RuntimeError, match="not built"):
        dflv.dflv_accept_greedy(1, 2, 4, 16, 16, 16, 16, 16, 16, 16, 16, 16)


def test_noalloc_scratch_size_matches_the_header():
    import re
    with open(dflv.HEADER) as f:
        m = re.search(r"#define DFLV_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", f.read())
    assert m and int(m.group(1)) << int(m.group(2)) == dflv.DFLV_NOALLOC_SCRATCH_BYTES
