"""ctypes binding of libdflv (include/dflv.h) -- argument marshalling only.

Every function keeps the C name and argument order.  Tensor arguments are
torch CUDA tensors (their ``data_ptr()`` is passed) or plain integers
(device addresses); ``stream`` defaults to torch's current stream.  Each call
returns the library's status code; ``check()`` turns a non-zero code into an
exception.  Every step of the tree-verify path runs in the CUDA library: this
module computes nothing, and there is no CPU fallback -- if the library is
not built, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libdflv.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "dflv.h")

DFLV_OK, DFLV_ERR_INVALID_ARG, DFLV_ERR_TOPOLOGY, DFLV_ERR_UNSUPPORTED, DFLV_ERR_CAPACITY, DFLV_ERR_CUDA = range(6)
DFLV_DEV_TOPOLOGY, DFLV_DEV_CAPACITY, DFLV_DEV_PATH, DFLV_DEV_TIMEOUT = 1, 2, 4, 8
DFLV_KV_Q8_0, DFLV_KV_Q4_0, DFLV_KV_F32, DFLV_KV_Q8_0_Q4_0, DFLV_KV_Q4_0_Q8_0, DFLV_KV_TQ3_0 = 0, 1, 2, 3, 4, 5
DFLV_FLAG_EARLY_PREFETCH = 1
DFLV_MAX_COMMIT_GDN_LAYERS, DFLV_MAX_COMMIT_ATTN_LAYERS = 128, 64
DFLV_MAX_CONV_LAYERS = 128

_c_i32 = ctypes.c_int32
_vp = ctypes.c_void_p


class dflv_gdn_desc(ctypes.Structure):
    _fields_ = [("B", _c_i32), ("N_max", _c_i32), ("Hk", _c_i32), ("Hv", _c_i32), ("dk", _c_i32), ("dv", _c_i32),
                ("flags", ctypes.c_uint32)]


class dflv_gdn_factors(ctypes.Structure):
    _fields_ = [("u", _vp), ("g", _vp), ("kcopy", _vp)]


class dflv_attn_desc(ctypes.Structure):
    _fields_ = [("B", _c_i32), ("N_max", _c_i32), ("Hq", _c_i32), ("Hkv", _c_i32), ("D", _c_i32),
                ("cap", _c_i32), ("window", _c_i32), ("type", ctypes.c_int), ("scale", ctypes.c_float),
                ("flags", ctypes.c_uint32)]


class dflv_kv_layer(ctypes.Structure):
    _fields_ = [("kq", _vp), ("vq", _vp), ("ks", _vp), ("vs", _vp)]


class dflv_conv_desc(ctypes.Structure):
    _fields_ = [("B", _c_i32), ("N_max", _c_i32), ("C", _c_i32), ("K", _c_i32), ("flags", ctypes.c_uint32)]


class dflv_ddtree_desc(ctypes.Structure):
    _fields_ = [("B", _c_i32), ("D", _c_i32), ("V", _c_i32), ("K", _c_i32), ("budget", _c_i32),
                ("tau", ctypes.c_float), ("flags", ctypes.c_uint32)]


class DflvError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (status {code})")


_lib = None


def load():
    """Loads libdflv.so; raises if it has not been built (no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libdflv.so is not built ({LIB_PATH} missing); run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P = _vp
    S = ctypes.c_size_t
    lib.dflv_tree_gdn_verify.argtypes = [ctypes.POINTER(dflv_gdn_desc)] + [P] * 9 + \
        [ctypes.POINTER(dflv_gdn_factors), P, P, S, P]
    lib.dflv_tree_gdn_verify_pending.argtypes = [ctypes.POINTER(dflv_gdn_desc)] + [P] * 8 + \
        [ctypes.POINTER(dflv_gdn_factors), P, P, P, ctypes.POINTER(dflv_gdn_factors), P, P, S, P]
    lib.dflv_tree_attn_verify.argtypes = [ctypes.POINTER(dflv_attn_desc)] + [P] * 6 + \
        [ctypes.POINTER(dflv_kv_layer), P, P, P, S, P]
    lib.dflv_tree_attn_verify_noalloc.argtypes = [ctypes.POINTER(dflv_attn_desc)] + [P] * 6 + \
        [ctypes.POINTER(dflv_kv_layer), P, P, P]
    lib.dflv_accept_greedy.argtypes = [_c_i32, _c_i32, _c_i32] + [P] * 10
    lib.dflv_commit_rollback.argtypes = [ctypes.POINTER(dflv_gdn_desc), _c_i32, P, ctypes.POINTER(dflv_gdn_factors),
                                         ctypes.POINTER(dflv_attn_desc), _c_i32, ctypes.POINTER(dflv_kv_layer),
                                         P, P, P, P, P]
    lib.dflv_tree_conv_verify.argtypes = [ctypes.POINTER(dflv_conv_desc)] + [P] * 7 + [P]
    lib.dflv_conv_commit.argtypes = [ctypes.POINTER(dflv_conv_desc), _c_i32, P, P, P, P, P, P]
    lib.dflv_ddtree_build.argtypes = [ctypes.POINTER(dflv_ddtree_desc)] + [P] * 10
    lib.dflv_gdn_workspace_size.argtypes = [ctypes.POINTER(dflv_gdn_desc)]
    lib.dflv_gdn_workspace_size.restype = S
    lib.dflv_attn_workspace_size.argtypes = [ctypes.POINTER(dflv_attn_desc)]
    lib.dflv_attn_workspace_size.restype = S
    lib.dflv_status_string.argtypes = [ctypes.c_int]
    lib.dflv_status_string.restype = ctypes.c_char_p
    for f in ("dflv_tree_gdn_verify", "dflv_tree_gdn_verify_pending", "dflv_tree_attn_verify",
              "dflv_tree_attn_verify_noalloc", "dflv_accept_greedy",
              "dflv_commit_rollback", "dflv_tree_conv_verify", "dflv_conv_commit", "dflv_ddtree_build"):
        getattr(lib, f).restype = ctypes.c_int
    _lib = lib
    return lib


def header_symbols():
    """Names of the functions include/dflv.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(dflv_\w+)\s*\(", text, flags=re.M)))


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def status_string(code: int) -> str:
    return load().dflv_status_string(int(code)).decode()


def check(code: int, where: str = "dflv"):
    if code != DFLV_OK:
        raise DflvError(code, where)
    return code


# ---------------------------------------------------------------- structs from tensors
def gdn_desc(B, N_max, Hk, Hv, dk, dv, flags=0):
    return dflv_gdn_desc(B, N_max, Hk, Hv, dk, dv, flags)


def gdn_factors(u, g, kcopy):
    """The factor buffers' pointers.  The struct holds references to the
    tensors it was made from, so that buffers passed as temporaries stay
    allocated for as long as the struct is in use."""
    f = dflv_gdn_factors(_ptr(u), _ptr(g), _ptr(kcopy))
    f._tensors = (u, g, kcopy)
    return f


def attn_desc(B, N_max, Hq, Hkv, D, cap, window, kv_type, scale, flags=0):
    return dflv_attn_desc(B, N_max, Hq, Hkv, D, cap, window, kv_type, scale, flags)


def kv_layer(kq, vq, ks=None, vs=None):
    """One layer's cache planes; holds references to the tensors, as
    gdn_factors does."""
    c = dflv_kv_layer(_ptr(kq), _ptr(vq), _ptr(ks), _ptr(vs))
    c._tensors = (kq, vq, ks, vs)
    return c


# ---------------------------------------------------------------- the C ABI
def dflv_tree_gdn_verify(desc, parent, n_nodes, q, k, v, beta, log_alpha, state, out, factors,
                         status_dev, workspace=None, ws_bytes=0, stream=None) -> int:
    return load().dflv_tree_gdn_verify(
        ctypes.byref(desc), _ptr(parent), _ptr(n_nodes), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
        _ptr(log_alpha), _ptr(state), _ptr(out), ctypes.byref(factors), _ptr(status_dev),
        _ptr(workspace), ws_bytes, _stream(stream))


def dflv_tree_gdn_verify_pending(desc, parent, n_nodes, q, k, v, beta, log_alpha, state, pending, pending_path,
                                 pending_len, out, factors, status_dev, workspace=None, ws_bytes=0,
                                 stream=None) -> int:
    return load().dflv_tree_gdn_verify_pending(
        ctypes.byref(desc), _ptr(parent), _ptr(n_nodes), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
        _ptr(log_alpha), _ptr(state), ctypes.byref(pending), _ptr(pending_path), _ptr(pending_len), _ptr(out),
        ctypes.byref(factors), _ptr(status_dev), _ptr(workspace), ws_bytes, _stream(stream))


def dflv_tree_attn_verify(desc, parent, n_nodes, n_past, q, k_new, v_new, cache, out, status_dev,
                          workspace=None, ws_bytes=0, stream=None) -> int:
    return load().dflv_tree_attn_verify(
        ctypes.byref(desc), _ptr(parent), _ptr(n_nodes), _ptr(n_past), _ptr(q), _ptr(k_new),
        _ptr(v_new), ctypes.byref(cache), _ptr(out), _ptr(status_dev), _ptr(workspace), ws_bytes,
        _stream(stream))


def dflv_tree_attn_verify_noalloc(desc, parent, n_nodes, n_past, q, k_new, v_new, cache, out, status_dev,
                                  stream=None) -> int:
    return load().dflv_tree_attn_verify_noalloc(
        ctypes.byref(desc), _ptr(parent), _ptr(n_nodes), _ptr(n_past), _ptr(q), _ptr(k_new),
        _ptr(v_new), ctypes.byref(cache), _ptr(out), _ptr(status_dev), _stream(stream))


DFLV_NOALLOC_SCRATCH_BYTES = 16 << 20


def dflv_accept_greedy(B, N_max, vocab, logits, tokens, parent, n_nodes, path, path_len, next_token,
                       best, status_dev, stream=None) -> int:
    return load().dflv_accept_greedy(B, N_max, vocab, _ptr(logits), _ptr(tokens), _ptr(parent),
                                     _ptr(n_nodes), _ptr(path), _ptr(path_len), _ptr(next_token),
                                     _ptr(best), _ptr(status_dev), _stream(stream))


def dflv_commit_rollback(gdn, n_gdn, states, factors, attn, n_attn, caches, path, path_len, n_past,
                         status_dev, stream=None) -> int:
    """``states``: sequence of state tensors (or addresses), ``factors``:
    sequence of dflv_gdn_factors, ``caches``: sequence of dflv_kv_layer."""
    st = (ctypes.c_void_p * max(1, n_gdn))(*[_ptr(s) for s in states][:n_gdn])
    fa = (dflv_gdn_factors * max(1, n_gdn))(*list(factors)[:n_gdn])
    ca = (dflv_kv_layer * max(1, n_attn))(*list(caches)[:n_attn])
    return load().dflv_commit_rollback(
        ctypes.byref(gdn) if gdn is not None else None, n_gdn, ctypes.cast(st, ctypes.c_void_p), fa,
        ctypes.byref(attn) if attn is not None else None, n_attn, ca, _ptr(path), _ptr(path_len),
        _ptr(n_past), _ptr(status_dev), _stream(stream))


def conv_desc(B, N_max, C, K, flags=0):
    return dflv_conv_desc(B, N_max, C, K, flags)


def dflv_tree_conv_verify(desc, parent, n_nodes, x, conv_state, weight, out, status_dev, stream=None) -> int:
    return load().dflv_tree_conv_verify(ctypes.byref(desc), _ptr(parent), _ptr(n_nodes), _ptr(x), _ptr(conv_state),
                                        _ptr(weight), _ptr(out), _ptr(status_dev), _stream(stream))


def dflv_conv_commit(desc, n_layers, states, xs, path, path_len, status_dev, stream=None) -> int:
    """``states``, ``xs``: sequences of tensors (or addresses), one per layer."""
    st = (ctypes.c_void_p * max(1, n_layers))(*[_ptr(s) for s in states][:n_layers])
    xa = (ctypes.c_void_p * max(1, n_layers))(*[_ptr(x) for x in xs][:n_layers])
    return load().dflv_conv_commit(ctypes.byref(desc), n_layers, ctypes.cast(st, ctypes.c_void_p),
                                   ctypes.cast(xa, ctypes.c_void_p), _ptr(path), _ptr(path_len), _ptr(status_dev),
                                   _stream(stream))


def ddtree_desc(B, D, V, K, budget, tau=-1.0, flags=0):
    """tau < 0 (default): no pruning."""
    return dflv_ddtree_desc(B, D, V, K, budget, tau, flags)


def dflv_ddtree_build(desc, draft_logits, root_token, topk_tok, topk_logp, parent, tokens, n_nodes, score,
                      status_dev, stream=None) -> int:
    return load().dflv_ddtree_build(ctypes.byref(desc), _ptr(draft_logits), _ptr(root_token), _ptr(topk_tok),
                                    _ptr(topk_logp), _ptr(parent), _ptr(tokens), _ptr(n_nodes), _ptr(score),
                                    _ptr(status_dev), _stream(stream))


def dflv_gdn_workspace_size(desc) -> int:
    return int(load().dflv_gdn_workspace_size(ctypes.byref(desc)))


def dflv_attn_workspace_size(desc) -> int:
    return int(load().dflv_attn_workspace_size(ctypes.byref(desc)))


def dflv_status_string(code: int) -> str:
    return status_string(code)
