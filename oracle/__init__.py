"""CPU oracle for the DDTree tree-verify step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product (the CUDA library and its binding)
never does, and this package never imports the product.

The arithmetic lives in ``oracle.c`` (plain C, fp64; see ``oracle.h`` for what
each function computes and which passage of the pages it follows).  This
module compiles it with gcc and wraps each entry point for numpy arrays laid
out exactly as the library's C ABI lays them out.  The draft-tree
construction is plain numpy / Python in ``ddtree.py`` (small, sequential).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .ddtree import build_ddtree, draft_topk  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_SOURCES = [os.path.join(_HERE, "oracle.c"), os.path.join(_HERE, "oracle.h")]
_lock = threading.Lock()
_lib = None

KV_Q8_0, KV_Q4_0, KV_F32, KV_Q8_0_Q4_0, KV_Q4_0_Q8_0, KV_TQ3_0 = 0, 1, 2, 3, 4, 5
OK, ERR_ARG, ERR_TOPOLOGY, ERR_CAPACITY = 0, 1, 2, 4


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_build/liboracle.so`` (gcc, -O2, no FMA
    contraction so x86 and Arm hosts round identically)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    newest_src = max(os.path.getmtime(p) for p in _SOURCES)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest_src:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-ffp-contract=off", "-fPIC",
               "-shared", _SOURCES[0], "-o", tmp, "-lm"]
        # OpenMP over independent (sequence, head) work when the compiler has
        # it; the results are the same either way
        r = subprocess.run(cmd[:1] + ["-fopenmp"] + cmd[1:], capture_output=True, text=True)
        if r.returncode != 0:
            subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_to_double.restype = ctypes.c_double
            lib.orc_half_to_float.argtypes = [ctypes.c_uint16]
            lib.orc_half_to_float.restype = ctypes.c_float
            lib.orc_float_to_half_rn.argtypes = [ctypes.c_float]
            lib.orc_float_to_half_rn.restype = ctypes.c_uint16
            lib.orc_tree_topology.argtypes = [I, P, P, P]
            lib.orc_gdn_step.argtypes = [I, I, P, P, P, P, ctypes.c_double, ctypes.c_double, P, P]
            lib.orc_gdn_step.restype = None
            lib.orc_tree_gdn_verify.argtypes = [I] * 6 + [P] * 10
            lib.orc_tree_gdn_verify_bruteforce.argtypes = [I] * 6 + [P] * 9
            lib.orc_gdn_commit.argtypes = [I] * 6 + [P] * 8
            for f in ("orc_quantize_q8_0", "orc_quantize_q4_0", "orc_quantize_tq3_0"):
                getattr(lib, f).argtypes = [P, P, P]
                getattr(lib, f).restype = None
            for f in ("orc_dequantize_q8_0", "orc_dequantize_q4_0", "orc_dequantize_tq3_0"):
                getattr(lib, f).argtypes = [P, ctypes.c_uint16, P]
                getattr(lib, f).restype = None
            lib.orc_fwht_f32.argtypes = [I, P]
            lib.orc_fwht_f32.restype = None
            lib.orc_tree_attn_verify.argtypes = [I] * 8 + [ctypes.c_double] + [P] * 11 + [P, I]
            lib.orc_accept_greedy.argtypes = [I, I, I] + [P] * 8
            lib.orc_kv_commit.argtypes = [I] * 6 + [P] * 7
            lib.orc_tree_conv_verify.argtypes = [I] * 4 + [P] * 6
            lib.orc_set_threads.argtypes = [I]
            lib.orc_set_threads.restype = I
            lib.orc_conv_commit.argtypes = [I] * 4 + [P] * 4
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    """C-contiguous array of the given dtype (a no-op for conforming input)."""
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != OK:
        raise OracleError(rc, f"{what} returned status {rc}")


class OracleError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(msg)
        self.code = code


# ---------------------------------------------------------------- scalars
def bf16_to_double(bits: int) -> float:
    return _load().orc_bf16_to_double(int(bits))


def half_to_float(bits: int) -> float:
    return _load().orc_half_to_float(int(bits))


def float_to_half_rn(x: float) -> int:
    return int(_load().orc_float_to_half_rn(float(x)))


# ---------------------------------------------------------------- topology
def tree_topology(parent):
    parent = _c(parent, np.int32)
    n = parent.shape[0]
    depth = np.zeros(max(n, 1), np.int32)
    anc = np.zeros(max(n, 1), np.uint64)
    rc = _load().orc_tree_topology(n, _p(parent), _p(depth), _p(anc))
    _check(rc, "tree_topology")
    return depth[:n], anc[:n]


# ---------------------------------------------------------------- GDN
def gdn_step(S, q, k, v, beta, alpha):
    """One gated delta-rule step in fp64; returns (S_out, o)."""
    S = _c(S, np.float64)
    dv, dk = S.shape
    q, k, v = _c(q, np.float64), _c(k, np.float64), _c(v, np.float64)
    S_out = np.empty_like(S)
    o = np.empty(dv, np.float64)
    _load().orc_gdn_step(dv, dk, _p(S), _p(q), _p(k), _p(v), float(beta), float(alpha),
                         _p(S_out), _p(o))
    return S_out, o


def tree_gdn_verify(parent, n_nodes, q, k, v, beta, log_alpha, state, want_states=False):
    """Tree verify of one gated-DeltaNet layer.

    q, k: [B][N][Hk][dk] uint16 (bf16 bits); v: [B][N][Hv][dv] uint16;
    beta, log_alpha: [B][N][Hv] float32; state: [B][Hv][dv][dk] float32.
    Returns out [B][N][Hv][dv] float32 (and node states fp64 if asked)."""
    parent, n_nodes = _c(parent, np.int32), _c(n_nodes, np.int32)
    q, k, v = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    beta, log_alpha, state = _c(beta, np.float32), _c(log_alpha, np.float32), _c(state, np.float32)
    B, N, Hk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    out = np.zeros((B, N, Hv, dv), np.float32)
    ns = np.zeros((B, N, Hv, dv, dk), np.float64) if want_states else None
    rc = _load().orc_tree_gdn_verify(B, N, Hk, Hv, dk, dv, _p(parent), _p(n_nodes), _p(q), _p(k),
                                     _p(v), _p(beta), _p(log_alpha), _p(state), _p(out), _p(ns))
    _check(rc, "tree_gdn_verify")
    return (out, ns) if want_states else out


def tree_gdn_verify_bruteforce(parent, n_nodes, q, k, v, beta, log_alpha, state):
    parent, n_nodes = _c(parent, np.int32), _c(n_nodes, np.int32)
    q, k, v = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    beta, log_alpha, state = _c(beta, np.float32), _c(log_alpha, np.float32), _c(state, np.float32)
    B, N, Hk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    out = np.zeros((B, N, Hv, dv), np.float32)
    rc = _load().orc_tree_gdn_verify_bruteforce(B, N, Hk, Hv, dk, dv, _p(parent), _p(n_nodes),
                                                _p(q), _p(k), _p(v), _p(beta), _p(log_alpha),
                                                _p(state), _p(out))
    _check(rc, "tree_gdn_verify_bruteforce")
    return out


def gdn_commit(q, k, v, beta, log_alpha, path, path_len, state):
    """Returns the committed state (a new float32 array): the accepted path
    decoded from ``state``."""
    q, k, v = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    beta, log_alpha = _c(beta, np.float32), _c(log_alpha, np.float32)
    path, path_len = _c(path, np.int32), _c(path_len, np.int32)
    st = np.array(state, dtype=np.float32, order="C", copy=True)
    B, N, Hk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    rc = _load().orc_gdn_commit(B, N, Hk, Hv, dk, dv, _p(q), _p(k), _p(v), _p(beta),
                                _p(log_alpha), _p(path), _p(path_len), _p(st))
    _check(rc, "gdn_commit")
    return st


# ---------------------------------------------------------------- quantisation
def quantize_q8_0(x):
    x = _c(x, np.float32)
    assert x.shape == (32,)
    qs = np.zeros(32, np.int8)
    d = np.zeros(1, np.uint16)
    _load().orc_quantize_q8_0(_p(x), _p(qs), _p(d))
    return qs, int(d[0])


def quantize_q4_0(x):
    x = _c(x, np.float32)
    assert x.shape == (32,)
    nib = np.zeros(16, np.uint8)
    d = np.zeros(1, np.uint16)
    _load().orc_quantize_q4_0(_p(x), _p(nib), _p(d))
    return nib, int(d[0])


def dequantize_q8_0(qs, d16):
    qs = _c(qs, np.int8)
    x = np.zeros(32, np.float64)
    _load().orc_dequantize_q8_0(_p(qs), int(d16), _p(x))
    return x


def dequantize_q4_0(nib, d16):
    nib = _c(nib, np.uint8)
    x = np.zeros(32, np.float64)
    _load().orc_dequantize_q4_0(_p(nib), int(d16), _p(x))
    return x


def quantize_tq3_0(x):
    """32 fp32 values -> (12 code bytes, fp16 scale bits)."""
    x = _c(x, np.float32)
    assert x.shape == (32,)
    codes = np.zeros(12, np.uint8)
    d = np.zeros(1, np.uint16)
    _load().orc_quantize_tq3_0(_p(x), _p(codes), _p(d))
    return codes, int(d[0])


def dequantize_tq3_0(codes, d16):
    codes = _c(codes, np.uint8)
    assert codes.shape == (12,)
    x = np.zeros(32, np.float64)
    _load().orc_dequantize_tq3_0(_p(codes), int(d16), _p(x))
    return x


def fwht(x):
    """The TQ3_0 rotation of each row of x (fp32, last axis a power of two),
    as the oracle's cache writes apply it."""
    y = np.array(x, dtype=np.float32, order="C", copy=True)
    n = y.shape[-1]
    for row in y.reshape(-1, n):
        _load().orc_fwht_f32(n, row.ctypes.data_as(ctypes.c_void_p))
    return y


# ---------------------------------------------------------------- attention
def tree_attn_verify(parent, n_nodes, n_past, q, k_new, v_new, cache, window, kv_type,
                     scale=None, rows=None):
    """Tree verify of one attention layer.

    ``cache`` is a dict with 'kq', 'vq' (quant planes) and 'ks', 'vs' (fp16
    scale planes, None for f32); it is MODIFIED in place (tree slots written).
    Returns out [B][N][Hq][D] float32 (rows not requested stay zero)."""
    parent, n_nodes, n_past = _c(parent, np.int32), _c(n_nodes, np.int32), _c(n_past, np.int32)
    q, k_new, v_new = _c(q, np.uint16), _c(k_new, np.uint16), _c(v_new, np.uint16)
    B, N, Hq, D = q.shape
    Hkv = k_new.shape[2]
    kq, vq = cache["kq"], cache["vq"]
    ks, vs = cache.get("ks"), cache.get("vs")
    for a in (kq, vq, ks, vs):
        assert a is None or a.flags["C_CONTIGUOUS"]
    cap = kq.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.zeros((B, N, Hq, D), np.float32)
    rows_arr = None if rows is None else _c(rows, np.int32)
    rc = _load().orc_tree_attn_verify(B, N, Hq, Hkv, D, cap, int(window), int(kv_type),
                                      float(scale), _p(parent), _p(n_nodes), _p(n_past), _p(q),
                                      _p(k_new), _p(v_new), _p(kq), _p(vq), _p(ks), _p(vs),
                                      _p(out), _p(rows_arr),
                                      0 if rows_arr is None else rows_arr.shape[0])
    _check(rc, "tree_attn_verify")
    return out


# ---------------------------------------------------------------- acceptance
def accept_greedy(logits, tokens, parent, n_nodes):
    """Returns (path [B][N], path_len [B], next_token [B], best [B][N])."""
    logits, tokens = _c(logits, np.float32), _c(tokens, np.int32)
    parent, n_nodes = _c(parent, np.int32), _c(n_nodes, np.int32)
    B, N, V = logits.shape
    path = np.full((B, N), -1, np.int32)
    path_len = np.zeros(B, np.int32)
    next_token = np.zeros(B, np.int32)
    best = np.full((B, N), -1, np.int32)
    rc = _load().orc_accept_greedy(B, N, V, _p(logits), _p(tokens), _p(parent), _p(n_nodes),
                                   _p(path), _p(path_len), _p(next_token), _p(best))
    _check(rc, "accept_greedy")
    return path, path_len, next_token, best


# ---------------------------------------------------------------- KV commit
def kv_commit(cache, kv_type, path, path_len, n_past):
    """Compacts the accepted path's slots in place (cache dict as above)."""
    path, path_len, n_past = _c(path, np.int32), _c(path_len, np.int32), _c(n_past, np.int32)
    B, N = path.shape
    kq = cache["kq"]
    Hkv, cap = kq.shape[1], kq.shape[2]
    D = (kq.shape[3] * 8 // 3 if kv_type == KV_TQ3_0
         else kq.shape[3] * (2 if kv_type in (KV_Q4_0, KV_Q4_0_Q8_0) else 1))
    rc = _load().orc_kv_commit(B, N, Hkv, D, cap, int(kv_type), _p(path), _p(path_len),
                               _p(n_past), _p(cache["kq"]), _p(cache["vq"]),
                               _p(cache.get("ks")), _p(cache.get("vs")))
    _check(rc, "kv_commit")


# ---------------------------------------------------------------- short convolution
def tree_conv_verify(parent, n_nodes, x, state, w):
    """x [B][N][C] bf16 bits, state [B][K-1][C] bf16 bits, w [C][K] f32 ->
    out [B][N][C] f32: each node's window of K inputs along its parent chain,
    continued into the conv state before the root."""
    parent, n_nodes = _c(parent, np.int32), _c(n_nodes, np.int32)
    x, state, w = _c(x, np.uint16), _c(state, np.uint16), _c(w, np.float32)
    B, N, C = x.shape
    K = w.shape[1]
    assert state.shape == (B, K - 1, C)
    out = np.zeros((B, N, C), np.float32)
    rc = _load().orc_tree_conv_verify(B, N, C, K, _p(parent), _p(n_nodes), _p(x), _p(state), _p(w), _p(out))
    _check(rc, "tree_conv_verify")
    return out


def conv_commit(x, path, path_len, state):
    """Returns the committed conv state (a new array): the last K-1 entries
    of [state ; x of the accepted path]."""
    x, path, path_len = _c(x, np.uint16), _c(path, np.int32), _c(path_len, np.int32)
    st = np.array(state, dtype=np.uint16, order="C", copy=True)
    B, N, C = x.shape
    K = st.shape[1] + 1
    rc = _load().orc_conv_commit(B, N, C, K, _p(x), _p(path), _p(path_len), _p(st))
    _check(rc, "conv_commit")
    return st


def set_threads(n: int) -> int:
    """Threads for the oracle's parallel loops (n > 0); returns the count in
    force (1 without OpenMP).  Results do not depend on it."""
    return int(_load().orc_set_threads(int(n)))
