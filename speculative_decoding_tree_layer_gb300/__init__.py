"""GB300-native tree verification for DDTree speculative decoding.

The compute lives in ``libdflv.so`` (hand-written CUDA for sm_103a, C ABI in
``include/dflv.h``); ``dflv`` is its ctypes binding with the same names.
"""
from . import dflv
from ._build import build
from .dflv import (DFLV_DEV_CAPACITY, DFLV_DEV_PATH, DFLV_DEV_TIMEOUT, DFLV_DEV_TOPOLOGY,
                   DFLV_ERR_CAPACITY, DFLV_ERR_CUDA, DFLV_ERR_INVALID_ARG, DFLV_ERR_TOPOLOGY,
                   DFLV_ERR_UNSUPPORTED, DFLV_FLAG_EARLY_PREFETCH, DFLV_KV_F32, DFLV_KV_Q4_0, DFLV_KV_Q8_0, DFLV_KV_Q8_0_Q4_0,
                   DFLV_KV_Q4_0_Q8_0, DFLV_KV_TQ3_0, DFLV_OK,
                   DflvError,
                   attn_desc, check, dflv_accept_greedy, dflv_attn_workspace_size, dflv_commit_rollback,
                   dflv_gdn_workspace_size, dflv_status_string, dflv_tree_attn_verify, dflv_tree_gdn_verify,
                   dflv_tree_gdn_verify_pending, dflv_tree_conv_verify, dflv_conv_commit, DFLV_MAX_CONV_LAYERS,
                   dflv_ddtree_build, conv_desc, ddtree_desc, gdn_desc, gdn_factors, kv_layer, load,
                   dflv_tree_attn_verify_noalloc, DFLV_NOALLOC_SCRATCH_BYTES)

__all__ = [n for n in dir() if n.startswith(("dflv", "DFLV", "Dflv")) or n in (
    "attn_desc", "conv_desc", "ddtree_desc", "gdn_desc", "gdn_factors", "kv_layer", "load", "build", "check")]
