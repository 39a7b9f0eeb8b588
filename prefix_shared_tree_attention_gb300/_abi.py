"""ctypes declarations mirroring include/tpa.h (argument marshalling only)."""
from __future__ import annotations

import ctypes as C
import os

from . import build as _build

TPA_OK = 0
STATUS = {
    0: "TPA_OK", -1: "TPA_ERR_INVALID_ARG", -2: "TPA_ERR_EMPTY_SEQUENCE", -3: "TPA_ERR_SEQ_TOO_LONG",
    -4: "TPA_ERR_NO_MEMORY", -5: "TPA_ERR_CUDA", -6: "TPA_ERR_DEVICE_TIMEOUT",
    -7: "TPA_ERR_UNSUPPORTED_DEVICE", -8: "TPA_ERR_BUFFER_TOO_SMALL",
}
BLOCK_SIZE = 128
LOGITS_COMPACT, LOGITS_PADDED = 0, 1
GRAD_F32, GRAD_BF16 = 0, 1
BALANCE_FFD, BALANCE_KK = 0, 1
MASK_U8, MASK_BITS = 0, 1

_i32p = C.POINTER(C.c_int32)
_i64p = C.POINTER(C.c_int64)


class TreeInfo(C.Structure):
    _fields_ = [
        ("n_trees", C.c_int32), ("t_pad", C.c_int32), ("n_seqs", C.c_int32), ("max_nodes", C.c_int32),
        ("total_seq_tokens", C.c_int64), ("total_tree_tokens", C.c_int64), ("total_nodes", C.c_int64),
        ("ancestor_pairs", C.c_int64), ("tree_token_ratio", C.c_double), ("blob_bytes", C.c_uint64),
        ("max_token", C.c_int32), ("reserved_", C.c_int32),
    ]


class TreeView(C.Structure):
    _fields_ = [
        ("n_trees", C.c_int32), ("t_pad", C.c_int32), ("n_seqs", C.c_int32), ("max_nodes", C.c_int32),
        ("total_seq_tokens", C.c_int64), ("total_tree_tokens", C.c_int64),
        ("max_token", C.c_int32), ("reserved_", C.c_int32), ("ancestor_pairs", C.c_int64),
        ("tokens", C.c_void_p), ("subtree_end", C.c_void_p), ("parent", C.c_void_p), ("depth", C.c_void_p),
        ("node_id", C.c_void_p), ("child_off", C.c_void_p), ("child_pos", C.c_void_p),
        ("n_tokens", C.c_void_p), ("tok_base", C.c_void_p), ("node_info", C.c_void_p),
        ("n_nodes", C.c_void_p), ("seq_tree", C.c_void_p), ("seq_off", C.c_void_p), ("seq_pos", C.c_void_p),
    ]


class BlockMaskView(C.Structure):
    _fields_ = [
        ("n_trees", C.c_int32), ("n_blk", C.c_int32), ("cap", C.c_int32), ("pad_", C.c_int32),
        ("cls", C.c_void_p), ("q_ptr", C.c_void_p), ("q_idx", C.c_void_p),
        ("k_ptr", C.c_void_p), ("k_idx", C.c_void_p), ("qmask", C.c_void_p), ("sched", C.c_void_p),
        ("line_count", C.c_void_p),
    ]


class PackingMetrics(C.Structure):
    _fields_ = [
        ("n_groups", C.c_int32), ("pad_", C.c_int32), ("total", C.c_int64), ("max_load", C.c_int64),
        ("min_load", C.c_int64), ("spread", C.c_int64), ("wasted", C.c_int64), ("mean", C.c_double),
        ("std_dev", C.c_double), ("cv", C.c_double), ("imbalance_ratio", C.c_double),
        ("utilization", C.c_double),
    ]


# name -> (restype, argtypes); every symbol declared in include/tpa.h
PROTOTYPES = {
    "tpa_tree_pack": (C.c_int, [_i32p, _i64p, C.c_int32, C.c_int32, C.POINTER(C.c_void_p)]),
    "tpa_extract_sequences": (C.c_int, [_i32p, C.POINTER(C.c_uint8), C.c_int32, C.c_int32, _i32p, _i64p]),
    "tpa_tree_pack_padded": (C.c_int, [_i32p, C.POINTER(C.c_uint8), C.c_int32, C.c_int32, C.c_int32,
                                       C.POINTER(C.c_void_p)]),
    "tpa_tree_get_info": (C.c_int, [C.c_void_p, C.POINTER(TreeInfo)]),
    "tpa_tree_host_blob": (C.c_void_p, [C.c_void_p]),
    "tpa_tree_make_view": (C.c_int, [C.c_void_p, C.c_void_p, C.POINTER(TreeView)]),
    "tpa_tree_upload": (C.c_int, [C.c_void_p, C.c_void_p, C.c_uint64, C.c_void_p]),
    "tpa_tree_free": (None, [C.c_void_p]),
    "tpa_balance": (C.c_int, [_i64p, C.c_int32, C.c_int64, C.c_int32, C.c_int32, C.c_int32, _i32p, _i32p,
                              _i32p]),
    "tpa_packing_metrics": (C.c_int, [_i64p, C.c_int32, _i32p, C.c_int32, C.c_int64,
                                      C.POINTER(PackingMetrics)]),
    "tpa_dense_mask_bytes": (C.c_uint64, [C.c_int32, C.c_int32, C.c_int32]),
    "tpa_dense_mask": (C.c_int, [C.POINTER(TreeView), C.c_void_p, C.c_uint64, C.c_int32, C.c_int32, C.c_void_p]),
    "tpa_blockmask_bytes": (C.c_uint64, [C.c_int32, C.c_int32]),
    "tpa_blockmask_make_view": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.POINTER(BlockMaskView)]),
    "tpa_block_classify": (C.c_int, [C.POINTER(TreeView), C.POINTER(BlockMaskView), C.c_void_p]),
    "tpa_tree_attn_fwd": (C.c_int, [C.POINTER(TreeView), C.POINTER(BlockMaskView), C.c_void_p, C.c_void_p,
                                    C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_int32,
                                    C.c_float, C.c_void_p]),
    "tpa_tree_attn_bwd_workspace_bytes": (C.c_uint64, [C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                                       C.c_int32, C.c_int32]),
    "tpa_tree_attn_bwd": (C.c_int, [C.POINTER(TreeView), C.POINTER(BlockMaskView), C.c_void_p, C.c_void_p,
                                    C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                    C.c_void_p, C.c_void_p, C.c_uint64, C.c_int32, C.c_int32, C.c_int32,
                                    C.c_float, C.c_int32, C.c_void_p]),
    "tpa_tree_attn_bwd_noalloc": (C.c_int, [C.POINTER(TreeView), C.POINTER(BlockMaskView), C.c_void_p,
                                            C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                            C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32, C.c_int32,
                                            C.c_int32, C.c_float, C.c_int32, C.c_void_p]),
    "tpa_tree_logprobs_entropy": (C.c_int, [C.POINTER(TreeView), C.c_void_p, C.c_int64, C.c_int32, C.c_int32,
                                            C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]),
    "tpa_lm_head_workspace_bytes": (C.c_uint64, [C.c_int64, C.c_int32, C.c_int32, C.c_int32]),
    "tpa_lm_head_logprobs_entropy": (C.c_int, [C.POINTER(TreeView), C.c_void_p, C.c_void_p, C.c_int32, C.c_int32,
                                               C.c_void_p, C.c_uint64, C.c_void_p, C.c_void_p, C.c_void_p,
                                               C.c_void_p, C.c_void_p]),
    "tpa_sync_status": (C.c_int, [C.c_void_p]),
    "tpa_device_check": (C.c_int, []),
    "tpa_wait_probe": (C.c_int, [C.c_uint64, C.c_int32, C.c_void_p]),
    "tpa_status_string": (C.c_char_p, [C.c_int]),
    "tpa_version": (C.c_int, []),
}

_LIB = None
_DEBUG_LIB = None


class TpaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")
        self.status = status
        self.name = STATUS.get(status, str(status))


def lib(build_if_missing: bool = True) -> C.CDLL:
    """The loaded libtpa.so. Raises if it cannot be built or loaded: there is
    no fallback implementation."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = _build.LIB_PATH
    if build_if_missing and (_build.is_stale() or not os.path.exists(path)):
        _build.build()
    if not os.path.exists(path):
        raise ImportError(f"libtpa.so not found at {path}; run prefix_shared_tree_attention_gb300.build")
    L = C.CDLL(path)
    for name, (res, args) in PROTOTYPES.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _LIB = L
    return L


def debug_lib(build_if_missing: bool = True) -> C.CDLL:
    """The TPA_DEBUG variant, libtpa_debug.so: the same ABI, with kernels that
    check every metadata index they read from a tree view before using it as
    an address (a bad one makes tpa_sync_status return TPA_ERR_INVALID_ARG)."""
    global _DEBUG_LIB
    if _DEBUG_LIB is not None:
        return _DEBUG_LIB
    path = _build.DEBUG_LIB_PATH
    if build_if_missing and (_build.is_stale(path) or not os.path.exists(path)):
        _build.build(debug=True)
    if not os.path.exists(path):
        raise ImportError(f"libtpa_debug.so not found at {path}; run prefix_shared_tree_attention_gb300.build --debug")
    L = C.CDLL(path)
    for name, (res, args) in PROTOTYPES.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _DEBUG_LIB = L
    return L


def check(fn: str, status: int) -> None:
    if status != TPA_OK:
        raise TpaError(fn, status)
