"""ctypes declarations of the C ABI in include/dsa.h (marshalling only)."""
from __future__ import annotations

import ctypes as C
import os

from . import _build

c_i32 = C.c_int32
c_p = C.c_void_p


class PagedKV(C.Structure):
    _fields_ = [("k_cache", c_p), ("v_cache", c_p), ("idx_cache", c_p), ("block_table", c_p),
                ("context_lens", c_p), ("num_blocks", c_i32), ("block_size", c_i32),
                ("num_kv_heads", c_i32), ("head_dim", c_i32), ("idx_dim", c_i32),
                ("max_blocks_per_seq", c_i32), ("batch", c_i32), ("max_context_len", c_i32),
                ("kv_row_stride", c_i32)]


class QuerySet(C.Structure):
    _fields_ = [("mode", c_i32), ("n_q", c_i32), ("seq", c_i32), ("pos0", c_i32)]


PKV = C.POINTER(PagedKV)
PQS = C.POINTER(QuerySet)

# name -> (restype, argtypes), in the order of include/dsa.h
SIGNATURES = {
    "dsa_status_string": (C.c_char_p, [c_i32]),
    "dsa_last_error_message": (C.c_char_p, []),
    "dsa_abi_version": (c_i32, []),
    "dsa_check_device_status": (c_i32, [c_p, C.POINTER(c_i32)]),
    "dsa_kv_alloc_create": (c_i32, [c_i32, C.POINTER(c_p)]),
    "dsa_kv_alloc_blocks": (c_i32, [c_p, c_i32, C.POINTER(c_i32)]),
    "dsa_kv_free_blocks": (c_i32, [c_p, C.POINTER(c_i32), c_i32]),
    "dsa_kv_alloc_num_free": (c_i32, [c_p]),
    "dsa_kv_alloc_destroy": (None, [c_p]),
    "dsa_kv_bitmap_create": (c_i32, [c_i32, c_i32, c_i32, c_p]),
    "dsa_kv_bitmap_alloc": (c_i32, [c_p, c_i32, c_i32, c_i32, c_p]),
    "dsa_kv_bitmap_free": (c_i32, [c_p, c_i32, c_i32, c_p, c_i32]),
    "dsa_kv_bitmap_num_free": (c_i32, [c_p, c_i32, c_i32]),
    "dsa_kv_bitmap_words": (c_i32, [c_p, c_i32, c_i32, c_p, c_i32]),
    "dsa_kv_bitmap_destroy": (None, [c_p]),
    "dsa_kv_write": (c_i32, [PKV, c_p, c_i32, c_p, c_p, c_p, c_p]),
    "dsa_kv_write_heads": (c_i32, [PKV, c_p, c_i32, c_p, c_p, c_p, c_p]),
    "dsa_workspace_size": (C.c_size_t, [c_i32, PKV, PQS, c_i32, c_i32, c_i32]),
    "dsa_workspace_init": (c_i32, [c_p, C.c_size_t, c_p]),
    "dsa_index_scores": (c_i32, [PKV, PQS, c_p, c_i32, c_p, c_i32, c_p, C.c_size_t, c_p]),
    "dsa_topk_select": (c_i32, [PKV, PQS, c_p, c_i32, c_i32, c_i32, c_p, c_p, c_p, C.c_size_t, c_p]),
    "dsa_kv_gather": (c_i32, [PKV, PQS, c_p, c_p, c_i32, c_i32, c_p, c_p, c_p]),
    "dsa_copy_async": (c_i32, [c_p, c_p, C.c_size_t, c_p]),
    "dsa_sparse_attn_decode": (c_i32, [PKV, c_p, c_i32, c_p, c_p, c_i32, c_i32, C.c_float, c_p, c_i32,
                                       c_p, c_p, C.c_size_t, c_p]),
    "dsa_sparse_attn_prefill": (c_i32, [PKV, PQS, c_p, c_i32, c_p, c_p, c_i32, c_i32, C.c_float, c_p,
                                        c_i32, c_p, c_p, C.c_size_t, c_p]),
    "dsa_sparse_attn_prefill_split": (c_i32, [PKV, PQS, c_p, c_i32, c_p, c_p, c_i32, c_i32, C.c_float, c_i32,
                                              c_p, c_i32, c_p, c_p, C.c_size_t, c_p]),
    "dsa_prefill_dense_queries": (c_i32, [PKV, PQS, c_i32, c_i32, c_i32]),
    "dsa_prefill_attn_workspace_size": (C.c_size_t, [PKV, PQS, c_i32, c_i32, c_i32, c_i32]),
    "dsa_heads_workspace_size": (C.c_size_t, [PKV, c_i32, c_i32, c_i32]),
    "dsa_decode_step_heads": (c_i32, [PKV, c_p, c_p, c_p, c_i32, c_i32, c_i32, C.c_float, c_p, c_i32, c_p, c_p,
                                      c_p, c_i32, c_p, c_p, C.c_size_t, c_p]),
    "dsa_prefill_select": (c_i32, [PKV, PQS, c_p, c_i32, c_i32, c_p, c_p, c_p]),
    "dsa_window_workspace_size": (C.c_size_t, [PKV, c_i32, c_i32]),
    "dsa_window_attn_decode": (c_i32, [PKV, c_p, c_i32, c_i32, C.c_float, c_p, c_i32, c_p, c_p, C.c_size_t, c_p]),
    "dsa_window_attn_prefill": (c_i32, [PKV, PQS, c_p, c_i32, c_i32, C.c_float, c_p, c_i32, c_p, c_p]),
    "dsa_prefill_step": (c_i32, [PKV, c_p, c_p, c_p, c_i32, c_i32, c_i32, C.c_float, c_p, c_i32, c_p, c_p, c_p,
                                 c_i32, c_p, c_p, C.c_size_t, c_p]),
    "dsa_decode_step": (c_i32, [PKV, c_p, c_p, c_i32, c_i32, c_i32, C.c_float, c_p, c_i32, c_p, c_p,
                                c_p, c_i32, c_p, c_p, C.c_size_t, c_p]),
    "dsa_topk_select_decode_noalloc": (c_i32, [PKV, c_p, c_i32, c_i32, c_i32, c_p, c_p, c_p]),
}

_LIB = None


def load():
    """Load libdsa_gb300.so (building it if it is missing or stale).  There is
    no fallback: without the library every op raises."""
    global _LIB
    if _LIB is None:
        path = _build.ensure_built()
        if not os.path.exists(path):
            raise RuntimeError(f"DSA library missing at {path}")
        lib = C.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB
