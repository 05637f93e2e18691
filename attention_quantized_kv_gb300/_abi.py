"""ctypes binding of libkvq's C ABI (include/kvq.h), names unchanged.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  When libkvq.so is missing the import fails loudly; there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libkvq.so")

KVQ_F16, KVQ_Q8_0, KVQ_Q4_0, KVQ_TURBO4 = 0, 1, 2, 3
KVQ_OK, KVQ_EINVAL, KVQ_EUNSUPPORTED, KVQ_ECAPACITY, KVQ_EALIGN, KVQ_EWORKSPACE, KVQ_ECUDA = range(7)
KVQ_DEVERR_CAPACITY, KVQ_DEVERR_MAXLEN, KVQ_DEVERR_TIMEOUT, KVQ_DEVERR_SEQLEN = 1, 2, 4, 8
KVQ_DEVERR_PAGE, KVQ_DEVERR_EVICT = 16, 32

# Every function the header declares (checked by the tests against include/kvq.h).
EXPORTS = ("kvq_status_str", "kvq_row_bytes", "kvq_cache_bytes", "kvq_pool_bytes",
           "kv_append_quantize",
           "attn_decode_workspace", "attn_decode", "attn_decode_append", "attn_decode_noalloc",
           "attn_prefill_workspace", "attn_prefill_chunk", "kv_requantize", "kvq_aggregate_bpv",
           "kvq_ladder_next", "kv_probe_scores", "kv_evict_select", "kv_compact")


class kvq_layer(ctypes.Structure):
    _fields_ = [
        ("n_seqs", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32),
        ("n_q_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("capacity", ctypes.c_int32),
        ("codec_k", ctypes.c_int32),
        ("codec_v", ctypes.c_int32),
        ("pages_per_seq", ctypes.c_int32),
        ("k_cache", ctypes.c_void_p),
        ("v_cache", ctypes.c_void_p),
        ("seq_lens", ctypes.c_void_p),
        ("err", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("n_pages", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


_lib = None


def load(path: str | None = None):
    """Load libkvq.so (building nothing); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise ImportError(f"libkvq.so not built at {path}: run __graft_entry__.build() "
                          "(attention_quantized_kv_gb300.build.build()) first")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    L = ctypes.POINTER(kvq_layer)
    i32, i64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    sz = ctypes.POINTER(ctypes.c_size_t)
    sig = {
        "kvq_status_str": (ctypes.c_char_p, [ctypes.c_int]),
        "kvq_row_bytes": (i64, [ctypes.c_int, i32]),
        "kvq_cache_bytes": (i64, [ctypes.c_int, i32, i32, i32, i32]),
        "kvq_pool_bytes": (i64, [ctypes.c_int, i32, i32, i32]),
        "kv_append_quantize": (ctypes.c_int, [L, P, P, P, i32, i32, P]),
        "attn_decode_workspace": (ctypes.c_int, [L, i32, sz]),
        "attn_decode": (ctypes.c_int, [L, P, f32, P, P, i32, P, ctypes.c_size_t, P]),
        "attn_decode_append": (ctypes.c_int, [L, P, P, P, f32, P, P, i32, P, ctypes.c_size_t,
                                              P]),
        "attn_decode_noalloc": (ctypes.c_int, [L, P, f32, P, P, i32, P]),
        "attn_prefill_workspace": (ctypes.c_int, [L, i32, i32, sz]),
        "attn_prefill_chunk": (ctypes.c_int, [L, i32, i32, i32, P, f32, P, P, P,
                                              ctypes.c_size_t, P]),
        "kv_requantize": (ctypes.c_int, [L, i32, i32, P, P]),
        "kvq_aggregate_bpv": (ctypes.c_double, [ctypes.POINTER(i32), i32]),
        "kvq_ladder_next": (ctypes.c_int, [ctypes.POINTER(i32), i32, ctypes.POINTER(i32), i32,
                                           ctypes.c_double, ctypes.POINTER(i32),
                                           ctypes.POINTER(i32)]),
        "kv_probe_scores": (ctypes.c_int, [L, P, f32, P, f32, P, P]),
        "kv_evict_select": (ctypes.c_int, [L, P, i32, i32, i32, P, P, P]),
        "kv_compact": (ctypes.c_int, [L, P, P, i32, P, P, P, P, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
