"""CPU oracle for attention over a block-quantized KV cache.

TEST INFRASTRUCTURE ONLY.  This package wraps ``kvq_oracle.c`` (plain C99,
fp32 block codecs written from their formulas, fp64 softmax attention) with
ctypes and numpy.  It shares no code with the CUDA library and must never be
imported by it: only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` use it.

Every function follows a definition stated in ``kvq_oracle.c``'s header:
the f16 / q8_0 / q4_0 block formats and the rotated turbo4 row format (sizes
from the "Codecs" table of the buun-llama-cpp listing), the cache layout of
the library's public header, and the plain softmax-attention definition
evaluated in fp64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libkvq_oracle.so")

F16, Q8_0, Q4_0, TURBO4 = 0, 1, 2, 3
SIDE_K, SIDE_V = 0, 1
D = 128
UNIT_TOKENS = 16
ROW_BYTES = {F16: 256, Q8_0: 136, Q4_0: 72, TURBO4: 66}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libkvq_oracle.so`` with gcc."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        u8p = ctypes.POINTER(ctypes.c_uint8)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        i32p = ctypes.POINTER(ctypes.c_int32)
        i64p = ctypes.POINTER(ctypes.c_int64)
        lib.kvqo_half_to_float.argtypes = [ctypes.c_uint16]
        lib.kvqo_half_to_float.restype = ctypes.c_float
        lib.kvqo_float_to_half_rn.argtypes = [ctypes.c_float]
        lib.kvqo_float_to_half_rn.restype = ctypes.c_uint16
        lib.kvqo_encode_rows.argtypes = [ctypes.c_int, ctypes.c_int64, u16p, u8p]
        lib.kvqo_decode_rows.argtypes = [ctypes.c_int, ctypes.c_int64, u8p, f64p]
        lib.kvqo_unit_offset.argtypes = [ctypes.c_int] * 4
        lib.kvqo_append_side.argtypes = [ctypes.c_int, ctypes.c_int, u8p, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, i32p, i32p, ctypes.c_int,
                                         u16p]
        lib.kvqo_dequant_stream.argtypes = [ctypes.c_int, ctypes.c_int, u8p, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int64, f64p]
        lib.kvqo_attend_rows.argtypes = [ctypes.c_int, u16p, ctypes.c_int64, f64p, f64p, i64p,
                                         ctypes.c_double, f64p, f64p]
        lib.kvqo_decode_layer.argtypes = [ctypes.c_int, ctypes.c_int, u8p, u8p, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_int, i32p, u16p,
                                          ctypes.c_double, u8p, f64p, f64p]
        lib.kvqo_prefill_chunk.argtypes = [ctypes.c_int, ctypes.c_int, u8p, u8p, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int64, ctypes.c_int, u16p, ctypes.c_double,
                                           u8p, f64p, f64p]
        lib.kvqo_requantize_side.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, u8p, u8p,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int, i32p]
        ip = ctypes.POINTER(ctypes.c_int)
        lib.kvqo_bits_per_value.argtypes = [ctypes.c_int]
        lib.kvqo_bits_per_value.restype = ctypes.c_double
        lib.kvqo_aggregate_bpv.argtypes = [ip, ctypes.c_int]
        lib.kvqo_aggregate_bpv.restype = ctypes.c_double
        lib.kvqo_ladder_next.argtypes = [ip, ctypes.c_int, ip, ctypes.c_int, ctypes.c_double,
                                         ip, ip]
        lib.kvqo_paged_unit.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                        i32p, ctypes.c_int, ctypes.c_int]
        lib.kvqo_paged_unit.restype = ctypes.c_int64
        lib.kvqo_page_move.argtypes = [ctypes.c_int, u8p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       i32p, ctypes.c_int, u8p, ctypes.c_int, ctypes.c_int]
        lib.kvqo_probe_mass.argtypes = [ctypes.c_int, u8p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, i32p, u16p, ctypes.c_double, f64p]
        f32p = ctypes.POINTER(ctypes.c_float)
        lib.kvqo_evict_select.argtypes = [f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, i32p]
        lib.kvqo_compact_side.argtypes = [ctypes.c_int, ctypes.c_int, u8p, u8p, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, i32p, i32p, i32p,
                                          ctypes.c_int]
        lib.kvqo_num_threads.restype = ctypes.c_int
        lib.kvqo_set_num_threads.argtypes = [ctypes.c_int]
        lib.kvqo_set_num_threads.restype = ctypes.c_int
        lib.kvqo_stream_absmax.argtypes = [ctypes.c_int, ctypes.c_int, u8p, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int64]
        lib.kvqo_stream_absmax.restype = ctypes.c_double
        u64p = ctypes.POINTER(ctypes.c_uint64)
        lib.kvqo_splitmix64_next.argtypes = [u64p]
        lib.kvqo_splitmix64_next.restype = ctypes.c_uint64
        lib.kvqo_turbo_signs.argtypes = [ip]
        lib.kvqo_fwht128_f32.argtypes = [ctypes.POINTER(ctypes.c_float)]
        lib.kvqo_fwht128_f64.argtypes = [f64p]
        lib.kvqo_turbo4_rotated.argtypes = [u8p, f64p]
        _lib = lib
        return lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _as_half_bits(x) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype == np.float16:
        return np.ascontiguousarray(x).view(np.uint16)
    if x.dtype == np.uint16:
        return np.ascontiguousarray(x)
    raise TypeError(f"expected float16 (or its uint16 bits), got {x.dtype}")


def num_threads() -> int:
    return int(_load().kvqo_num_threads())


class threads:
    """Context manager: run the oracle's OpenMP regions on n threads."""

    def __init__(self, n: int):
        self.n = int(n)

    def __enter__(self):
        self.old = int(_load().kvqo_set_num_threads(self.n))
        return self

    def __exit__(self, *exc):
        _load().kvqo_set_num_threads(self.old)
        return False


# --------------------------------------------------------------------------- fp16

def half_to_float(bits: int) -> float:
    return float(_load().kvqo_half_to_float(int(bits)))


def float_to_half_bits(x: float) -> int:
    return int(_load().kvqo_float_to_half_rn(float(np.float32(x))))


# --------------------------------------------------------------------------- turbo4 pieces

def splitmix64(seed: int, n: int) -> list:
    """The first n outputs of SplitMix64 from ``seed``."""
    st = ctypes.c_uint64(seed)
    return [int(_load().kvqo_splitmix64_next(ctypes.byref(st))) for _ in range(n)]


def turbo_signs() -> np.ndarray:
    out = np.zeros(D, np.int32)
    _load().kvqo_turbo_signs(out.ctypes.data_as(ctypes.POINTER(ctypes.c_int)))
    return out


def fwht128(x, dtype=np.float64) -> np.ndarray:
    """Unnormalised Sylvester-order FWHT of a 128-vector in fp32 or fp64."""
    a = np.ascontiguousarray(x, dtype=dtype).copy()
    assert a.shape == (D,)
    if dtype == np.float32:
        _load().kvqo_fwht128_f32(_ptr(a, ctypes.c_float))
    else:
        _load().kvqo_fwht128_f64(_ptr(a, ctypes.c_double))
    return a


def turbo4_rotated(row: np.ndarray) -> np.ndarray:
    """y^ = d16 * (q - 8) of one canonical turbo4 row."""
    r = np.ascontiguousarray(row, dtype=np.uint8)
    out = np.zeros(D, np.float64)
    _load().kvqo_turbo4_rotated(_ptr(r, ctypes.c_uint8), _ptr(out, ctypes.c_double))
    return out


# --------------------------------------------------------------------------- codecs

def encode_rows(codec: int, x) -> np.ndarray:
    """fp16 [n, 128] -> canonical row bytes uint8 [n, row_bytes]."""
    xb = _as_half_bits(x).reshape(-1, D)
    out = np.zeros((xb.shape[0], ROW_BYTES[codec]), np.uint8)
    rc = _load().kvqo_encode_rows(codec, xb.shape[0], _ptr(xb, ctypes.c_uint16),
                                  _ptr(out, ctypes.c_uint8))
    if rc:
        raise ValueError(f"oracle encode failed ({rc}): non-finite input?")
    return out


def decode_rows(codec: int, rows: np.ndarray) -> np.ndarray:
    """canonical row bytes [n, row_bytes] -> fp64 [n, 128]."""
    rows = np.ascontiguousarray(rows, dtype=np.uint8).reshape(-1, ROW_BYTES[codec])
    out = np.zeros((rows.shape[0], D), np.float64)
    _load().kvqo_decode_rows(codec, rows.shape[0], _ptr(rows, ctypes.c_uint8),
                             _ptr(out, ctypes.c_double))
    return out


def unit_offset(codec: int, side: int, r: int, cb: int) -> int:
    return int(_load().kvqo_unit_offset(codec, side, r, cb))


def unit_offset_table(codec: int, side: int) -> np.ndarray:
    """int32 [16, row_bytes]: unit byte offset of canonical byte cb of row r."""
    rb = ROW_BYTES[codec]
    lib = _load()
    return np.array([[lib.kvqo_unit_offset(codec, side, r, cb) for cb in range(rb)]
                     for r in range(UNIT_TOKENS)], np.int32)


# --------------------------------------------------------------------------- cache

def cache_bytes(codec: int, n_seqs: int, n_kv: int, capacity: int) -> int:
    return n_seqs * n_kv * capacity * ROW_BYTES[codec]


def append_side(codec: int, side: int, cache: np.ndarray, n_seqs: int, n_kv: int,
                capacity: int, seq_lens, n_new, x_new) -> None:
    """Quantize-on-append into ``cache`` (uint8, modified in place).

    ``x_new``: fp16 [n_seqs, max_new, n_kv, 128]; row i < n_new[s] goes to
    position seq_lens[s] + i.  ``seq_lens`` is not modified.
    """
    assert cache.dtype == np.uint8 and cache.flags["C_CONTIGUOUS"]
    xb = _as_half_bits(x_new)
    max_new = xb.shape[1]
    sl = np.ascontiguousarray(seq_lens, np.int32)
    nn = np.ascontiguousarray(n_new, np.int32)
    rc = _load().kvqo_append_side(codec, side, _ptr(cache, ctypes.c_uint8), n_seqs, n_kv,
                                  capacity, _ptr(sl, ctypes.c_int32), _ptr(nn, ctypes.c_int32),
                                  max_new, _ptr(xb, ctypes.c_uint16))
    if rc:
        raise ValueError(f"oracle append failed ({rc})")


def dequant_stream(codec: int, side: int, cache: np.ndarray, n_kv: int, capacity: int,
                   seq: int, kvh: int, n_tokens: int) -> np.ndarray:
    out = np.zeros((n_tokens, D), np.float64)
    rc = _load().kvqo_dequant_stream(codec, side, _ptr(cache, ctypes.c_uint8), n_kv, capacity,
                                     seq, kvh, n_tokens, _ptr(out, ctypes.c_double))
    if rc:
        raise ValueError("oracle dequant failed")
    return out


def stream_absmax(codec: int, side: int, cache: np.ndarray, n_kv: int, capacity: int,
                  seq: int, kvh: int, n_tokens: int) -> float:
    """max |x^| over the first n_tokens decoded rows of one stream."""
    cache = np.ascontiguousarray(cache, dtype=np.uint8)
    m = float(_load().kvqo_stream_absmax(codec, side, _ptr(cache, ctypes.c_uint8), n_kv,
                                         capacity, seq, kvh, n_tokens))
    if m < 0:
        raise ValueError("oracle absmax failed")
    return m


# --------------------------------------------------------------------------- attention

def attend_rows(q, K: np.ndarray, V: np.ndarray, limit, scale: float):
    """q fp16 [n, 128]; K, V fp64 [T, 128]; row r attends keys < limit[r]."""
    qb = _as_half_bits(q).reshape(-1, D)
    K = np.ascontiguousarray(K, np.float64)
    V = np.ascontiguousarray(V, np.float64)
    lim = np.ascontiguousarray(np.broadcast_to(np.asarray(limit, np.int64), (qb.shape[0],)))
    out = np.zeros((qb.shape[0], D), np.float64)
    lse = np.zeros(qb.shape[0], np.float64)
    rc = _load().kvqo_attend_rows(qb.shape[0], _ptr(qb, ctypes.c_uint16), K.shape[0],
                                  _ptr(K, ctypes.c_double), _ptr(V, ctypes.c_double),
                                  _ptr(lim, ctypes.c_int64), float(scale),
                                  _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double))
    if rc:
        raise MemoryError("oracle attend failed")
    return out, lse


def decode_layer(codec_k: int, codec_v: int, cache_k: np.ndarray, cache_v: np.ndarray,
                 n_seqs: int, n_kv: int, n_q: int, capacity: int, seq_lens, q, scale: float,
                 sel=None):
    """Decode attention of one layer; ``sel`` (bool [n_seqs, n_kv]) limits the groups."""
    qb = _as_half_bits(q).reshape(n_seqs, n_q, D)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    out = np.full((n_seqs, n_q, D), np.nan)
    lse = np.full((n_seqs, n_q), np.nan)
    selp = None
    if sel is not None:
        s8 = np.ascontiguousarray(np.asarray(sel, bool).reshape(n_seqs, n_kv), np.uint8)
        selp = _ptr(s8, ctypes.c_uint8)
    rc = _load().kvqo_decode_layer(codec_k, codec_v, _ptr(cache_k, ctypes.c_uint8),
                                   _ptr(cache_v, ctypes.c_uint8), n_seqs, n_kv, n_q, capacity,
                                   _ptr(sl, ctypes.c_int32), _ptr(qb, ctypes.c_uint16),
                                   float(scale), selp, _ptr(out, ctypes.c_double),
                                   _ptr(lse, ctypes.c_double))
    if rc:
        raise ValueError(f"oracle decode failed ({rc})")
    return out, lse


def prefill_chunk(codec_k: int, codec_v: int, cache_k: np.ndarray, cache_v: np.ndarray,
                  n_kv: int, n_q: int, capacity: int, seq: int, q_start: int, q, scale: float,
                  rows=None):
    """Causal chunk attention; q fp16 [n_tok, n_q, 128]; ``rows`` limits query rows."""
    qb = _as_half_bits(q)
    n_tok = qb.shape[0]
    qb = qb.reshape(n_tok, n_q, D)
    out = np.full((n_tok, n_q, D), np.nan)
    lse = np.full((n_tok, n_q), np.nan)
    selp = None
    if rows is not None:
        s8 = np.zeros(n_tok, np.uint8)
        s8[np.asarray(rows)] = 1
        selp = _ptr(s8, ctypes.c_uint8)
    rc = _load().kvqo_prefill_chunk(codec_k, codec_v, _ptr(cache_k, ctypes.c_uint8),
                                    _ptr(cache_v, ctypes.c_uint8), n_kv, n_q, capacity, seq,
                                    q_start, n_tok, _ptr(qb, ctypes.c_uint16), float(scale), selp,
                                    _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double))
    if rc:
        raise ValueError(f"oracle prefill failed ({rc})")
    return out, lse


# --------------------------------------------------------------------------- degrade ladder

def requantize_side(src_codec: int, dst_codec: int, side: int, cache: np.ndarray, n_seqs: int,
                    n_kv: int, capacity: int, seq_lens) -> np.ndarray:
    """Re-encode tokens [0, seq_lens[s]) of one side's cache into a new cache of
    dst_codec (zero elsewhere)."""
    cache = np.ascontiguousarray(cache, dtype=np.uint8)
    out = np.zeros(cache_bytes(dst_codec, n_seqs, n_kv, capacity), np.uint8)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    rc = _load().kvqo_requantize_side(src_codec, dst_codec, side, _ptr(cache, ctypes.c_uint8),
                                      _ptr(out, ctypes.c_uint8), n_seqs, n_kv, capacity,
                                      _ptr(lens, ctypes.c_int32))
    if rc:
        raise ValueError(f"oracle requantize failed ({rc})")
    return out


def bits_per_value(codec: int) -> float:
    return float(_load().kvqo_bits_per_value(codec))


def aggregate_bpv(codecs) -> float:
    c = np.ascontiguousarray(codecs, dtype=np.intc)
    return float(_load().kvqo_aggregate_bpv(_ptr(c, ctypes.c_int), len(c)))


def ladder_next(codecs, order, floor_bpv: float):
    """(tensor, new codec) of the next banded degrade step, or None."""
    c = np.ascontiguousarray(codecs, dtype=np.intc)
    o = np.ascontiguousarray(order, dtype=np.intc)
    t, k = ctypes.c_int(-1), ctypes.c_int(-1)
    got = _load().kvqo_ladder_next(_ptr(c, ctypes.c_int), len(c), _ptr(o, ctypes.c_int), len(o),
                                   float(floor_bpv), ctypes.byref(t), ctypes.byref(k))
    return (t.value, k.value) if got else None


# --------------------------------------------------------------------------- paged layout

PAGE_TOKENS = 256


def pool_bytes(codec: int, n_pages: int, n_kv: int) -> int:
    return n_pages * n_kv * PAGE_TOKENS * ROW_BYTES[codec]


def paged_unit(s: int, h: int, j: int, n_kv: int, table, n_pages: int) -> int:
    t = np.ascontiguousarray(table, dtype=np.int32)
    return int(_load().kvqo_paged_unit(s, h, j, n_kv, _ptr(t, ctypes.c_int32), t.shape[1],
                                       n_pages))


def to_pool(codec: int, cache: np.ndarray, n_seqs: int, n_kv: int, capacity: int, table,
            n_pages: int, pool: np.ndarray = None) -> np.ndarray:
    """Scatter a contiguous cache into a page pool (new zeroed pool unless given)."""
    t = np.ascontiguousarray(table, dtype=np.int32)
    if pool is None:
        pool = np.zeros(pool_bytes(codec, n_pages, n_kv), np.uint8)
    cache = np.ascontiguousarray(cache, dtype=np.uint8)
    rc = _load().kvqo_page_move(codec, _ptr(cache, ctypes.c_uint8), n_seqs, n_kv, capacity,
                                _ptr(t, ctypes.c_int32), t.shape[1], _ptr(pool, ctypes.c_uint8),
                                n_pages, 1)
    if rc:
        raise ValueError("bad paged geometry")
    return pool


def from_pool(codec: int, pool: np.ndarray, n_seqs: int, n_kv: int, capacity: int, table,
              n_pages: int) -> np.ndarray:
    """Gather a page pool back into a contiguous cache (unmapped pages zero)."""
    t = np.ascontiguousarray(table, dtype=np.int32)
    cache = np.zeros(cache_bytes(codec, n_seqs, n_kv, capacity), np.uint8)
    pool = np.ascontiguousarray(pool, dtype=np.uint8)
    rc = _load().kvqo_page_move(codec, _ptr(cache, ctypes.c_uint8), n_seqs, n_kv, capacity,
                                _ptr(t, ctypes.c_int32), t.shape[1], _ptr(pool, ctypes.c_uint8),
                                n_pages, 0)
    if rc:
        raise ValueError("bad paged geometry")
    return cache


# --------------------------------------------------------------------------- probe-scored eviction

def probe_mass(codec_k: int, cache_k: np.ndarray, n_seqs: int, n_kv: int, n_q: int,
               capacity: int, seq_lens, q, scale: float) -> np.ndarray:
    """fp64 [n_seqs, capacity]: per token, the softmax weight summed over query heads."""
    qb = _as_half_bits(q).reshape(-1)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    cache_k = np.ascontiguousarray(cache_k, dtype=np.uint8)
    out = np.zeros((n_seqs, capacity), np.float64)
    rc = _load().kvqo_probe_mass(codec_k, _ptr(cache_k, ctypes.c_uint8), n_seqs, n_kv, n_q,
                                 capacity, _ptr(lens, ctypes.c_int32), _ptr(qb, ctypes.c_uint16),
                                 float(scale), _ptr(out, ctypes.c_double))
    if rc:
        raise ValueError("oracle probe failed")
    return out


def evict_select(score, length: int, n_sink: int, n_recent: int, n_evict: int) -> np.ndarray:
    sc = np.ascontiguousarray(score, dtype=np.float32)
    out = np.zeros(max(n_evict, 1), np.int32)
    w = _load().kvqo_evict_select(_ptr(sc, ctypes.c_float), int(length), int(n_sink),
                                  int(n_recent), int(n_evict), _ptr(out, ctypes.c_int32))
    if w < 0:
        raise MemoryError
    return out[:w]


def compact_side(codec: int, side: int, cache: np.ndarray, n_seqs: int, n_kv: int,
                 capacity: int, seq_lens, evict) -> np.ndarray:
    """Cache with the listed positions of each sequence removed (evict: list of
    increasing position lists)."""
    me = max(1, max(len(e) for e in evict))
    ev = np.zeros((n_seqs, me), np.int32)
    nev = np.zeros(n_seqs, np.int32)
    for s, e in enumerate(evict):
        ev[s, :len(e)] = e
        nev[s] = len(e)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    cache = np.ascontiguousarray(cache, dtype=np.uint8)
    out = np.zeros(cache_bytes(codec, n_seqs, n_kv, capacity), np.uint8)
    rc = _load().kvqo_compact_side(codec, side, _ptr(cache, ctypes.c_uint8),
                                   _ptr(out, ctypes.c_uint8), n_seqs, n_kv, capacity,
                                   _ptr(lens, ctypes.c_int32), _ptr(ev, ctypes.c_int32),
                                   _ptr(nev, ctypes.c_int32), me)
    if rc:
        raise ValueError("oracle compaction failed")
    return out
