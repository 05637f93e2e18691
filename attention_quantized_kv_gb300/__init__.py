"""attention_quantized_kv_gb300: attention over a block-quantized KV cache on GB300.

A thin Python layer over libkvq's C ABI (include/kvq.h).  PyTorch provides
device memory and streams; every step of the path (quantize-on-append,
split-K decode attention with its log-sum-exp merge, chunked-prefill
attention, the degrade ladder's re-encode, probe-scored eviction) runs in the
library's sm_103a kernels.  The functions below only
marshal arguments: they take torch tensors, pass their device pointers and
raise ``KVQError`` on a non-zero status.
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import _abi
from ._abi import (KVQ_F16, KVQ_Q8_0, KVQ_Q4_0, KVQ_TURBO4, KVQ_DEVERR_CAPACITY,
                   KVQ_DEVERR_EVICT,
                   KVQ_DEVERR_MAXLEN, KVQ_DEVERR_PAGE, KVQ_DEVERR_SEQLEN, KVQ_DEVERR_TIMEOUT,
                   kvq_layer)

__all__ = ["KVQ_F16", "KVQ_Q8_0", "KVQ_Q4_0", "KVQ_TURBO4", "CODEC_NAMES", "KVQError", "KVLayer",
           "kv_append_quantize", "attn_decode_workspace", "attn_decode", "attn_decode_append",
           "attn_prefill_workspace", "attn_prefill_chunk", "kvq_row_bytes", "kvq_cache_bytes",
           "kvq_pool_bytes", "KVQ_DEVERR_PAGE", "kv_requantize", "degrade", "aggregate_bpv",
           "ladder_next", "default_scale", "KVQ_DEVERR_EVICT", "kv_probe_scores",
           "kv_evict_select", "kv_compact", "evict"]

CODEC_NAMES = {KVQ_F16: "f16", KVQ_Q8_0: "q8_0", KVQ_Q4_0: "q4_0", KVQ_TURBO4: "turbo4"}
HEAD_DIM = 128


class KVQError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = _abi.load().kvq_status_str(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")
        self.status = status


def _check(status: int, where: str) -> None:
    if status != 0:
        raise KVQError(status, where)


def _stream_ptr(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _ptr(t) -> int | None:
    return None if t is None else int(t.data_ptr())


def default_scale(head_dim: int = HEAD_DIM) -> float:
    return 1.0 / math.sqrt(head_dim)


def kvq_row_bytes(codec: int, head_dim: int = HEAD_DIM) -> int:
    return int(_abi.load().kvq_row_bytes(codec, head_dim))


def kvq_cache_bytes(codec: int, n_seqs: int, n_kv_heads: int, capacity: int,
                    head_dim: int = HEAD_DIM) -> int:
    return int(_abi.load().kvq_cache_bytes(codec, n_seqs, n_kv_heads, capacity, head_dim))


def kvq_pool_bytes(codec: int, n_pages: int, n_kv_heads: int,
                   head_dim: int = HEAD_DIM) -> int:
    return int(_abi.load().kvq_pool_bytes(codec, n_pages, n_kv_heads, head_dim))


class KVLayer:
    """One layer's cache: torch-owned device buffers plus the C descriptor.

    ``k_cache``/``v_cache`` are uint8 tensors in the layout of include/kvq.h,
    ``seq_lens`` int32 [n_seqs] and ``err`` one int32 error word.  Paged
    layers (``n_pages`` > 0) hold page pools instead, and ``block_table``
    (int32 [n_seqs][capacity / 256], device) maps each sequence's pages to
    pool pages (-1: not mapped; default: every page mapped, in order).
    """

    def __init__(self, n_seqs: int, n_kv_heads: int, n_q_heads: int, capacity: int,
                 codec_k: int, codec_v: int, device="cuda", head_dim: int = HEAD_DIM,
                 k_cache=None, v_cache=None, n_pages: int = 0, block_table=None):
        self.n_seqs, self.n_kv_heads, self.n_q_heads = n_seqs, n_kv_heads, n_q_heads
        self.capacity, self.codec_k, self.codec_v, self.head_dim = (capacity, codec_k, codec_v,
                                                                    head_dim)
        self.n_pages = int(n_pages)
        self.block_table = None
        if self.n_pages > 0:
            pps = capacity // 256
            if block_table is None:
                block_table = torch.arange(n_seqs * pps, dtype=torch.int32,
                                           device=device).reshape(n_seqs, pps)
            assert block_table.dtype == torch.int32 and block_table.shape == (n_seqs, pps)
            self.block_table = block_table.contiguous()
            kb = kvq_pool_bytes(codec_k, self.n_pages, n_kv_heads, head_dim)
            vb = kvq_pool_bytes(codec_v, self.n_pages, n_kv_heads, head_dim)
        else:
            kb = kvq_cache_bytes(codec_k, n_seqs, n_kv_heads, capacity, head_dim)
            vb = kvq_cache_bytes(codec_v, n_seqs, n_kv_heads, capacity, head_dim)
        if kb < 0 or vb < 0:
            raise ValueError("invalid cache geometry (capacity must be a multiple of 256, "
                             "head_dim 128, codecs f16/q8_0/q4_0/turbo4)")
        self.k_cache = k_cache if k_cache is not None else torch.empty(kb, dtype=torch.uint8,
                                                                        device=device)
        self.v_cache = v_cache if v_cache is not None else torch.empty(vb, dtype=torch.uint8,
                                                                        device=device)
        assert self.k_cache.numel() == kb and self.v_cache.numel() == vb
        self.seq_lens = torch.zeros(n_seqs, dtype=torch.int32, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self._desc = None
        self._desc_key = None

    def desc(self) -> kvq_layer:
        """The C descriptor (rebuilt only when a buffer was replaced)."""
        key = (_ptr(self.k_cache), _ptr(self.v_cache), _ptr(self.seq_lens), _ptr(self.err),
               self.codec_k, self.codec_v, _ptr(self.block_table), self.n_pages)
        if self._desc is None or self._desc_key != key:
            d = kvq_layer()
            d.n_seqs, d.n_kv_heads, d.n_q_heads = self.n_seqs, self.n_kv_heads, self.n_q_heads
            d.head_dim, d.capacity = self.head_dim, self.capacity
            d.codec_k, d.codec_v, d.reserved = self.codec_k, self.codec_v, 0
            d.k_cache, d.v_cache, d.seq_lens, d.err = key[:4]
            if self.n_pages > 0:
                d.pages_per_seq, d.block_table, d.n_pages = (self.capacity // 256,
                                                             _ptr(self.block_table), self.n_pages)
            else:
                d.pages_per_seq, d.block_table, d.n_pages = 0, None, 0
            self._desc, self._desc_key = d, key
        return self._desc


def kv_append_quantize(layer: KVLayer, k_new, v_new, n_new, update_lens: bool = True,
                       stream=None) -> None:
    """k_new, v_new: fp16 [n_seqs, max_new, n_kv, 128]; n_new: int32 [n_seqs] (device)."""
    assert k_new.dtype == torch.float16 and v_new.dtype == torch.float16
    assert k_new.is_contiguous() and v_new.is_contiguous() and n_new.dtype == torch.int32
    max_new = int(k_new.shape[1])
    d = layer.desc()
    _check(_abi.load().kv_append_quantize(ctypes.byref(d), _ptr(k_new), _ptr(v_new),
                                          _ptr(n_new), max_new, int(bool(update_lens)),
                                          _stream_ptr(stream)), "kv_append_quantize")


def attn_decode_workspace(layer: KVLayer, max_len: int) -> int:
    """Bytes of decode workspace; allocate it zero-filled (torch.zeros)."""
    n = ctypes.c_size_t(0)
    d = layer.desc()
    _check(_abi.load().attn_decode_workspace(ctypes.byref(d), int(max_len), ctypes.byref(n)),
           "attn_decode_workspace")
    return int(n.value)


def attn_decode(layer: KVLayer, q, scale: float, out, lse, max_len: int, workspace,
                stream=None) -> None:
    """q, out: fp16 [n_seqs, n_q, 128]; lse: fp32 [n_seqs, n_q] or None."""
    assert q.dtype == torch.float16 and out.dtype == torch.float16 and q.is_contiguous()
    d = layer.desc()
    _check(_abi.load().attn_decode(ctypes.byref(d), _ptr(q), float(scale), _ptr(out), _ptr(lse),
                                   int(max_len), _ptr(workspace), int(workspace.numel() *
                                                                      workspace.element_size()),
                                   _stream_ptr(stream)), "attn_decode")


def attn_decode_append(layer: KVLayer, k_new, v_new, q, scale: float, out, lse, max_len: int,
                       workspace, stream=None) -> None:
    """One decode step in one launch: append k_new / v_new (fp16 [n_seqs, n_kv, 128], one
    token per sequence), attend seq_lens + 1 keys, advance seq_lens.  q, out: fp16
    [n_seqs, n_q, 128]; lse: fp32 [n_seqs, n_q] or None; workspace as attn_decode."""
    assert k_new.dtype == torch.float16 and v_new.dtype == torch.float16
    assert k_new.is_contiguous() and v_new.is_contiguous()
    assert q.dtype == torch.float16 and out.dtype == torch.float16 and q.is_contiguous()
    d = layer.desc()
    _check(_abi.load().attn_decode_append(ctypes.byref(d), _ptr(k_new), _ptr(v_new), _ptr(q),
                                          float(scale), _ptr(out), _ptr(lse), int(max_len),
                                          _ptr(workspace),
                                          int(workspace.numel() * workspace.element_size()),
                                          _stream_ptr(stream)), "attn_decode_append")


def attn_prefill_workspace(layer: KVLayer, q_start: int, n_q_tok: int) -> int:
    n = ctypes.c_size_t(0)
    d = layer.desc()
    _check(_abi.load().attn_prefill_workspace(ctypes.byref(d), int(q_start), int(n_q_tok),
                                              ctypes.byref(n)), "attn_prefill_workspace")
    return int(n.value)


def attn_prefill_chunk(layer: KVLayer, seq: int, q_start: int, q, scale: float, out, lse,
                       workspace, stream=None) -> None:
    """q, out: fp16 [n_q_tok, n_q, 128]; lse: fp32 [n_q_tok, n_q] or None."""
    assert q.dtype == torch.float16 and out.dtype == torch.float16 and q.is_contiguous()
    d = layer.desc()
    _check(_abi.load().attn_prefill_chunk(ctypes.byref(d), int(seq), int(q_start),
                                          int(q.shape[0]), _ptr(q), float(scale), _ptr(out),
                                          _ptr(lse), _ptr(workspace),
                                          int(workspace.numel() * workspace.element_size()),
                                          _stream_ptr(stream)), "attn_prefill_chunk")


# --------------------------------------------------------------------------- degrade ladder

def _side_bytes(layer: KVLayer, codec: int) -> int:
    if layer.n_pages > 0:
        return kvq_pool_bytes(codec, layer.n_pages, layer.n_kv_heads, layer.head_dim)
    return kvq_cache_bytes(codec, layer.n_seqs, layer.n_kv_heads, layer.capacity, layer.head_dim)


def kv_requantize(layer: KVLayer, side: int, dst_codec: int, dst_cache, stream=None) -> None:
    """Re-encode side ``side`` (0 = K, 1 = V) of ``layer`` with ``dst_codec`` into
    ``dst_cache`` (uint8 device tensor of kvq_cache_bytes(dst_codec, ...) bytes)."""
    assert dst_cache.dtype == torch.uint8 and dst_cache.is_contiguous()
    nb = _side_bytes(layer, dst_codec)
    if dst_cache.numel() != nb:
        raise ValueError(f"dst_cache must hold {nb} bytes")
    d = layer.desc()
    _check(_abi.load().kv_requantize(ctypes.byref(d), int(side), int(dst_codec), _ptr(dst_cache),
                                     _stream_ptr(stream)), "kv_requantize")


def degrade(layer: KVLayer, side: int, dst_codec: int, stream=None) -> None:
    """Move one side of ``layer`` to ``dst_codec``: a new, zeroed cache buffer
    (torch allocation; rows past the lengths stay zero), the re-encode, then
    the layer points at the new buffer."""
    nb = _side_bytes(layer, dst_codec)
    src = layer.k_cache if side == 0 else layer.v_cache
    dst = torch.zeros(nb, dtype=torch.uint8, device=src.device)
    kv_requantize(layer, side, dst_codec, dst, stream)
    if side == 0:
        layer.k_cache, layer.codec_k = dst, dst_codec
    else:
        layer.v_cache, layer.codec_v = dst, dst_codec


def aggregate_bpv(codecs) -> float:
    arr = (ctypes.c_int32 * len(codecs))(*[int(c) for c in codecs])
    v = float(_abi.load().kvq_aggregate_bpv(arr, len(codecs)))
    if v < 0:
        raise ValueError("invalid codecs")
    return v


def ladder_next(codecs, floor_bpv: float, order=None):
    """(tensor, codec) of the next banded degrade step, or None."""
    arr = (ctypes.c_int32 * len(codecs))(*[int(c) for c in codecs])
    if order is None:
        ordp, n_order = None, 0
    else:
        ordp = (ctypes.c_int32 * len(order))(*[int(t) for t in order])
        n_order = len(order)
    t, k = ctypes.c_int32(-1), ctypes.c_int32(-1)
    _check(_abi.load().kvq_ladder_next(arr, len(codecs), ordp, n_order, float(floor_bpv),
                                       ctypes.byref(t), ctypes.byref(k)), "kvq_ladder_next")
    return None if t.value < 0 else (t.value, k.value)


# --------------------------------------------------------------------------- probe eviction

def kv_probe_scores(layer: KVLayer, q, scale: float, lse, decay: float, scores,
                    stream=None) -> None:
    """Fold one probe into ``scores`` (fp32 [n_seqs, capacity], device, in place):
    score = decay * score + the softmax mass the decode query ``q`` (fp16
    [n_seqs, n_q, 128]) puts on each token, summed over the query heads; ``lse``
    is attn_decode's fp32 [n_seqs, n_q] output for the same q and scale."""
    assert q.dtype == torch.float16 and q.is_contiguous()
    assert lse.dtype == torch.float32 and lse.is_contiguous()
    assert scores.dtype == torch.float32 and scores.is_contiguous()
    assert scores.numel() == layer.n_seqs * layer.capacity
    assert lse.numel() == layer.n_seqs * layer.n_q_heads
    d = layer.desc()
    _check(_abi.load().kv_probe_scores(ctypes.byref(d), _ptr(q), float(scale), _ptr(lse),
                                       float(decay), _ptr(scores), _stream_ptr(stream)),
           "kv_probe_scores")


def kv_evict_select(layer: KVLayer, scores, n_sink: int, n_recent: int, n_evict: int, evict,
                    n_evicted, stream=None) -> None:
    """Per sequence, the n_evict lowest (score, position) middle positions in
    increasing order into ``evict`` (int32 [n_seqs, n_evict]) and their count
    into ``n_evicted`` (int32 [n_seqs])."""
    assert scores.dtype == torch.float32 and scores.numel() == layer.n_seqs * layer.capacity
    assert evict.dtype == torch.int32 and evict.numel() >= layer.n_seqs * max(int(n_evict), 0)
    assert n_evicted.dtype == torch.int32 and n_evicted.numel() == layer.n_seqs
    d = layer.desc()
    _check(_abi.load().kv_evict_select(ctypes.byref(d), _ptr(scores), int(n_sink), int(n_recent),
                                       int(n_evict), _ptr(evict), _ptr(n_evicted),
                                       _stream_ptr(stream)), "kv_evict_select")


def kv_compact(layer: KVLayer, evict, n_evicted, k_dst, v_dst, scores=None, scores_dst=None,
               lens_dst=None, stream=None) -> None:
    """Remove the listed positions (``evict`` int32 [n_seqs, max_evict]) from both
    sides into ``k_dst``/``v_dst`` (uint8, the sizes of the layer's caches);
    optionally the scores and the new lengths too."""
    assert evict.dtype == torch.int32 and evict.dim() == 2 and evict.is_contiguous()
    assert n_evicted.dtype == torch.int32 and n_evicted.numel() == layer.n_seqs
    assert k_dst.dtype == torch.uint8 and v_dst.dtype == torch.uint8
    if k_dst.numel() != _side_bytes(layer, layer.codec_k) or \
            v_dst.numel() != _side_bytes(layer, layer.codec_v):
        raise ValueError("k_dst / v_dst must have the sizes of the layer's caches")
    d = layer.desc()
    _check(_abi.load().kv_compact(ctypes.byref(d), _ptr(evict), _ptr(n_evicted),
                                  int(evict.shape[1]), _ptr(k_dst), _ptr(v_dst), _ptr(scores),
                                  _ptr(scores_dst), _ptr(lens_dst), _stream_ptr(stream)),
           "kv_compact")


def evict(layer: KVLayer, scores, n_sink: int, n_recent: int, n_evict: int, stream=None):
    """Select and remove up to n_evict tokens per sequence: new zeroed cache
    buffers (torch allocations), the layer repointed at them and at the new
    lengths.  Returns (compacted scores, evict list, n_evicted)."""
    dev = layer.k_cache.device
    ev = torch.zeros((layer.n_seqs, max(int(n_evict), 1)), dtype=torch.int32, device=dev)
    nev = torch.zeros(layer.n_seqs, dtype=torch.int32, device=dev)
    kv_evict_select(layer, scores, n_sink, n_recent, n_evict, ev, nev, stream)
    k_dst = torch.zeros_like(layer.k_cache)
    v_dst = torch.zeros_like(layer.v_cache)
    s_dst = torch.zeros_like(scores)
    lens = torch.empty_like(layer.seq_lens)
    kv_compact(layer, ev, nev, k_dst, v_dst, scores, s_dst, lens, stream)
    layer.k_cache, layer.v_cache, layer.seq_lens = k_dst, v_dst, lens
    return s_dst, ev, nev
