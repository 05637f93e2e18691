"""Shared helpers of the GPU tests: fill caches through the CUDA append path
and build the matching oracle caches from the same seeded draws."""
import math

import numpy as np
import torch

import attention_quantized_kv_gb300 as kvq
from attention_quantized_kv_gb300 import workloads as wl

import oracle

ROW = {0: 256, 1: 136, 2: 72, 3: 66}


def gpu_layer(w, layer_idx, device="cuda", chunk=4096, lens=None):
    """A KVLayer of workload w filled through kv_append_quantize (zero-initialised)."""
    ck, cv = w.codecs[layer_idx]
    L = kvq.KVLayer(w.n_seqs, w.n_kv, w.n_q, w.capacity, ck, cv, device=device,
                    k_cache=torch.zeros(kvq.kvq_cache_bytes(ck, w.n_seqs, w.n_kv, w.capacity),
                                        dtype=torch.uint8, device=device),
                    v_cache=torch.zeros(kvq.kvq_cache_bytes(cv, w.n_seqs, w.n_kv, w.capacity),
                                        dtype=torch.uint8, device=device))
    lens = w.lens if lens is None else lens
    for start in range(0, max(lens), chunk):
        n = [max(0, min(chunk, ln - start)) for ln in lens]
        mx = max(n)
        k_new = torch.zeros((w.n_seqs, mx, w.n_kv, 128), dtype=torch.float16, device=device)
        v_new = torch.zeros_like(k_new)
        for s in range(w.n_seqs):
            if n[s]:
                k_new[s, :n[s]] = wl.kv_rows(w, layer_idx, 0, s, start, n[s], device)
                v_new[s, :n[s]] = wl.kv_rows(w, layer_idx, 1, s, start, n[s], device)
        kvq.kv_append_quantize(L, k_new, v_new, torch.tensor(n, dtype=torch.int32, device=device))
    return L


def oracle_stream(w, layer_idx, seq, kvh, n_tokens, device="cuda"):
    """Oracle caches (K side, V side) of ONE (seq, kv head) stream as a 1x1 layer."""
    ck, cv = w.codecs[layer_idx]
    cap = w.capacity
    out = []
    for side, codec in ((0, ck), (1, cv)):
        rows = wl.kv_rows(w, layer_idx, side, seq, 0, n_tokens, device)[:, kvh]
        x = rows.cpu().numpy().reshape(1, n_tokens, 1, 128)
        c = np.zeros(oracle.cache_bytes(codec, 1, 1, cap), np.uint8)
        oracle.append_side(codec, side, c, 1, 1, cap, [0], [n_tokens], x)
        out.append(c)
    return out


def oracle_layer(w, layer_idx, lens, device="cuda", chunk=16384):
    """Oracle caches (K side, V side) of a whole layer: tokens [0, lens[s])
    of every sequence appended by the oracle from the same seeded draws."""
    ck, cv = w.codecs[layer_idx]
    out = []
    for side, codec in ((0, ck), (1, cv)):
        c = np.zeros(oracle.cache_bytes(codec, w.n_seqs, w.n_kv, w.capacity), np.uint8)
        for start in range(0, max(lens), chunk):
            n = [max(0, min(chunk, ln - start)) for ln in lens]
            x = np.zeros((w.n_seqs, max(n), w.n_kv, 128), np.float16)
            for s in range(w.n_seqs):
                if n[s]:
                    x[s, :n[s]] = wl.kv_rows(w, layer_idx, side, s, start, n[s],
                                             device).cpu().numpy()
            oracle.append_side(codec, side, c, w.n_seqs, w.n_kv, w.capacity,
                               [min(start, ln) for ln in lens], n, x)
        out.append(c)
    return out


def gpu_stream_bytes(L, side, seq, kvh):
    cache = L.k_cache if side == 0 else L.v_cache
    codec = L.codec_k if side == 0 else L.codec_v
    n = L.capacity * ROW[codec]
    s0 = (seq * L.n_kv_heads + kvh) * n
    return cache[s0:s0 + n].cpu().numpy()


def tol(vmax):
    return 2e-3 * vmax


def boundary_rows(codec, n_rows, rng):
    """fp16 rows whose quotients x/d fall at or within a few fp32 ulps of the
    encoder's rounding boundaries (half-integers for q8_0; half-integers, so
    that u = x/d + 8.5 is near an integer, for q4_0).  Each 32-value block
    keeps one value of the largest magnitude and fills the rest from the fp16
    values whose quotient lies nearest such a boundary."""
    f16 = np.arange(1 << 16, dtype=np.uint16).view(np.float16)
    f16 = f16[np.isfinite(f16)].astype(np.float32)
    rows = np.zeros((n_rows, 128), np.float32)
    for r in range(n_rows):
        for b in range(4):
            amax = np.float32(rng.choice([1.0, 0.3, 7.5, 1e-3, 250.0])) * np.float32(rng.uniform(0.5, 2))
            amax = np.float32(np.float16(amax))
            sign = np.float32(rng.choice([-1.0, 1.0]))
            if codec == 1:
                d = np.float32(amax / np.float32(127))
            else:
                d = np.float32(sign * amax / np.float32(-8))
            cand = f16[np.abs(f16) < amax]
            t = (cand / d).astype(np.float32).astype(np.float64)
            dist = np.abs(np.abs(t - np.floor(t)) - 0.5)
            pick = cand[np.argsort(dist)[:48]]
            blk = rng.choice(pick, 32)
            blk[rng.integers(0, 32)] = sign * amax
            rows[r, 32 * b:32 * b + 32] = blk
    return rows.astype(np.float16)
