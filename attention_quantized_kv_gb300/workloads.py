"""Seeded synthetic workloads: shapes, codec choices and input draws.

This module holds no arithmetic of the method.  It only says what each
workload looks like and draws its inputs, so that the CUDA path and the CPU
oracle receive identical tensors.  Draws use a seeded ``torch.Generator`` on
the device where the tensors are made (fast for multi-GB caches; the oracle
gets a host copy of the same values); small structural choices (ragged
lengths, outlier channels, the per-(layer, side) codec ladder) use numpy's
``default_rng`` with the workload's seed.

Workloads (head_dim 128 throughout):
  decode_q8_ctx4k        1 sequence, 8 query / 2 KV heads, 4096 cached keys,
                         K and V q8_0, N(0,1) fp16, seed 0; one decode token.
  append_decode_q4_ctx32k
                         1 sequence, 32 query / 8 KV heads, 32768 cached keys,
                         K and V q4_0, N(0,1) with 1% of the (kv head, dim)
                         channels of each side scaled x8 (outlier channels),
                         seed 1; append one token, then decode over 32769 keys.
  decode_ragged16_kf16_vq8
                         16 sequences, lengths uniform in [1024, 65536] from
                         seed 2, 40 query / 8 KV heads, K f16 / V q8_0 (the
                         asymmetric contract), N(0,1); one decode token each.
  decode_16layer_ladder_2x200704
                         16 layers, 2 sequences x 200704 keys, 32 query / 4 KV
                         heads; each of the 32 (layer, side) tensors is f16,
                         q8_0 or q4_0 (11/11/10, shuffled by seed 3), N(0,1).
  evict_ragged16_kf16_vq8
                         the decode_ragged16_kf16_vq8 cache and query; one
                         probe-scored eviction step: decode (with its
                         log-sum-exp), probe scores (decay 0.9), selection of
                         the 2048 lowest middle cells per sequence (4 sink and
                         1024 recent cells protected) and compaction of K, V,
                         scores and lengths into second buffers.
  append_decode_turbo4_ctx32k
                         append_decode_q4_ctx32k with K and V turbo4 (the
                         rotated 4-bit rows, 4.125 bits per value).
  prefill_q8_32k_plus_2k 1 sequence with 32768 cached keys plus a 2048-token
                         ubatch quantize-appended, then causal attention of the
                         2048 queries over 34816 keys; 32 query / 8 KV heads,
                         K and V q8_0, N(0,1), seed 4.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import re

import numpy as np
import torch

F16, Q8_0, Q4_0, TURBO4 = 0, 1, 2, 3
HEAD_DIM = 128


@dataclass
class Workload:
    name: str
    kind: str                 # "decode", "prefill", "degrade" or "evict"
    n_seqs: int
    n_q: int
    n_kv: int
    lens: list                # cached keys per sequence before the timed step
    codecs: list              # [(codec_k, codec_v)] per layer
    seed: int
    append_new: int = 0       # tokens appended per sequence inside the timed step
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    description: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def n_layers(self) -> int:
        return len(self.codecs)

    @property
    def capacity(self) -> int:
        need = max(self.lens) + self.append_new
        return max(256, (need + 255) // 256 * 256)

    def final_lens(self) -> list:
        return [n + self.append_new for n in self.lens]


def _ladder(seed: int, n_layers: int = 16) -> list:
    rng = np.random.default_rng(seed)
    tensors = rng.permutation([F16] * 11 + [Q8_0] * 11 + [Q4_0] * 10)
    return [(int(tensors[2 * l]), int(tensors[2 * l + 1])) for l in range(n_layers)]


def get(name: str) -> Workload:
    if name == "decode_q8_ctx4k":
        return Workload(name, "decode", 1, 8, 2, [4096], [(Q8_0, Q8_0)], 0,
                        description="1 seq, 8q/2kv heads, ctx 4096, K/V q8_0, 1 decode token")
    if name == "append_decode_q4_ctx32k":
        return Workload(name, "decode", 1, 32, 8, [32768], [(Q4_0, Q4_0)], 1, append_new=1,
                        outlier_frac=0.01, outlier_scale=8.0,
                        description="1 seq, 32q/8kv heads, ctx 32768, K/V q4_0, 1% outlier "
                                    "channels x8; append 1 token then decode")
    if name == "append_decode_turbo4_ctx32k":
        return Workload(name, "decode", 1, 32, 8, [32768], [(TURBO4, TURBO4)], 1, append_new=1,
                        outlier_frac=0.01, outlier_scale=8.0,
                        description="append_decode_q4_ctx32k with K/V turbo4 (Hadamard-rotated "
                                    "4-bit rows, 4.125 bpv) instead of q4_0")
    if name == "decode_ragged16_kf16_vq8":
        lens = [int(x) for x in np.random.default_rng(2).integers(1024, 65537, 16)]
        return Workload(name, "decode", 16, 40, 8, lens, [(F16, Q8_0)], 2,
                        description="16 seqs, ragged lengths U[1024,65536], 40q/8kv heads, "
                                    "K f16 / V q8_0, 1 decode token per seq")
    if name == "decode_16layer_ladder_2x200704":
        return Workload(name, "decode", 2, 32, 4, [200704, 200704], _ladder(3), 3,
                        description="16 layers, 2 seqs x 200704 keys, 32q/4kv heads, "
                                    "per-(layer, side) f16/q8_0/q4_0 ladder")
    m = re.fullmatch(r"decode_ladder_layer(\d+)_2x200704", name)
    if m and int(m.group(1)) < 16:
        # one layer of the 16-layer ladder alone (a profiling size: 0.23 to
        # 0.82 GB of cache)
        l = int(m.group(1))
        w = get("decode_16layer_ladder_2x200704")
        codecs = w.codecs[l]
        names = ["f16", "q8_0", "q4_0"]
        return Workload(name, "decode", 2, 32, 4, [200704, 200704], [codecs], 3,
                        description=f"layer {l} of decode_16layer_ladder_2x200704 alone "
                                    f"(K {names[codecs[0]]} / V {names[codecs[1]]})")
    if name == "prefill_q8_32k_plus_2k":
        return Workload(name, "prefill", 1, 32, 8, [32768], [(Q8_0, Q8_0)], 4, append_new=2048,
                        description="1 seq, 32768 cached + 2048-token ubatch appended, causal "
                                    "attention of 2048 queries over 34816 keys, 32q/8kv, q8_0")
    if name == "decode_ragged16_kf16_vq8_paged":
        w = get("decode_ragged16_kf16_vq8")
        w.name = name
        w.extra = {"paged": True, "page_seed": 12}
        w.description = ("decode_ragged16_kf16_vq8 over a paged pool: 256-token pages, "
                         "block table shuffled from seed 12, pool = pages needed + 5%")
        return w
    if name == "degrade_f16_q8_2x200704":
        return Workload(name, "degrade", 2, 32, 4, [200704, 200704], [(F16, F16)], 3,
                        extra={"side": 0, "dst": Q8_0},
                        description="one degrade-ladder step: re-encode the K side of a "
                                    "2 x 200704-key layer (4 kv heads) from f16 to q8_0")
    if name == "degrade_v_f16_q8_2x200704":
        w = get("degrade_f16_q8_2x200704")
        w.name = name
        w.extra = {"side": 1, "dst": Q8_0}
        w.description = ("one degrade-ladder step on the V side: re-encode the V side of a "
                         "2 x 200704-key layer (4 kv heads) from f16 to q8_0")
        return w
    if name == "evict_ragged16_kf16_vq8":
        w = get("decode_ragged16_kf16_vq8")
        w.name, w.kind = name, "evict"
        w.extra = {"n_sink": 4, "n_recent": 1024, "n_evict": 2048, "decay": 0.9,
                   "score_seed": 13}
        w.description = ("decode_ragged16_kf16_vq8 + one probe-scored eviction: probe "
                         "(decay 0.9), 2048 lowest middle cells per seq (4 sink / 1024 recent "
                         "protected), compaction of K, V, scores and lengths")
        return w
    if name == "evict_ragged4_kf16_vq8":
        w = get("evict_ragged16_kf16_vq8")
        w.name, w.n_seqs, w.lens = name, 4, w.lens[:4]
        w.description = ("the first 4 sequences of evict_ragged16_kf16_vq8 (a profiling "
                         "size: ~1.4 GB of caches with the compaction's second buffers)")
        return w
    raise KeyError(name)


ALL = ["decode_q8_ctx4k", "append_decode_q4_ctx32k", "decode_ragged16_kf16_vq8",
       "decode_16layer_ladder_2x200704", "decode_ladder_layer0_2x200704",
       "decode_ladder_layer8_2x200704", "prefill_q8_32k_plus_2k", "degrade_f16_q8_2x200704",
       "degrade_v_f16_q8_2x200704",
       "decode_ragged16_kf16_vq8_paged", "evict_ragged16_kf16_vq8", "evict_ragged4_kf16_vq8",
       "append_decode_turbo4_ctx32k"]


def n_evicted(w: Workload) -> list:
    """Cells an eviction step of workload w removes from each sequence."""
    e = w.extra
    return [max(0, min(e["n_evict"], n - e["n_sink"] - e["n_recent"])) for n in w.final_lens()]


def initial_scores(w: Workload, device="cpu") -> torch.Tensor:
    """fp32 [n_seqs, capacity]: the running scores before the step (a probe
    history), uniform in [0, 1) from the workload's score seed."""
    g = _gen(device, w.extra["score_seed"], 0)
    return torch.rand((w.n_seqs, w.capacity), generator=g, device=device, dtype=torch.float32)


# ------------------------------------------------------------------ draws

def _gen(device, seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + stream * 7919) % (2 ** 63))
    return g


def normal_fp16(shape, seed: int, stream: int, device="cpu", scale_channels=None) -> torch.Tensor:
    """N(0,1) draws rounded to fp16.  ``scale_channels`` = (mask, factor):
    the values of the masked trailing (kv head, dim) channels are multiplied
    by ``factor`` before the fp16 rounding."""
    x = torch.randn(shape, generator=_gen(device, seed, stream), device=device,
                    dtype=torch.float32)
    if scale_channels is not None:
        mask, factor = scale_channels
        x = torch.where(mask.to(device), x * factor, x)
    return x.to(torch.float16)


def outlier_mask(w: Workload, side: int) -> torch.Tensor | None:
    """bool [n_kv, 128]: the outlier channels of one side (None if none)."""
    if w.outlier_frac <= 0:
        return None
    n = int(round(w.outlier_frac * w.n_kv * HEAD_DIM))
    rng = np.random.default_rng(w.seed * 10 + side)
    idx = rng.choice(w.n_kv * HEAD_DIM, size=n, replace=False)
    m = torch.zeros(w.n_kv * HEAD_DIM, dtype=torch.bool)
    m[torch.from_numpy(idx)] = True
    return m.view(w.n_kv, HEAD_DIM)


_BLOCK = 4096


def kv_rows(w: Workload, layer: int, side: int, seq: int, start: int, count: int,
            device="cpu") -> torch.Tensor:
    """fp16 [count, n_kv, 128]: the K (side 0) or V (side 1) rows of tokens
    start..start+count-1 of one sequence.  Rows are drawn in 4096-token blocks
    keyed by (layer, side, seq, block), so any token range can be re-drawn."""
    out = torch.empty((count, w.n_kv, HEAD_DIM), dtype=torch.float16, device=device)
    mask = outlier_mask(w, side)
    sc = (mask, w.outlier_scale) if mask is not None else None
    t = start
    while t < start + count:
        blk = t // _BLOCK
        b0 = blk * _BLOCK
        key = ((layer * 2 + side) * 64 + seq) * 4096 + blk
        rows = normal_fp16((_BLOCK, w.n_kv, HEAD_DIM), w.seed, 1 + key, device, sc)
        lo = t - b0
        hi = min(_BLOCK, start + count - b0)
        out[t - start:t - start + hi - lo] = rows[lo:hi]
        t = b0 + hi
    return out


def queries(w: Workload, layer: int, n_tok: int, device="cpu") -> torch.Tensor:
    """fp16 [n_seqs, n_tok, n_q, 128] query rows of one layer."""
    return normal_fp16((w.n_seqs, n_tok, w.n_q, HEAD_DIM), w.seed, 900_000 + layer, device)


def page_table(w: Workload):
    """(block table int32 [n_seqs][capacity/256], pool pages) of a paged
    workload: every page a sequence uses (final lengths) mapped to a distinct
    pool page, in an order shuffled from the workload's page seed; unused
    pages -1."""
    pps = w.capacity // 256
    need = [(n + 255) // 256 for n in w.final_lens()]
    n_pages = int(sum(need) * 1.05) + 1
    pages = np.random.default_rng(w.extra["page_seed"]).permutation(n_pages)
    t = -np.ones((w.n_seqs, pps), np.int32)
    k = 0
    for s in range(w.n_seqs):
        t[s, :need[s]] = pages[k:k + need[s]]
        k += need[s]
    return t, n_pages
