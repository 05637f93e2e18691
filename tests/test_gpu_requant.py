"""Degrade ladder on the GPU: re-encoded cache bytes bit-exact against the
oracle, and attention over a model walked down the banded ladder."""
import math

import numpy as np
import pytest
import torch

import attention_quantized_kv_gb300 as kvq
from attention_quantized_kv_gb300 import workloads as wl

import oracle
from tests._helpers import gpu_layer, tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from attention_quantized_kv_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _rows(rng, n_seqs, n_tok, n_kv, scales):
    x = rng.standard_normal((n_seqs, n_tok, n_kv, 128)) * np.asarray(scales)[:, None, None, None]
    x[..., 5] *= 8.0  # an outlier channel
    return x.astype(np.float16)


@pytest.mark.parametrize("side", [0, 1])
@pytest.mark.parametrize("src,dst", [(a, b) for a in (0, 1, 2, 3) for b in (0, 1, 2, 3)])
def test_requantize_bit_exact(src, dst, side):
    n_seqs, n_kv, cap = 3, 2, 512
    lens = [0, 37, 300]  # empty, ragged inside a unit, several units
    rng = np.random.default_rng(20 + 3 * src + dst + 9 * side)
    rows = _rows(rng, n_seqs, max(lens), n_kv, [1.0, 1e-3, 40.0])
    # oracle: append with the source codec, then re-encode
    o_src = np.zeros(oracle.cache_bytes(src, n_seqs, n_kv, cap), np.uint8)
    oracle.append_side(src, side, o_src, n_seqs, n_kv, cap, [0] * n_seqs, lens, rows)
    o_dst = oracle.requantize_side(src, dst, side, o_src, n_seqs, n_kv, cap, lens)
    # GPU: the same appends through the library, then kv_requantize
    ck, cv = (src, 1) if side == 0 else (1, src)
    L = kvq.KVLayer(n_seqs, n_kv, 2 * n_kv, cap, ck, cv,
                    k_cache=torch.zeros(kvq.kvq_cache_bytes(ck, n_seqs, n_kv, cap),
                                        dtype=torch.uint8, device="cuda"),
                    v_cache=torch.zeros(kvq.kvq_cache_bytes(cv, n_seqs, n_kv, cap),
                                        dtype=torch.uint8, device="cuda"))
    x = torch.from_numpy(rows).cuda()
    kvq.kv_append_quantize(L, x, x, torch.tensor(lens, dtype=torch.int32, device="cuda"))
    src_gpu = (L.k_cache if side == 0 else L.v_cache).cpu().numpy()
    assert np.array_equal(src_gpu, o_src)
    dst_gpu = torch.zeros(kvq.kvq_cache_bytes(dst, n_seqs, n_kv, cap), dtype=torch.uint8,
                          device="cuda")
    kvq.kv_requantize(L, side, dst, dst_gpu)
    torch.cuda.synchronize()
    assert L.err.item() == 0
    assert np.array_equal(dst_gpu.cpu().numpy(), o_dst)


@pytest.mark.parametrize("side", [0, 1])
@pytest.mark.parametrize("src,dst", [(0, 1), (0, 2), (1, 2), (2, 0), (1, 1)])
def test_requantize_many_runs_per_cta(src, dst, side):
    """Thousands of 64-token runs, more than the persistent grid holds at
    once, mostly empty ones (a whole empty sequence, a short one) between
    long streams with a partial last unit: every CTA walks several runs
    through both buffers each way."""
    n_seqs, n_kv, cap = 3, 2, 40960
    lens = [0, 37, 40001]
    rng = np.random.default_rng(70 + 3 * src + dst + 9 * side)
    rows = _rows(rng, n_seqs, max(lens), n_kv, [1.0, 1e-3, 40.0])
    o_src = np.zeros(oracle.cache_bytes(src, n_seqs, n_kv, cap), np.uint8)
    oracle.append_side(src, side, o_src, n_seqs, n_kv, cap, [0] * n_seqs, lens, rows)
    o_dst = oracle.requantize_side(src, dst, side, o_src, n_seqs, n_kv, cap, lens)
    ck, cv = (src, 1) if side == 0 else (1, src)
    L = kvq.KVLayer(n_seqs, n_kv, 2 * n_kv, cap, ck, cv,
                    k_cache=torch.zeros(kvq.kvq_cache_bytes(ck, n_seqs, n_kv, cap),
                                        dtype=torch.uint8, device="cuda"),
                    v_cache=torch.zeros(kvq.kvq_cache_bytes(cv, n_seqs, n_kv, cap),
                                        dtype=torch.uint8, device="cuda"))
    x = torch.from_numpy(rows).cuda()
    kvq.kv_append_quantize(L, x, x, torch.tensor(lens, dtype=torch.int32, device="cuda"))
    assert np.array_equal((L.k_cache if side == 0 else L.v_cache).cpu().numpy(), o_src)
    # bytes past the lengths must survive: start the destination from a pattern
    dst_gpu = torch.full((kvq.kvq_cache_bytes(dst, n_seqs, n_kv, cap),), 0xA5, dtype=torch.uint8,
                         device="cuda")
    kvq.kv_requantize(L, side, dst, dst_gpu)
    torch.cuda.synchronize()
    assert L.err.item() == 0
    # expected: the oracle's bytes for rows below the length, the pattern for
    # every other byte (the row of each unit byte from the oracle's layout)
    ub = oracle.cache_bytes(dst, 1, 1, 16)
    row_of = np.empty(ub, np.int32)
    table = oracle.unit_offset_table(dst, side)
    for r in range(16):
        row_of[table[r]] = r
    tok = (np.arange(cap // 16)[:, None] * 16 + row_of[None, :]).reshape(-1)  # per stream byte
    want = np.full(o_dst.shape, 0xA5, np.uint8)
    per_stream = (cap // 16) * ub
    for s_ in range(n_seqs):
        for h in range(n_kv):
            base = (s_ * n_kv + h) * per_stream
            keep = tok < lens[s_]
            want[base:base + per_stream][keep] = o_dst[base:base + per_stream][keep]
    np.testing.assert_array_equal(dst_gpu.cpu().numpy(), want)


def test_requantize_rejects_overlap_and_bad_arguments():
    L = kvq.KVLayer(1, 1, 1, 256, 0, 0)
    with pytest.raises(kvq.KVQError):
        kvq.kv_requantize(L, 0, 1, L.k_cache[:kvq.kvq_cache_bytes(1, 1, 1, 256)])
    dst = torch.zeros(kvq.kvq_cache_bytes(1, 1, 1, 256), dtype=torch.uint8, device="cuda")
    with pytest.raises(kvq.KVQError):
        kvq.kv_requantize(L, 2, 1, dst)
    with pytest.raises(ValueError):  # no cache size for an unknown codec
        kvq.kv_requantize(L, 0, 7, dst)


def test_ladder_walk_decode_matches_oracle_at_every_band():
    """A 2-layer model (4 tensors) walked down the banded ladder by the
    library's planner; after each step every layer's decode matches the oracle
    run over the oracle's own degraded caches, and the planner agrees with the
    oracle's."""
    n_layers, n_seqs, n_kv, n_q, cap = 2, 2, 2, 8, 512
    lens = [200, 77]
    rng = np.random.default_rng(31)
    rows = [[_rows(rng, n_seqs, max(lens), n_kv, [1.0, 2.0]) for _ in range(2)]
            for _ in range(n_layers)]
    q = (rng.standard_normal((n_layers, n_seqs, n_q, 128))).astype(np.float16)
    scale = 1 / math.sqrt(128)
    codecs = [0] * (2 * n_layers)   # tensor t = 2 * layer + side
    layers, ocaches = [], []
    for l in range(n_layers):
        L = kvq.KVLayer(n_seqs, n_kv, n_q, cap, 0, 0,
                        k_cache=torch.zeros(kvq.kvq_cache_bytes(0, n_seqs, n_kv, cap),
                                            dtype=torch.uint8, device="cuda"),
                        v_cache=torch.zeros(kvq.kvq_cache_bytes(0, n_seqs, n_kv, cap),
                                            dtype=torch.uint8, device="cuda"))
        kvq.kv_append_quantize(L, torch.from_numpy(rows[l][0]).cuda(),
                               torch.from_numpy(rows[l][1]).cuda(),
                               torch.tensor(lens, dtype=torch.int32, device="cuda"))
        layers.append(L)
        oc = []
        for side in (0, 1):
            c = np.zeros(oracle.cache_bytes(0, n_seqs, n_kv, cap), np.uint8)
            oracle.append_side(0, side, c, n_seqs, n_kv, cap, [0] * n_seqs, lens, rows[l][side])
            oc.append(c)
        ocaches.append(oc)
    order = [3, 1, 2, 0]   # a price order: V sides first
    steps = 0
    while True:
        step = kvq.ladder_next(codecs, 4.5, order)
        assert step == oracle.ladder_next(codecs, order, 4.5)
        if step is None:
            break
        t, k = step
        l, side = divmod(t, 2)
        kvq.degrade(layers[l], side, k)
        ocaches[l][side] = oracle.requantize_side(codecs[t], k, side, ocaches[l][side], n_seqs,
                                                  n_kv, cap, lens)
        codecs[t] = k
        steps += 1
        assert abs(kvq.aggregate_bpv(codecs) - oracle.aggregate_bpv(codecs)) == 0
        for ll in range(n_layers):
            L = layers[ll]
            got_bytes = (L.k_cache if side == 0 else L.v_cache).cpu().numpy()
            if ll == l:
                assert np.array_equal(got_bytes, ocaches[l][side])
            qq = torch.from_numpy(q[ll]).cuda()
            out = torch.empty_like(qq)
            lse = torch.empty(qq.shape[:2], dtype=torch.float32, device="cuda")
            ws = torch.zeros(kvq.attn_decode_workspace(L, max(lens)), dtype=torch.uint8,
                             device="cuda")
            kvq.attn_decode(L, qq, scale, out, lse, max(lens), ws)
            ro, rl = oracle.decode_layer(L.codec_k, L.codec_v, ocaches[ll][0], ocaches[ll][1],
                                         n_seqs, n_kv, n_q, cap, lens, q[ll], scale)
            vmax = max(np.abs(oracle.dequant_stream(L.codec_v, 1, ocaches[ll][1], n_kv, cap, s,
                                                    h, lens[s])).max()
                       for s in range(n_seqs) for h in range(n_kv))
            assert np.abs(out.float().cpu().numpy() - ro).max() <= tol(vmax)
    assert steps == 2 * len(order) and codecs == [2] * 4


def test_requantize_full_size_ladder_layer_sampled():
    """One side of a 2 x 200,704-key layer, f16 -> q8_0 -> q4_0, checked
    against the oracle on sampled (seq, kv head) streams."""
    w = wl.get("decode_16layer_ladder_2x200704")
    w = wl.Workload("t", "decode", w.n_seqs, w.n_q, w.n_kv, w.lens, [(0, 0)], 3)
    L = gpu_layer(w, 0)
    cap = w.capacity
    for side, (a, b) in ((0, (0, 1)), (1, (0, 2))):
        dst = torch.zeros(kvq.kvq_cache_bytes(b, w.n_seqs, w.n_kv, cap), dtype=torch.uint8,
                          device="cuda")
        kvq.kv_requantize(L, side, b, dst)
        torch.cuda.synchronize()
        for s, h in ((0, 0), (1, 3)):
            n = w.lens[s]
            x = wl.kv_rows(w, 0, side, s, 0, n, "cuda")[:, h].cpu().numpy().reshape(1, n, 1, 128)
            o_src = np.zeros(oracle.cache_bytes(a, 1, 1, cap), np.uint8)
            oracle.append_side(a, side, o_src, 1, 1, cap, [0], [n], x)
            o_dst = oracle.requantize_side(a, b, side, o_src, 1, 1, cap, [n])
            per = cap * {0: 256, 1: 136, 2: 72}[b]
            got = dst[(s * w.n_kv + h) * per:(s * w.n_kv + h + 1) * per].cpu().numpy()
            assert np.array_equal(got, o_dst), f"side {side} stream ({s}, {h})"
