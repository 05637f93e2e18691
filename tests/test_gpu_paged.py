"""Paged KV (block-table pools) on the GPU: pool bytes bit-exact against the
oracle's page moves, attention identical to the contiguous layout and within
tolerance of the oracle, out-of-pool entries flagged without faults."""
import math

import numpy as np
import pytest
import torch

import attention_quantized_kv_gb300 as kvq

import oracle
from tests._helpers import tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from attention_quantized_kv_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _rows(rng, n_seqs, n_tok, n_kv):
    return rng.standard_normal((n_seqs, n_tok, n_kv, 128)).astype(np.float16)


def _table(rng, n_seqs, pps, n_pages, lens):
    """Shuffled pages for every page a sequence uses; -1 for the rest."""
    need = [(ln + 255) // 256 for ln in lens]
    pages = rng.permutation(n_pages)
    t = -np.ones((n_seqs, pps), np.int32)
    k = 0
    for s in range(n_seqs):
        t[s, :need[s]] = pages[k:k + need[s]]
        k += need[s]
    assert k <= n_pages
    return t


def _layers(ck, cv, n_seqs, n_kv, n_q, cap, n_pages, table):
    paged = kvq.KVLayer(n_seqs, n_kv, n_q, cap, ck, cv, n_pages=n_pages,
                        block_table=torch.from_numpy(table).cuda(),
                        k_cache=torch.zeros(kvq.kvq_pool_bytes(ck, n_pages, n_kv),
                                            dtype=torch.uint8, device="cuda"),
                        v_cache=torch.zeros(kvq.kvq_pool_bytes(cv, n_pages, n_kv),
                                            dtype=torch.uint8, device="cuda"))
    flat = kvq.KVLayer(n_seqs, n_kv, n_q, cap, ck, cv,
                       k_cache=torch.zeros(kvq.kvq_cache_bytes(ck, n_seqs, n_kv, cap),
                                           dtype=torch.uint8, device="cuda"),
                       v_cache=torch.zeros(kvq.kvq_cache_bytes(cv, n_seqs, n_kv, cap),
                                           dtype=torch.uint8, device="cuda"))
    return paged, flat


def _append_in_pieces(L, krows, vrows, lens, pieces):
    """Append each sequence's rows in `pieces` chunks (crossing page boundaries)."""
    n_seqs = len(lens)
    done = [0] * n_seqs
    for p in range(pieces):
        n = [(lens[s] * (p + 1)) // pieces - done[s] for s in range(n_seqs)]
        mx = max(max(n), 1)
        k = np.zeros((n_seqs, mx) + krows.shape[2:], np.float16)
        v = np.zeros_like(k)
        for s in range(n_seqs):
            k[s, :n[s]] = krows[s, done[s]:done[s] + n[s]]
            v[s, :n[s]] = vrows[s, done[s]:done[s] + n[s]]
        kvq.kv_append_quantize(L, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                               torch.tensor(n, dtype=torch.int32, device="cuda"))
        done = [done[s] + n[s] for s in range(n_seqs)]


@pytest.mark.parametrize("ck,cv", [(0, 1), (1, 1), (2, 2), (2, 0), (1, 2), (3, 3), (3, 0)])
def test_paged_append_decode_bit_exact_pools_and_identical_outputs(ck, cv):
    n_seqs, n_kv, n_q, pps, n_pages = 4, 2, 8, 6, 40
    cap = pps * 256
    lens = [1, 300, 1536, 777]  # one token, mid-page, six full pages, ragged
    rng = np.random.default_rng(60 + 3 * ck + cv)
    table = _table(rng, n_seqs, pps, n_pages, lens)
    kr, vr = _rows(rng, n_seqs, max(lens), n_kv), _rows(rng, n_seqs, max(lens), n_kv)
    paged, flat = _layers(ck, cv, n_seqs, n_kv, n_q, cap, n_pages, table)
    _append_in_pieces(paged, kr, vr, lens, 3)
    _append_in_pieces(flat, kr, vr, lens, 3)
    torch.cuda.synchronize()
    assert paged.err.item() == 0 and flat.err.item() == 0
    # pool bytes: the oracle's contiguous caches moved into pages
    for side, codec, rows in ((0, ck, kr), (1, cv, vr)):
        c = np.zeros(oracle.cache_bytes(codec, n_seqs, n_kv, cap), np.uint8)
        oracle.append_side(codec, side, c, n_seqs, n_kv, cap, [0] * n_seqs, lens, rows)
        want = oracle.to_pool(codec, c, n_seqs, n_kv, cap, table, n_pages)
        got = (paged.k_cache if side == 0 else paged.v_cache).cpu().numpy()
        assert np.array_equal(got, want), f"side {side}"
    # decode: the same bits as the contiguous layout, and the oracle bar
    q = torch.from_numpy(rng.standard_normal((n_seqs, n_q, 128)).astype(np.float16)).cuda()
    scale = 1 / math.sqrt(128)
    outs = []
    for L in (paged, flat):
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
        ws = torch.zeros(kvq.attn_decode_workspace(L, cap), dtype=torch.uint8, device="cuda")
        kvq.attn_decode(L, q, scale, out, lse, cap, ws)
        outs.append((out, lse))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    assert paged.err.item() == 0
    ok = oracle.from_pool(ck, paged.k_cache.cpu().numpy(), n_seqs, n_kv, cap, table, n_pages)
    ov = oracle.from_pool(cv, paged.v_cache.cpu().numpy(), n_seqs, n_kv, cap, table, n_pages)
    ro, rl = oracle.decode_layer(ck, cv, ok, ov, n_seqs, n_kv, n_q, cap, lens,
                                 q.cpu().numpy(), scale)
    vmax = max(np.abs(oracle.dequant_stream(cv, 1, ov, n_kv, cap, s, h, lens[s])).max()
               for s in range(n_seqs) for h in range(n_kv))
    assert np.abs(outs[0][0].float().cpu().numpy() - ro).max() <= tol(vmax)


def test_paged_prefill_matches_contiguous_and_requantize_bit_exact():
    n_seqs, n_kv, n_q, pps, n_pages = 2, 2, 8, 4, 12
    cap = pps * 256
    q_start, n_tok = 300, 200
    lens = [q_start + n_tok, 130]
    rng = np.random.default_rng(70)
    table = _table(rng, n_seqs, pps, n_pages, lens)
    kr, vr = _rows(rng, n_seqs, max(lens), n_kv), _rows(rng, n_seqs, max(lens), n_kv)
    paged, flat = _layers(1, 2, n_seqs, n_kv, n_q, cap, n_pages, table)
    for L in (paged, flat):
        _append_in_pieces(L, kr, vr, lens, 2)
    q = torch.from_numpy(rng.standard_normal((n_tok, n_q, 128)).astype(np.float16)).cuda()
    scale = 1 / math.sqrt(128)
    outs = []
    for L in (paged, flat):
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
        ws = torch.zeros(kvq.attn_prefill_workspace(L, q_start, n_tok), dtype=torch.uint8,
                         device="cuda")
        kvq.attn_prefill_chunk(L, 0, q_start, q, scale, out, lse, ws)
        outs.append((out, lse))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    # re-encode the V side of the pool: the oracle's re-encode moved into pages
    ov = oracle.from_pool(2, paged.v_cache.cpu().numpy(), n_seqs, n_kv, cap, table, n_pages)
    want = oracle.to_pool(1, oracle.requantize_side(2, 1, 1, ov, n_seqs, n_kv, cap, lens),
                          n_seqs, n_kv, cap, table, n_pages)
    kvq.degrade(paged, 1, 1)
    torch.cuda.synchronize()
    assert paged.err.item() == 0
    assert np.array_equal(paged.v_cache.cpu().numpy(), want)


@pytest.mark.parametrize("side", [0, 1])
@pytest.mark.parametrize("src,dst", [(0, 1), (1, 2), (2, 0), (0, 3)])
def test_paged_requantize_many_pages_bit_exact(src, dst, side):
    """Re-encode one side of a shuffled pool of 64 pages (three ragged
    sequences, one of them empty): every warp walks many pool units, each
    looked up in the block table, and the bytes equal the oracle's re-encode
    moved into the same pages; the other side is untouched."""
    n_seqs, n_kv, n_q, pps, n_pages = 3, 2, 4, 24, 64
    cap = pps * 256
    lens = [6000, 0, 4097]
    rng = np.random.default_rng(90 + 3 * src + dst + 11 * side)
    table = _table(rng, n_seqs, pps, n_pages, lens)
    ck, cv = (src, 1) if side == 0 else (1, src)
    kr, vr = _rows(rng, n_seqs, max(lens), n_kv), _rows(rng, n_seqs, max(lens), n_kv)
    paged, _ = _layers(ck, cv, n_seqs, n_kv, n_q, cap, n_pages, table)
    _append_in_pieces(paged, kr, vr, lens, 3)
    torch.cuda.synchronize()
    codec = ck if side == 0 else cv
    cache = paged.k_cache if side == 0 else paged.v_cache
    other = (paged.v_cache if side == 0 else paged.k_cache).clone()
    o = oracle.from_pool(codec, cache.cpu().numpy(), n_seqs, n_kv, cap, table, n_pages)
    re = oracle.requantize_side(codec, dst, side, o, n_seqs, n_kv, cap, lens)
    want = oracle.to_pool(dst, re, n_seqs, n_kv, cap, table, n_pages)
    got = torch.zeros(kvq.kvq_pool_bytes(dst, n_pages, n_kv), dtype=torch.uint8, device="cuda")
    kvq.kv_requantize(paged, side, dst, got)
    torch.cuda.synchronize()
    assert paged.err.item() == 0
    # pool units no sequence uses were not written (the oracle's pool is zero there)
    assert np.array_equal(got.cpu().numpy(), want)
    assert torch.equal(other, paged.v_cache if side == 0 else paged.k_cache)


def test_out_of_pool_entries_are_flagged_not_faulted():
    n_seqs, n_kv, n_q, pps, n_pages = 1, 1, 2, 2, 2
    cap = pps * 256
    table = np.array([[1, 5]], np.int32)  # page 1 of the sequence points past the pool
    paged, _ = _layers(1, 1, n_seqs, n_kv, n_q, cap, n_pages, table)
    rows = np.ones((1, 300, 1, 128), np.float16)
    kvq.kv_append_quantize(paged, torch.from_numpy(rows).cuda(), torch.from_numpy(rows).cuda(),
                           torch.tensor([300], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert paged.err.item() & kvq.KVQ_DEVERR_PAGE
    # the mapped page was written, the pool's other page untouched
    got = paged.k_cache.cpu().numpy().reshape(n_pages, -1)
    assert got[1].any() and not got[0].any()
    # attention over the unmapped page reads pool page 0 and still completes
    paged.err.zero_()
    q = torch.ones((1, n_q, 128), dtype=torch.float16, device="cuda")
    out = torch.empty_like(q)
    ws = torch.zeros(kvq.attn_decode_workspace(paged, cap), dtype=torch.uint8, device="cuda")
    kvq.attn_decode(paged, q, 0.1, out, None, cap, ws)
    torch.cuda.synchronize()
    assert paged.err.item() & kvq.KVQ_DEVERR_PAGE
    assert torch.isfinite(out.float()).all()
