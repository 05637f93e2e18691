"""Probe-scored eviction on the GPU (the "Sparse KV eviction" item of the
"How It Works" section of the GitHot listing of VITRIOL): probe scores within the derived tolerance of
the oracle's fp64 probe mass, selections identical to the oracle's on
oracle-side scores, compacted caches bit-exact against the oracle's
compaction, and the whole decode -> probe -> select -> compact -> decode
loop against the oracle.

Tolerance of the probe (fp32 on the GPU, fp64 in the oracle): each weight is
exp2(s * scale * log2(e) - lse * log2(e)) with s an fp32 tensor-core dot
product of exact operands (|error| < 2^-22 * scale * log2(e) * sum |q_i k_i|,
about 1e-5 in log2 units at head_dim 128) and lse the decode's fp32
log-sum-exp (about 2 ulp of |lse| plus the relative error of its fp32 sum,
both below 1e-5); ex2.approx adds 2^-22 relative and the fp32 sums over at
most 64 heads 64 * 2^-24.  The relative error of a token's mass is therefore
below 2e-5; the tests allow 1e-4 * mass.  The decayed update is one fused
multiply-add: 2^-24 * |score| more.  Over turbo4 keys the kernels use the
rotated query H (s q) / 16, computed in fp32 and carried as an fp16 pair
(high and low halves, within 2^-22 of the fp32 value), so the same bound
holds.
"""
import math

import numpy as np
import pytest
import torch

import attention_quantized_kv_gb300 as kvq

import oracle
from tests._helpers import tol

pytestmark = pytest.mark.gpu

MASS_RTOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    from attention_quantized_kv_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _rows(rng, n_seqs, n_tok, n_kv, outlier=True):
    x = rng.standard_normal((n_seqs, n_tok, n_kv, 128))
    if outlier:
        x[..., 7] *= 8.0
    return x.astype(np.float16)


def _caches(ck, cv, n_seqs, n_kv, n_q, cap, lens, kr, vr, n_pages=0, table=None):
    """(GPU layer filled by the append kernel, oracle K bytes, oracle V bytes)."""
    ok = np.zeros(oracle.cache_bytes(ck, n_seqs, n_kv, cap), np.uint8)
    ov = np.zeros(oracle.cache_bytes(cv, n_seqs, n_kv, cap), np.uint8)
    oracle.append_side(ck, 0, ok, n_seqs, n_kv, cap, [0] * n_seqs, lens, kr)
    oracle.append_side(cv, 1, ov, n_seqs, n_kv, cap, [0] * n_seqs, lens, vr)
    if n_pages:
        L = kvq.KVLayer(n_seqs, n_kv, n_q, cap, ck, cv, n_pages=n_pages,
                        block_table=torch.from_numpy(table).cuda(),
                        k_cache=torch.zeros(kvq.kvq_pool_bytes(ck, n_pages, n_kv),
                                            dtype=torch.uint8, device="cuda"),
                        v_cache=torch.zeros(kvq.kvq_pool_bytes(cv, n_pages, n_kv),
                                            dtype=torch.uint8, device="cuda"))
    else:
        L = kvq.KVLayer(n_seqs, n_kv, n_q, cap, ck, cv,
                        k_cache=torch.zeros(kvq.kvq_cache_bytes(ck, n_seqs, n_kv, cap),
                                            dtype=torch.uint8, device="cuda"),
                        v_cache=torch.zeros(kvq.kvq_cache_bytes(cv, n_seqs, n_kv, cap),
                                            dtype=torch.uint8, device="cuda"))
    kvq.kv_append_quantize(L, torch.from_numpy(kr).cuda(), torch.from_numpy(vr).cuda(),
                           torch.tensor(lens, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert L.err.item() == 0
    if n_pages:
        assert np.array_equal(L.k_cache.cpu().numpy(),
                              oracle.to_pool(ck, ok, n_seqs, n_kv, cap, table, n_pages))
    else:
        assert np.array_equal(L.k_cache.cpu().numpy(), ok)
        assert np.array_equal(L.v_cache.cpu().numpy(), ov)
    return L, ok, ov


def _decode_lse(L, q, scale):
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    ws = torch.zeros(kvq.attn_decode_workspace(L, L.capacity), dtype=torch.uint8, device="cuda")
    kvq.attn_decode(L, q, scale, out, lse, L.capacity, ws)
    return out, lse


def _table(rng, n_seqs, pps, n_pages, lens):
    need = [(ln + 255) // 256 for ln in lens]
    pages = rng.permutation(n_pages)
    t = -np.ones((n_seqs, pps), np.int32)
    k = 0
    for s in range(n_seqs):
        t[s, :need[s]] = pages[k:k + need[s]]
        k += need[s]
    return t


def _check_scores(got, old, mass, decay, lens):
    want = decay * old.astype(np.float64) + mass
    for s, ln in enumerate(lens):
        err = np.abs(got[s, :ln] - want[s, :ln])
        bound = MASS_RTOL * mass[s, :ln] + 2.0 ** -23 * np.abs(want[s, :ln]) + 1e-12
        assert (err <= bound).all(), f"seq {s}: worst excess {(err - bound).max()}"
        assert np.array_equal(got[s, ln:], old[s, ln:]), "entries past the length changed"


@pytest.mark.parametrize("ck", [0, 1, 2, 3])
@pytest.mark.parametrize("n_kv,n_q", [(2, 10), (1, 12), (3, 3)])
def test_probe_scores_match_oracle(ck, n_kv, n_q):
    """Ragged lengths (one token, inside a unit, several pages), groups of 5,
    12 (two head groups, the second partial) and 1 query heads."""
    n_seqs, cap = 3, 1024
    lens = [1, 300, 777]
    rng = np.random.default_rng(80 + 7 * ck + n_q)
    kr, vr = _rows(rng, n_seqs, max(lens), n_kv), _rows(rng, n_seqs, max(lens), n_kv)
    L, ok, _ = _caches(ck, 1, n_seqs, n_kv, n_q, cap, lens, kr, vr)
    q = torch.from_numpy(rng.standard_normal((n_seqs, n_q, 128)).astype(np.float16)).cuda()
    scale = 1 / math.sqrt(128)
    _, lse = _decode_lse(L, q, scale)
    old = rng.uniform(0.0, 3.0, (n_seqs, cap)).astype(np.float32)
    scores = torch.from_numpy(old).cuda()
    kvq.kv_probe_scores(L, q, scale, lse, 0.75, scores)
    torch.cuda.synchronize()
    assert L.err.item() == 0
    mass = oracle.probe_mass(ck, ok, n_seqs, n_kv, n_q, cap, lens, q.cpu().numpy(), scale)
    _check_scores(scores.cpu().numpy(), old, mass, 0.75, lens)


@pytest.mark.parametrize("ck", [0, 2, 3])
def test_probe_paged_identical_to_contiguous(ck):
    n_seqs, n_kv, n_q, pps, n_pages = 3, 2, 8, 4, 16
    cap = pps * 256
    lens = [1000, 5, 513]
    rng = np.random.default_rng(90 + ck)
    table = _table(rng, n_seqs, pps, n_pages, lens)
    kr, vr = _rows(rng, n_seqs, max(lens), n_kv), _rows(rng, n_seqs, max(lens), n_kv)
    paged, ok, _ = _caches(ck, 1, n_seqs, n_kv, n_q, cap, lens, kr, vr, n_pages, table)
    flat, _, _ = _caches(ck, 1, n_seqs, n_kv, n_q, cap, lens, kr, vr)
    q = torch.from_numpy(rng.standard_normal((n_seqs, n_q, 128)).astype(np.float16)).cuda()
    scale = 1 / math.sqrt(128)
    _, lse = _decode_lse(flat, q, scale)
    res = []
    for L in (paged, flat):
        sc = torch.zeros((n_seqs, cap), dtype=torch.float32, device="cuda")
        kvq.kv_probe_scores(L, q, scale, lse, 0.5, sc)
        res.append(sc)
    torch.cuda.synchronize()
    assert paged.err.item() == 0
    assert torch.equal(res[0], res[1])
    mass = oracle.probe_mass(ck, ok, n_seqs, n_kv, n_q, cap, lens, q.cpu().numpy(), scale)
    _check_scores(res[0].cpu().numpy(), np.zeros((n_seqs, cap), np.float32), mass, 0.5, lens)


def test_probe_full_context_q4_against_oracle_and_sum():
    """The 32k-token q4_0 decode shape (32 query / 8 kv heads, 1% outlier
    channels x8): every token's mass within tolerance of the oracle, and the
    masses of each head summing to one (their total to n_q)."""
    n_seqs, n_kv, n_q, cap = 1, 8, 32, 33024
    lens = [32769]
    rng = np.random.default_rng(5)
    kr = rng.standard_normal((1, lens[0], n_kv, 128))
    vr = rng.standard_normal((1, lens[0], n_kv, 128))
    ch = rng.choice(128, 2, replace=False)
    kr[..., ch] *= 8.0
    vr[..., ch] *= 8.0
    kr, vr = kr.astype(np.float16), vr.astype(np.float16)
    L, ok, _ = _caches(2, 2, n_seqs, n_kv, n_q, cap, lens, kr, vr)
    q = torch.from_numpy(rng.standard_normal((n_seqs, n_q, 128)).astype(np.float16)).cuda()
    scale = 1 / math.sqrt(128)
    _, lse = _decode_lse(L, q, scale)
    sc = torch.zeros((n_seqs, cap), dtype=torch.float32, device="cuda")
    kvq.kv_probe_scores(L, q, scale, lse, 0.0, sc)
    got = sc.cpu().numpy()
    assert abs(got[0, :lens[0]].astype(np.float64).sum() - n_q) <= MASS_RTOL * n_q
    mass = oracle.probe_mass(2, ok, n_seqs, n_kv, n_q, cap, lens, q.cpu().numpy(), scale)
    _check_scores(got, np.zeros_like(got), mass, 0.0, lens)


def _oracle_select_all(scores, lens, n_sink, n_recent, n_evict):
    return [oracle.evict_select(scores[s], lens[s], n_sink, n_recent, n_evict)
            for s in range(len(lens))]


@pytest.mark.parametrize("case", ["ties", "spread", "signed_zero", "tiny_range"])
def test_select_matches_oracle(case):
    rng = np.random.default_rng({"ties": 1, "spread": 2, "signed_zero": 3, "tiny_range": 4}[case])
    n_seqs, cap = 5, 4096
    lens = [0, 3, 700, 4096, 2500]
    if case == "ties":  # few distinct values: the lower position wins every tie
        sc = rng.integers(0, 4, (n_seqs, cap)).astype(np.float32) * 0.25
    elif case == "spread":  # many orders of magnitude, both signs
        sc = (rng.standard_normal((n_seqs, cap)) * 10.0 ** rng.integers(-30, 30, (n_seqs, cap))
              ).astype(np.float32)
    elif case == "signed_zero":
        sc = rng.choice(np.array([-0.0, 0.0, 1.0, -1.0], np.float32), (n_seqs, cap))
    else:  # keys that differ only in the lowest bits (the last radix digit)
        sc = (1.0 + rng.integers(0, 1 << 10, (n_seqs, cap)) * 2.0 ** -23).astype(np.float32)
    scores = torch.from_numpy(sc).cuda()
    L = kvq.KVLayer(n_seqs, 1, 1, cap, 0, 0)
    L.seq_lens.copy_(torch.tensor(lens, dtype=torch.int32))
    for n_sink, n_recent, n_evict in [(4, 64, 100), (0, 0, 1), (10, 10, 5000), (3, 2, 0),
                                      (1, 0, 999)]:
        ev = torch.full((n_seqs, max(n_evict, 1)), -7, dtype=torch.int32, device="cuda")
        nev = torch.full((n_seqs,), -7, dtype=torch.int32, device="cuda")
        kvq.kv_evict_select(L, scores, n_sink, n_recent, n_evict, ev, nev)
        torch.cuda.synchronize()
        want = _oracle_select_all(sc, lens, n_sink, n_recent, n_evict)
        got_n = nev.cpu().numpy()
        got = ev.cpu().numpy()
        for s in range(n_seqs):
            assert got_n[s] == len(want[s]), (s, n_sink, n_recent, n_evict)
            assert np.array_equal(got[s, :got_n[s]], want[s]), (s, n_sink, n_recent, n_evict)


def test_select_long_sequence_against_oracle():
    """A 200704-token score row (the longest context of the workloads) with
    ties among a few thousand distinct values."""
    cap, n = 200704, 200704
    rng = np.random.default_rng(11)
    sc = (rng.integers(0, 3000, (1, cap)) * 1e-3).astype(np.float32)
    L = kvq.KVLayer(1, 1, 1, cap, 0, 0)
    L.seq_lens.fill_(n)
    ev = torch.zeros((1, 2048), dtype=torch.int32, device="cuda")
    nev = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kv_evict_select(L, torch.from_numpy(sc).cuda(), 4, 4096, 2048, ev, nev)
    want = oracle.evict_select(sc[0], n, 4, 4096, 2048)
    assert nev.item() == 2048
    assert np.array_equal(ev.cpu().numpy()[0], want)


def _evict_lists(rng, lens, kind):
    out = []
    for ln in lens:
        if ln == 0 or kind == "none":
            out.append(np.zeros(0, np.int32))
        elif kind == "random":
            k = rng.integers(0, ln + 1) // 3
            out.append(np.sort(rng.choice(ln, k, replace=False)).astype(np.int32))
        elif kind == "light":  # ~5%: a run's sources fit the stage (the pipelined path)
            out.append(np.sort(rng.choice(ln, ln // 20, replace=False)).astype(np.int32))
        elif kind == "span":  # one long run: sources jump across many units
            a = ln // 5
            out.append(np.arange(a, a + ln // 2, dtype=np.int32))
        elif kind == "sparse_keep":  # 15 of every 16 go: one source row per unit
            out.append(np.array([t for t in range(ln) if t % 16 != 3], np.int32))
        else:  # all
            out.append(np.arange(ln, dtype=np.int32))
    return out


@pytest.mark.parametrize("ck,cv", [(0, 1), (1, 2), (2, 0), (2, 2), (1, 1), (0, 0), (3, 3), (3, 1)])
@pytest.mark.parametrize("kind", ["random", "light", "span", "sparse_keep", "none", "all"])
def test_compact_bit_exact(ck, cv, kind):
    n_seqs, n_kv, n_q, cap = 4, 2, 4, 2048
    lens = [0, 37, 1500, 2048]
    rng = np.random.default_rng(100 + 3 * ck + cv)
    kr, vr = _rows(rng, n_seqs, cap, n_kv), _rows(rng, n_seqs, cap, n_kv)
    L, ok, ov = _caches(ck, cv, n_seqs, n_kv, n_q, cap, lens, kr, vr)
    evl = _evict_lists(rng, lens, kind)
    me = max(1, max(len(e) for e in evl))
    ev = np.zeros((n_seqs, me), np.int32)
    for s, e in enumerate(evl):
        ev[s, :len(e)] = e
    nev = np.array([len(e) for e in evl], np.int32)
    sc = rng.uniform(0, 1, (n_seqs, cap)).astype(np.float32)
    k_dst, v_dst = torch.zeros_like(L.k_cache), torch.zeros_like(L.v_cache)
    s_dst = torch.zeros((n_seqs, cap), dtype=torch.float32, device="cuda")
    lens_dst = torch.full((n_seqs,), -1, dtype=torch.int32, device="cuda")
    kvq.kv_compact(L, torch.from_numpy(ev).cuda(), torch.from_numpy(nev).cuda(), k_dst, v_dst,
                   torch.from_numpy(sc).cuda(), s_dst, lens_dst)
    torch.cuda.synchronize()
    assert L.err.item() == 0
    want_k = oracle.compact_side(ck, 0, ok, n_seqs, n_kv, cap, lens, evl)
    want_v = oracle.compact_side(cv, 1, ov, n_seqs, n_kv, cap, lens, evl)
    assert np.array_equal(k_dst.cpu().numpy(), want_k)
    assert np.array_equal(v_dst.cpu().numpy(), want_v)
    new_lens = [ln - len(e) for ln, e in zip(lens, evl)]
    assert lens_dst.cpu().tolist() == new_lens
    got_s = s_dst.cpu().numpy()
    for s in range(n_seqs):
        kept = np.delete(sc[s, :lens[s]], evl[s])
        assert np.array_equal(got_s[s, :new_lens[s]], kept)


@pytest.mark.parametrize("ck,cv", [(0, 1), (2, 3)])
def test_compact_many_kv_heads(ck, cv):
    """8 kv heads: each run's 16 (kv head, side) pairs cycle through the two
    stage buffers several times; light and heavy eviction mixed over the
    sequences (pipelined and round-by-round runs in one launch)."""
    n_seqs, n_kv, n_q, cap = 3, 8, 16, 2048
    lens = [2048, 1999, 700]
    rng = np.random.default_rng(400 + 3 * ck + cv)
    kr, vr = _rows(rng, n_seqs, cap, n_kv), _rows(rng, n_seqs, cap, n_kv)
    L, ok, ov = _caches(ck, cv, n_seqs, n_kv, n_q, cap, lens, kr, vr)
    evl = [np.sort(rng.choice(2048, 90, replace=False)).astype(np.int32),
           np.sort(rng.choice(1999, 700, replace=False)).astype(np.int32),
           np.arange(100, 400, dtype=np.int32)]
    me = max(len(e) for e in evl)
    ev = np.zeros((n_seqs, me), np.int32)
    for s, e in enumerate(evl):
        ev[s, :len(e)] = e
    nev = np.array([len(e) for e in evl], np.int32)
    k_dst, v_dst = torch.zeros_like(L.k_cache), torch.zeros_like(L.v_cache)
    kvq.kv_compact(L, torch.from_numpy(ev).cuda(), torch.from_numpy(nev).cuda(), k_dst, v_dst)
    torch.cuda.synchronize()
    assert L.err.item() == 0
    want_k = oracle.compact_side(ck, 0, ok, n_seqs, n_kv, cap, lens, evl)
    want_v = oracle.compact_side(cv, 1, ov, n_seqs, n_kv, cap, lens, evl)
    assert np.array_equal(k_dst.cpu().numpy(), want_k)
    assert np.array_equal(v_dst.cpu().numpy(), want_v)


def test_compact_paged_pools_bit_exact():
    n_seqs, n_kv, n_q, pps, n_pages = 3, 2, 4, 4, 14
    cap = pps * 256
    lens = [1024, 300, 700]
    rng = np.random.default_rng(120)
    table = _table(rng, n_seqs, pps, n_pages, lens)
    kr, vr = _rows(rng, n_seqs, cap, n_kv), _rows(rng, n_seqs, cap, n_kv)
    L, ok, ov = _caches(2, 1, n_seqs, n_kv, n_q, cap, lens, kr, vr, n_pages, table)
    evl = _evict_lists(rng, lens, "random")
    me = max(1, max(len(e) for e in evl))
    ev = np.zeros((n_seqs, me), np.int32)
    for s, e in enumerate(evl):
        ev[s, :len(e)] = e
    nev = np.array([len(e) for e in evl], np.int32)
    k_dst, v_dst = torch.zeros_like(L.k_cache), torch.zeros_like(L.v_cache)
    kvq.kv_compact(L, torch.from_numpy(ev).cuda(), torch.from_numpy(nev).cuda(), k_dst, v_dst)
    torch.cuda.synchronize()
    assert L.err.item() == 0
    want_k = oracle.to_pool(2, oracle.compact_side(2, 0, ok, n_seqs, n_kv, cap, lens, evl),
                            n_seqs, n_kv, cap, table, n_pages)
    want_v = oracle.to_pool(1, oracle.compact_side(1, 1, ov, n_seqs, n_kv, cap, lens, evl),
                            n_seqs, n_kv, cap, table, n_pages)
    assert np.array_equal(k_dst.cpu().numpy(), want_k)
    assert np.array_equal(v_dst.cpu().numpy(), want_v)


def test_compact_flags_a_bad_list_without_faulting():
    n_seqs, n_kv, n_q, cap = 1, 1, 1, 256
    lens = [200]
    rng = np.random.default_rng(130)
    kr, vr = _rows(rng, 1, 200, 1), _rows(rng, 1, 200, 1)
    L, _, _ = _caches(1, 2, n_seqs, n_kv, n_q, cap, lens, kr, vr)
    for bad in ([5, 3], [7, 7], [250], [-1]):
        L.err.zero_()
        ev = torch.tensor([bad], dtype=torch.int32, device="cuda")
        nev = torch.tensor([len(bad)], dtype=torch.int32, device="cuda")
        kvq.kv_compact(L, ev, nev, torch.zeros_like(L.k_cache), torch.zeros_like(L.v_cache))
        torch.cuda.synchronize()
        assert L.err.item() & kvq.KVQ_DEVERR_EVICT, bad


def test_rejects_overlapping_destinations():
    L = kvq.KVLayer(1, 1, 1, 256, 1, 1)
    ev = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    nev = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(kvq.KVQError):
        kvq.kv_compact(L, ev, nev, L.k_cache, torch.zeros_like(L.v_cache))
    with pytest.raises(kvq.KVQError):
        kvq.kv_compact(L, ev, nev, torch.zeros_like(L.k_cache), L.v_cache)
    sc = torch.zeros((1, 256), dtype=torch.float32, device="cuda")
    with pytest.raises(kvq.KVQError):  # scores compacted onto themselves
        kvq.kv_compact(L, ev, nev, torch.zeros_like(L.k_cache), torch.zeros_like(L.v_cache),
                       sc, sc)


def test_decode_probe_evict_decode_loop_matches_oracle():
    """Two rounds of decode -> probe (decayed) -> select -> compact through the
    library, then a decode over the compacted cache: the library's selection
    is a valid lowest-(score, position) choice on its own scores, and the
    final attention matches the oracle over the oracle's compaction of the
    same lists."""
    n_seqs, n_kv, n_q, cap = 2, 2, 8, 2048
    lens = [1800, 999]
    rng = np.random.default_rng(140)
    kr, vr = _rows(rng, n_seqs, max(lens), n_kv), _rows(rng, n_seqs, max(lens), n_kv)
    L, ok, ov = _caches(1, 2, n_seqs, n_kv, n_q, cap, lens, kr, vr)
    scale = 1 / math.sqrt(128)
    scores = torch.zeros((n_seqs, cap), dtype=torch.float32, device="cuda")
    cur_lens = list(lens)
    n_sink, n_recent, n_evict = 4, 128, 200
    for step in range(2):
        q = torch.from_numpy(rng.standard_normal((n_seqs, n_q, 128)).astype(np.float16)).cuda()
        _, lse = _decode_lse(L, q, scale)
        kvq.kv_probe_scores(L, q, scale, lse, 0.9, scores)
        sc_before = scores.cpu().numpy()
        scores, ev, nev = kvq.evict(L, scores, n_sink, n_recent, n_evict)
        torch.cuda.synchronize()
        assert L.err.item() == 0
        evl = []
        for s in range(n_seqs):
            e = ev.cpu().numpy()[s, :nev[s].item()]
            lo, hi = n_sink, cur_lens[s] - n_recent
            assert len(e) == min(n_evict, hi - lo)
            assert (np.diff(e) > 0).all() and e[0] >= lo and e[-1] < hi
            # a valid choice: no kept middle cell is below an evicted one in (score, t)
            mid = np.arange(lo, hi)
            kept = np.setdiff1d(mid, e)
            worst_ev = max((sc_before[s, t], t) for t in e)
            best_kept = min((sc_before[s, t], t) for t in kept)
            assert worst_ev < best_kept
            evl.append(e)
        ok = oracle.compact_side(1, 0, ok, n_seqs, n_kv, cap, cur_lens, evl)
        ov = oracle.compact_side(2, 1, ov, n_seqs, n_kv, cap, cur_lens, evl)
        cur_lens = [ln - len(e) for ln, e in zip(cur_lens, evl)]
        assert L.seq_lens.cpu().tolist() == cur_lens
        assert np.array_equal(L.k_cache.cpu().numpy(), ok)
        assert np.array_equal(L.v_cache.cpu().numpy(), ov)
    q = torch.from_numpy(rng.standard_normal((n_seqs, n_q, 128)).astype(np.float16)).cuda()
    out, _ = _decode_lse(L, q, scale)
    ro, _ = oracle.decode_layer(1, 2, ok, ov, n_seqs, n_kv, n_q, cap, cur_lens,
                                q.cpu().numpy(), scale)
    vmax = max(np.abs(oracle.dequant_stream(2, 1, ov, n_kv, cap, s, h, cur_lens[s])).max()
               for s in range(n_seqs) for h in range(n_kv))
    assert np.abs(out.float().cpu().numpy() - ro).max() <= tol(vmax)
