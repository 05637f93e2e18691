"""The fused decode step (attn_decode_append) against the two-call step.

attn_decode_append must leave exactly what kv_append_quantize (one token per
sequence, lengths advanced) followed by attn_decode leaves: the same cache
bytes, the same lengths and the same outputs.  The partition of the work
depends only on the lengths, so out and lse are compared bit for bit; the
outputs are also checked against the fp64 oracle on sampled groups.
"""
import math

import numpy as np
import pytest
import torch

import attention_quantized_kv_gb300 as kvq
from attention_quantized_kv_gb300 import workloads as wl

import oracle
from tests._helpers import gpu_layer, oracle_stream

pytestmark = pytest.mark.gpu

SCALE = 1 / math.sqrt(128)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from attention_quantized_kv_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def clone_layer(L):
    M = kvq.KVLayer(L.n_seqs, L.n_kv_heads, L.n_q_heads, L.capacity, L.codec_k, L.codec_v,
                    k_cache=L.k_cache.clone(), v_cache=L.v_cache.clone(), device="cuda",
                    n_pages=L.n_pages, block_table=L.block_table)
    M.seq_lens.copy_(L.seq_lens)
    return M


def new_rows(w, lens):
    """Token lens[s] of every sequence (the next one of the seeded draws)."""
    k = torch.stack([wl.kv_rows(w, 0, 0, s, lens[s], 1, "cuda")[0] for s in range(w.n_seqs)])
    v = torch.stack([wl.kv_rows(w, 0, 1, s, lens[s], 1, "cuda")[0] for s in range(w.n_seqs)])
    return k.contiguous(), v.contiguous()


def two_call_step(L, k, v, q, max_len, ws):
    n_new = torch.ones(L.n_seqs, dtype=torch.int32, device="cuda")
    kvq.kv_append_quantize(L, k[:, None].contiguous(), v[:, None].contiguous(), n_new)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    kvq.attn_decode(L, q, SCALE, out, lse, max_len, ws)
    return out, lse


def fused_step(L, k, v, q, max_len, ws):
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    kvq.attn_decode_append(L, k, v, q, SCALE, out, lse, max_len, ws)
    return out, lse


def assert_same(A, B, oa, ob):
    torch.cuda.synchronize()
    assert torch.equal(A.seq_lens, B.seq_lens), (A.seq_lens, B.seq_lens)
    assert torch.equal(A.k_cache, B.k_cache), "K cache bytes differ"
    assert torch.equal(A.v_cache, B.v_cache), "V cache bytes differ"
    assert torch.equal(oa[0], ob[0]), "out differs"
    assert torch.equal(oa[1], ob[1]), "lse differs"
    assert int(A.err.item()) == int(B.err.item())


def check_oracle(w, B, q, out, lse, lens_after, groups):
    G = w.n_q // w.n_kv
    ck, cv = w.codecs[0]
    qn, on, ln = q.cpu().numpy(), out.float().cpu().numpy(), lse.cpu().numpy()
    for s, h in groups:
        T = lens_after[s]
        ok, ov = oracle_stream(w, 0, s, h, T)
        ro, rl = oracle.decode_layer(ck, cv, ok, ov, 1, 1, G, w.capacity, [T],
                                     qn[s, h * G:(h + 1) * G], SCALE)
        V = oracle.dequant_stream(cv, 1, ov, 1, w.capacity, 0, 0, T)
        err = np.abs(on[s, h * G:(h + 1) * G] - ro[0]).max()
        assert err <= 2e-3 * np.abs(V).max(), (s, h, err)
        assert np.abs(ln[s, h * G:(h + 1) * G] - rl[0]).max() < 1e-3


PAIRS = [(a, b) for a in (0, 1, 2, 3) for b in (0, 1, 2, 3)]


@pytest.mark.parametrize("ck,cv", PAIRS)
def test_fused_step_equals_two_calls(ck, cv):
    # new tokens land on unit and item boundaries (positions 0, 15, 16, 31, 32, ...)
    lens = [0, 1, 15, 16, 31, 32, 100, 257, 1000]
    w = wl.Workload("t", "decode", len(lens), 8, 2, lens, [(ck, cv)], 300 + 4 * ck + cv)
    A = gpu_layer(w, 0)
    B = clone_layer(A)
    k, v = new_rows(w, lens)
    q = wl.queries(w, 0, 1, "cuda")[:, 0].contiguous()
    max_len = max(lens) + 1
    wsa = torch.zeros(kvq.attn_decode_workspace(A, max_len), dtype=torch.uint8, device="cuda")
    wsb = torch.zeros_like(wsa)
    oa = two_call_step(A, k, v, q, max_len, wsa)
    ob = fused_step(B, k, v, q, max_len, wsb)
    assert_same(A, B, oa, ob)
    assert int(B.err.item()) == 0
    assert not wsb[:65536].any(), "workspace counters must be zero after the call"
    after = [n + 1 for n in lens]
    check_oracle(w, B, q, ob[0], ob[1], after, [(0, 0), (2, 1), (5, 0), (8, 1)])


@pytest.mark.parametrize("G", [1, 5, 8, 12])
def test_fused_step_group_sizes(G):
    lens = [300, 33, 4095]
    w = wl.Workload("t", "decode", 3, 2 * G, 2, lens, [(1, 2)], 50 + G)
    A = gpu_layer(w, 0)
    B = clone_layer(A)
    k, v = new_rows(w, lens)
    q = wl.queries(w, 0, 1, "cuda")[:, 0].contiguous()
    max_len = 4096
    ws = torch.zeros(kvq.attn_decode_workspace(A, max_len), dtype=torch.uint8, device="cuda")
    oa = two_call_step(A, k, v, q, max_len, ws)
    ob = fused_step(B, k, v, q, max_len, ws)
    assert_same(A, B, oa, ob)
    check_oracle(w, B, q, ob[0], ob[1], [n + 1 for n in lens], [(0, 1), (2, 0)])


def test_fused_steps_in_a_row_reuse_the_workspace():
    """40 steps (lengths cross unit, item and page boundaries) on one workspace,
    q4_0 on both sides (two-unit items)."""
    lens = [200, 5, 250]
    w = wl.Workload("t", "decode", 3, 8, 2, lens, [(2, 2)], 77, append_new=40)
    assert w.capacity == 512
    A = gpu_layer(w, 0)
    B = clone_layer(A)
    max_len = 512
    wsa = torch.zeros(kvq.attn_decode_workspace(A, max_len), dtype=torch.uint8, device="cuda")
    wsb = torch.zeros_like(wsa)
    cur = list(lens)
    for step in range(40):
        k, v = new_rows(w, cur)
        q = (torch.randn((3, 8, 128), generator=torch.Generator().manual_seed(step)) * 1.0
             ).to(torch.float16).cuda()
        oa = two_call_step(A, k, v, q, max_len, wsa)
        ob = fused_step(B, k, v, q, max_len, wsb)
        assert_same(A, B, oa, ob)
        cur = [n + 1 for n in cur]
    assert B.seq_lens.tolist() == cur
    check_oracle(w, B, q, ob[0], ob[1], cur, [(0, 0), (1, 1), (2, 0)])


def test_fused_step_many_empty_ctas():
    """Short sequences under a large max_len: most CTAs get an empty slice and
    only count themselves; the lengths still advance exactly once."""
    lens = [0, 1, 2, 3]
    w = wl.Workload("t", "decode", 4, 8, 2, lens, [(0, 1)], 91, append_new=8189)
    assert w.capacity == 8192
    A = gpu_layer(w, 0)
    B = clone_layer(A)
    k, v = new_rows(w, lens)
    q = wl.queries(w, 0, 1, "cuda")[:, 0].contiguous()
    max_len = 8192
    ws = torch.zeros(kvq.attn_decode_workspace(A, max_len), dtype=torch.uint8, device="cuda")
    oa = two_call_step(A, k, v, q, max_len, ws)
    ob = fused_step(B, k, v, q, max_len, ws)
    assert_same(A, B, oa, ob)
    assert B.seq_lens.tolist() == [1, 2, 3, 4]
    assert not ws[:65536].any()


def test_fused_step_at_capacity():
    """A full sequence gets no token (KVQ_DEVERR_CAPACITY) and attends its keys."""
    lens = [256, 100]
    w = wl.Workload("t", "decode", 2, 8, 2, lens, [(1, 1)], 5)
    assert w.capacity == 256
    A = gpu_layer(w, 0)
    B = clone_layer(A)
    k, v = new_rows(w, [0, 100])
    q = wl.queries(w, 0, 1, "cuda")[:, 0].contiguous()
    ws = torch.zeros(kvq.attn_decode_workspace(A, 256), dtype=torch.uint8, device="cuda")
    oa = two_call_step(A, k, v, q, 256, ws)
    ob = fused_step(B, k, v, q, 256, ws)
    assert_same(A, B, oa, ob)
    assert B.seq_lens.tolist() == [256, 101]
    assert int(B.err.item()) & kvq.KVQ_DEVERR_CAPACITY


def test_fused_step_paged():
    """Paged layer over a shuffled pool: the same bytes and outputs as the
    two-call step on the same pool."""
    lens = [255, 256, 700]
    w = wl.Workload("t", "decode", 3, 8, 2, lens, [(2, 1)], 13)
    pps = w.capacity // 256
    n_pages = 3 * pps + 2
    perm = np.random.default_rng(4).permutation(n_pages)[:3 * pps].astype(np.int32)
    table = torch.from_numpy(perm.reshape(3, pps)).cuda()
    ck, cv = w.codecs[0]
    A = kvq.KVLayer(3, 2, 8, w.capacity, ck, cv, device="cuda", n_pages=n_pages, block_table=table)
    A.k_cache.zero_()
    A.v_cache.zero_()
    mx = max(lens)
    kk = torch.zeros((3, mx, 2, 128), dtype=torch.float16, device="cuda")
    vv = torch.zeros_like(kk)
    for s in range(3):
        kk[s, :lens[s]] = wl.kv_rows(w, 0, 0, s, 0, lens[s], "cuda")
        vv[s, :lens[s]] = wl.kv_rows(w, 0, 1, s, 0, lens[s], "cuda")
    kvq.kv_append_quantize(A, kk, vv, torch.tensor(lens, dtype=torch.int32, device="cuda"))
    B = clone_layer(A)
    k, v = new_rows(w, lens)
    q = wl.queries(w, 0, 1, "cuda")[:, 0].contiguous()
    assert w.capacity == 768
    ws = torch.zeros(kvq.attn_decode_workspace(A, 768), dtype=torch.uint8, device="cuda")
    oa = two_call_step(A, k, v, q, 768, ws)
    ob = fused_step(B, k, v, q, 768, ws)
    assert_same(A, B, oa, ob)


def test_fused_step_full_size_q4():
    """The 32,768-token q4_0 workload with outlier channels (32 query / 8 kv
    heads): one fused step equals the two-call step."""
    w = wl.get("append_decode_q4_ctx32k")
    A = gpu_layer(w, 0, chunk=8192)
    B = clone_layer(A)
    k, v = new_rows(w, w.lens)
    q = wl.queries(w, 0, 1, "cuda")[:, 0].contiguous()
    max_len = w.lens[0] + 1
    ws = torch.zeros(kvq.attn_decode_workspace(A, max_len), dtype=torch.uint8, device="cuda")
    oa = two_call_step(A, k, v, q, max_len, ws)
    ob = fused_step(B, k, v, q, max_len, ws)
    assert_same(A, B, oa, ob)
    check_oracle(w, B, q, ob[0], ob[1], [w.lens[0] + 1], [(0, 0), (0, 7)])


def test_fused_step_argument_checks():
    w = wl.Workload("t", "decode", 1, 8, 2, [10], [(1, 1)], 1)
    L = gpu_layer(w, 0)
    q = torch.zeros((1, 8, 128), dtype=torch.float16, device="cuda")
    k = torch.zeros((1, 2, 128), dtype=torch.float16, device="cuda")
    ws = torch.zeros(kvq.attn_decode_workspace(L, 64), dtype=torch.uint8, device="cuda")
    with pytest.raises(kvq.KVQError):
        kvq.attn_decode_append(L, k, k, q, SCALE, torch.empty_like(q), None, 64, ws[:16])
    with pytest.raises(kvq.KVQError):
        kvq.attn_decode_append(L, k, k, q, SCALE, torch.empty_like(q), None, L.capacity + 1, ws)


@pytest.mark.parametrize("ck,cv", [(1, 2), (2, 2), (0, 3)])
def test_fused_step_many_short_sequences(ck, cv):
    """1024 short sequences (the per-call maximum): every CTA holds several
    stream ends and some warps several new-row items; two steps in a row."""
    rng = np.random.default_rng(11 + ck)
    lens = [int(x) for x in rng.integers(0, 90, 1024)]
    w = wl.Workload("t", "decode", 1024, 4, 2, lens, [(ck, cv)], 500 + ck, append_new=2)
    A = gpu_layer(w, 0, chunk=256)
    B = clone_layer(A)
    max_len = max(lens) + 2
    wsa = torch.zeros(kvq.attn_decode_workspace(A, max_len), dtype=torch.uint8, device="cuda")
    wsb = torch.zeros_like(wsa)
    cur = list(lens)
    for step in range(2):
        k, v = new_rows(w, cur)
        q = (torch.randn((1024, 4, 128), generator=torch.Generator().manual_seed(step))
             ).to(torch.float16).cuda()
        oa = two_call_step(A, k, v, q, max_len, wsa)
        ob = fused_step(B, k, v, q, max_len, wsb)
        assert_same(A, B, oa, ob)
        cur = [n + 1 for n in cur]
    assert B.seq_lens.tolist() == cur
    assert not wsb[:65536].any()
    check_oracle(w, B, q, ob[0], ob[1], cur, [(0, 0), (511, 1), (1023, 0)])
