"""Quantize-on-append on the GPU: cache bytes bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import attention_quantized_kv_gb300 as kvq
from attention_quantized_kv_gb300 import workloads as wl

import oracle
from tests._helpers import boundary_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from attention_quantized_kv_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


CODECS = [(0, 0), (1, 1), (2, 2), (0, 1), (1, 2), (2, 0), (3, 3), (3, 0), (1, 3)]


@pytest.mark.parametrize("ck,cv", CODECS)
def test_ragged_appends_bit_exact(ck, cv):
    """Several appends of ragged sizes starting mid-unit, every codec on both sides."""
    torch.manual_seed(0)
    n_seqs, n_kv, n_q, cap = 3, 2, 4, 512
    L = kvq.KVLayer(n_seqs, n_kv, n_q, cap, ck, cv,
                    k_cache=torch.zeros(kvq.kvq_cache_bytes(ck, n_seqs, n_kv, cap),
                                        dtype=torch.uint8, device="cuda"),
                    v_cache=torch.zeros(kvq.kvq_cache_bytes(cv, n_seqs, n_kv, cap),
                                        dtype=torch.uint8, device="cuda"))
    ok = np.zeros(oracle.cache_bytes(ck, n_seqs, n_kv, cap), np.uint8)
    ov = np.zeros(oracle.cache_bytes(cv, n_seqs, n_kv, cap), np.uint8)
    lens = np.zeros(n_seqs, np.int32)
    rng = np.random.default_rng(ck * 3 + cv)
    for step, n_new in enumerate(([1, 0, 17], [16, 33, 5], [40, 1, 100], [3, 64, 1])):
        mx = max(n_new)
        scale = [1.0, 1e-4, 300.0, 8.0][step]
        k = (torch.randn((n_seqs, mx, n_kv, 128), device="cuda") * scale).half()
        v = (torch.randn((n_seqs, mx, n_kv, 128), device="cuda") * scale).half()
        if step == 3:  # zero blocks and signed ties
            k[0, 0, 0, :32] = 0
            v[0, 0, 0, 32:64] = 0
            k[1, 0, 1, :32] = torch.tensor([1.0, -1.0] * 16)
            v[1, 1, 1, 64:96] = torch.tensor([-2.0, 2.0] * 16)
        nn = torch.tensor(n_new, dtype=torch.int32, device="cuda")
        kvq.kv_append_quantize(L, k, v, nn)
        oracle.append_side(ck, 0, ok, n_seqs, n_kv, cap, lens, n_new, k.cpu().numpy())
        oracle.append_side(cv, 1, ov, n_seqs, n_kv, cap, lens, n_new, v.cpu().numpy())
        lens += np.array(n_new, np.int32)
    torch.cuda.synchronize()
    assert np.array_equal(L.seq_lens.cpu().numpy(), lens)
    assert L.err.item() == 0
    gk, gv = L.k_cache.cpu().numpy(), L.v_cache.cpu().numpy()
    assert np.array_equal(gk, ok), f"K bytes differ at {np.flatnonzero(gk != ok)[:10]}"
    assert np.array_equal(gv, ov), f"V bytes differ at {np.flatnonzero(gv != ov)[:10]}"


def test_append_leaves_other_bytes_untouched_and_flags_capacity():
    n_seqs, n_kv, cap = 2, 1, 256
    L = kvq.KVLayer(n_seqs, n_kv, 1, cap, 1, 2,
                    k_cache=torch.full((kvq.kvq_cache_bytes(1, n_seqs, n_kv, cap),), 0xAB,
                                       dtype=torch.uint8, device="cuda"),
                    v_cache=torch.full((kvq.kvq_cache_bytes(2, n_seqs, n_kv, cap),), 0xAB,
                                       dtype=torch.uint8, device="cuda"))
    L.seq_lens.copy_(torch.tensor([250, 7], dtype=torch.int32))
    k = torch.randn((n_seqs, 10, n_kv, 128), device="cuda").half()
    nn = torch.tensor([10, 3], dtype=torch.int32, device="cuda")
    kvq.kv_append_quantize(L, k, k.clone(), nn)
    torch.cuda.synchronize()
    assert L.err.item() & kvq.KVQ_DEVERR_CAPACITY
    # rows 250..255 of seq 0 and 7..9 of seq 1 were written; everything else kept 0xAB
    tab_k = oracle.unit_offset_table(1, 0)
    gk = L.k_cache.cpu().numpy().reshape(n_seqs, cap // 16, 16 * 136)
    written = np.zeros_like(gk, bool)
    for s, rows in ((0, range(250, 256)), (1, range(7, 10))):
        for p in rows:
            written[s, p // 16, tab_k[p % 16]] = True
    assert np.all(gk[~written] == 0xAB)
    assert L.seq_lens.cpu().tolist() == [256, 10]


def test_decode_workload_fill_matches_oracle_stream():
    """The chunked fill used by the parity tests: one stream, byte for byte."""
    w = wl.get("decode_q8_ctx4k")
    from tests._helpers import gpu_layer, oracle_stream, gpu_stream_bytes
    L = gpu_layer(w, 0, chunk=1000)
    for kvh in range(w.n_kv):
        ok, ov = oracle_stream(w, 0, 0, kvh, w.lens[0])
        # the oracle's 1x1 stream holds the same bytes as this stream of the layer
        assert np.array_equal(gpu_stream_bytes(L, 0, 0, kvh), ok)
        assert np.array_equal(gpu_stream_bytes(L, 1, 0, kvh), ov)


@pytest.mark.parametrize("codec", [1, 2])
def test_rounding_boundary_rows_bit_exact(codec):
    """Quotients at the encoders' rounding boundaries (the exact-division path
    of the encoders) on both sides: bytes identical to the oracle."""
    rng = np.random.default_rng(40 + codec)
    n_seqs, n_kv, n_q, cap, n = 1, 2, 4, 256, 48
    L = kvq.KVLayer(n_seqs, n_kv, n_q, cap, codec, codec,
                    k_cache=torch.zeros(kvq.kvq_cache_bytes(codec, n_seqs, n_kv, cap),
                                        dtype=torch.uint8, device="cuda"),
                    v_cache=torch.zeros(kvq.kvq_cache_bytes(codec, n_seqs, n_kv, cap),
                                        dtype=torch.uint8, device="cuda"))
    x = boundary_rows(codec, n_seqs * n * n_kv, rng).reshape(n_seqs, n, n_kv, 128)
    xt = torch.from_numpy(x).cuda()
    kvq.kv_append_quantize(L, xt, xt, torch.tensor([n], dtype=torch.int32, device="cuda"))
    ok = np.zeros(oracle.cache_bytes(codec, n_seqs, n_kv, cap), np.uint8)
    ov = np.zeros_like(ok)
    oracle.append_side(codec, 0, ok, n_seqs, n_kv, cap, [0], [n], x)
    oracle.append_side(codec, 1, ov, n_seqs, n_kv, cap, [0], [n], x)
    torch.cuda.synchronize()
    assert np.array_equal(L.k_cache.cpu().numpy(), ok)
    assert np.array_equal(L.v_cache.cpu().numpy(), ov)
