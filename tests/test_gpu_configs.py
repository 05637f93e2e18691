"""The benchmark workloads at full size, in the launch configuration bench.py
times (same plan: max_len = the longest sequence), checked against the
oracle: every (sequence, kv head) group of every layer, whole caches compared
byte for byte, outputs within 2e-3 * max|V^| of each group and lse within
1e-3."""
import math

import numpy as np
import pytest
import torch

import attention_quantized_kv_gb300 as kvq
from attention_quantized_kv_gb300 import workloads as wl

import oracle
from tests._helpers import gpu_layer, gpu_stream_bytes, oracle_layer, oracle_stream

pytestmark = pytest.mark.gpu
SCALE = 1 / math.sqrt(128)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from attention_quantized_kv_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _decode(L, q, max_len):
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    ws = torch.zeros(kvq.attn_decode_workspace(L, max_len), dtype=torch.uint8, device=q.device)
    kvq.attn_decode(L, q, SCALE, out, lse, max_len, ws)
    torch.cuda.synchronize()
    return out, lse


def _check_groups(w, layer_idx, L, q, out, lse, groups, lens):
    G = w.n_q // w.n_kv
    ck, cv = w.codecs[layer_idx]
    qn, on, ln = q.cpu().numpy(), out.float().cpu().numpy(), lse.cpu().numpy()
    for s, h in groups:
        T = lens[s]
        ok, ov = oracle_stream(w, layer_idx, s, h, T)
        assert np.array_equal(gpu_stream_bytes(L, 0, s, h), ok), f"K bytes (seq {s}, kvh {h})"
        assert np.array_equal(gpu_stream_bytes(L, 1, s, h), ov), f"V bytes (seq {s}, kvh {h})"
        ro, rl = oracle.decode_layer(ck, cv, ok, ov, 1, 1, G, w.capacity, [T],
                                     qn[s, h * G:(h + 1) * G], SCALE)
        vmax = np.abs(oracle.dequant_stream(cv, 1, ov, 1, w.capacity, 0, 0, T)).max()
        err = np.abs(on[s, h * G:(h + 1) * G] - ro[0]).max()
        assert err <= 2e-3 * vmax, f"layer {layer_idx} seq {s} kvh {h}: {err} > {2e-3 * vmax}"
        assert np.abs(ln[s, h * G:(h + 1) * G] - rl[0]).max() < 1e-3


def test_decode_q8_ctx4k_full():
    w = wl.get("decode_q8_ctx4k")
    L = gpu_layer(w, 0)
    q = wl.queries(w, 0, 1, "cuda")[:, 0].contiguous()
    out, lse = _decode(L, q, max(w.lens))
    _check_groups(w, 0, L, q, out, lse, [(0, 0), (0, 1)], w.lens)


def test_append_decode_q4_ctx32k_full():
    """32768 cached keys, then the timed step's append of one token, then decode."""
    w = wl.get("append_decode_q4_ctx32k")
    L = gpu_layer(w, 0)
    ks = torch.stack([wl.kv_rows(w, 0, 0, s, w.lens[s], 1, "cuda") for s in range(w.n_seqs)])
    vs = torch.stack([wl.kv_rows(w, 0, 1, s, w.lens[s], 1, "cuda") for s in range(w.n_seqs)])
    kvq.kv_append_quantize(L, ks.contiguous(), vs.contiguous(),
                           torch.ones(w.n_seqs, dtype=torch.int32, device="cuda"))
    q = wl.queries(w, 0, 1, "cuda")[:, 0].contiguous()
    out, lse = _decode(L, q, max(w.final_lens()))
    assert L.seq_lens.tolist() == w.final_lens()
    _check_groups(w, 0, L, q, out, lse, [(0, h) for h in range(w.n_kv)], w.final_lens())


def _check_layer_full(w, layer_idx, L, q, out, lse, lens):
    """Every group of one layer: both caches byte for byte against the
    oracle's append of the same draws, then the oracle's attention of every
    query head (one call over the whole layer)."""
    ck, cv = w.codecs[layer_idx]
    G = w.n_q // w.n_kv
    kc, vc = oracle_layer(w, layer_idx, lens)
    assert np.array_equal(L.k_cache.cpu().numpy(), kc), f"layer {layer_idx}: K cache bytes"
    assert np.array_equal(L.v_cache.cpu().numpy(), vc), f"layer {layer_idx}: V cache bytes"
    ro, rl = oracle.decode_layer(ck, cv, kc, vc, w.n_seqs, w.n_kv, w.n_q, w.capacity, lens,
                                 q.cpu().numpy(), SCALE)
    on, ln = out.float().cpu().numpy(), lse.cpu().numpy()
    for s in range(w.n_seqs):
        for h in range(w.n_kv):
            rows = slice(h * G, (h + 1) * G)
            vmax = oracle.stream_absmax(cv, 1, vc, w.n_kv, w.capacity, s, h, lens[s])
            err = np.abs(on[s, rows] - ro[s, rows]).max()
            assert err <= 2e-3 * vmax, f"layer {layer_idx} seq {s} kvh {h}: {err} > {2e-3 * vmax}"
            assert np.abs(ln[s, rows] - rl[s, rows]).max() < 1e-3, (layer_idx, s, h)


def test_decode_ragged16_kf16_vq8_full():
    """All 128 (sequence, kv head) groups of the ragged 16-sequence layer."""
    w = wl.get("decode_ragged16_kf16_vq8")
    L = gpu_layer(w, 0)
    q = wl.queries(w, 0, 1, "cuda")[:, 0].contiguous()
    out, lse = _decode(L, q, max(w.lens))
    assert L.err.item() == 0
    _check_layer_full(w, 0, L, q, out, lse, w.lens)


@pytest.mark.parametrize("layer_idx", range(16))
def test_decode_16layer_ladder_every_layer(layer_idx):
    """Each of the 16 ladder layers in full: both caches, all 8 groups."""
    w = wl.get("decode_16layer_ladder_2x200704")
    L = gpu_layer(w, layer_idx, chunk=16384)
    q = wl.queries(w, layer_idx, 1, "cuda")[:, 0].contiguous()
    out, lse = _decode(L, q, max(w.lens))
    assert L.err.item() == 0
    _check_layer_full(w, layer_idx, L, q, out, lse, w.lens)


def test_ragged_many_streams_small_rings():
    """Many streams and long per-warp runs for the largest stages (f16 K and V)."""
    rng = np.random.default_rng(21)
    lens = [int(x) for x in rng.integers(1, 6000, 24)]
    w = wl.Workload("t", "decode", 24, 20, 4, lens, [(0, 0)], 22)
    L = gpu_layer(w, 0)
    q = wl.queries(w, 0, 1, "cuda")[:, 0].contiguous()
    out, lse = _decode(L, q, max(lens))
    assert L.err.item() == 0
    _check_groups(w, 0, L, q, out, lse, [(0, 0), (5, 3), (11, 1), (23, 2)], lens)
