"""Decode attention on the GPU against the fp64 oracle.

Bar: max |out - oracle| <= 2e-3 * max |V^| over the attended (dequantized)
values, and the log-sum-exp output within 1e-3 (absolute, natural log).
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


@pytest.fixture(scope="module", autouse=True)
def _built():
    from attention_quantized_kv_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def run_decode(L, q, max_len, scale):
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    ws = torch.zeros(kvq.attn_decode_workspace(L, max_len), dtype=torch.uint8, device=q.device)
    kvq.attn_decode(L, q, scale, out, lse, max_len, ws)
    torch.cuda.synchronize()
    return out, lse


def check_against_oracle(w, layer_idx, L, q, out, lse, scale, groups=None, lens=None):
    """Compare (seq, kv head) groups; returns the worst error / bound ratio."""
    lens = w.lens if lens is None else lens
    G = w.n_q // w.n_kv
    ck, cv = w.codecs[layer_idx]
    qn = q.cpu().numpy()
    on = out.float().cpu().numpy()
    ln = lse.cpu().numpy()
    groups = groups or [(s, h) for s in range(w.n_seqs) for h in range(w.n_kv)]
    worst = 0.0
    for s, h in groups:
        T = lens[s]
        ok, ov = oracle_stream(w, layer_idx, s, h, T)
        qg = qn[s, h * G:(h + 1) * G]
        ro, rl = oracle.decode_layer(ck, cv, ok, ov, 1, 1, G, w.capacity, [T], qg, scale)
        V = oracle.dequant_stream(cv, 1, ov, 1, w.capacity, 0, 0, T)
        bound = 2e-3 * np.abs(V).max()
        err = np.abs(on[s, h * G:(h + 1) * G] - ro[0]).max()
        assert err <= bound, f"seq {s} kvh {h}: err {err:.3g} > {bound:.3g}"
        assert np.abs(ln[s, h * G:(h + 1) * G] - rl[0]).max() < 1e-3
        worst = max(worst, err / bound)
    return worst


PAIRS = [(a, b) for a in (0, 1, 2, 3) for b in (0, 1, 2, 3)]


@pytest.mark.parametrize("ck,cv", PAIRS)
def test_all_codec_pairs_ragged(ck, cv):
    lens = [1, 15, 16, 17, 100, 257, 1000]
    w = wl.Workload("t", "decode", len(lens), 8, 2, lens, [(ck, cv)], 100 + 3 * ck + cv)
    L = gpu_layer(w, 0)
    q = wl.queries(w, 0, 1, "cuda")[:, 0].contiguous()
    scale = 1 / math.sqrt(128)
    out, lse = run_decode(L, q, max(lens), scale)
    check_against_oracle(w, 0, L, q, out, lse, scale)


@pytest.mark.parametrize("G", [1, 4, 5, 8, 12])
def test_gqa_group_sizes(G):
    lens = [300, 33]
    w = wl.Workload("t", "decode", 2, 2 * G, 2, lens, [(1, 2)], 7 + G)
    L = gpu_layer(w, 0)
    q = wl.queries(w, 0, 1, "cuda")[:, 0].contiguous()
    out, lse = run_decode(L, q, max(lens), 0.09)
    check_against_oracle(w, 0, L, q, out, lse, 0.09)


def test_many_splits_and_outlier_channels():
    w = wl.Workload("t", "decode", 1, 16, 4, [20000], [(2, 2)], 31, outlier_frac=0.01,
                    outlier_scale=8.0)
    L = gpu_layer(w, 0)
    q = wl.queries(w, 0, 1, "cuda")[:, 0].contiguous()
    out, lse = run_decode(L, q, 20000, 1 / math.sqrt(128))
    check_against_oracle(w, 0, L, q, out, lse, 1 / math.sqrt(128))


def test_max_len_larger_than_lengths_and_zero_length_sequence():
    lens = [0, 40, 5]
    w = wl.Workload("t", "decode", 3, 4, 1, [0, 40, 5], [(1, 1)], 9)
    L = gpu_layer(w, 0, lens=[1, 40, 5])      # fill, then declare seq 0 empty
    L.seq_lens[0] = 0
    q = wl.queries(w, 0, 1, "cuda")[:, 0].contiguous()
    out, lse = run_decode(L, q, w.capacity, 0.1)
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
    check_against_oracle(w, 0, L, q, out, lse, 0.1, groups=[(1, 0), (2, 0)], lens=lens)
    assert L.err.item() == 0


def test_seq_len_beyond_max_len_sets_error_bit():
    w = wl.Workload("t", "decode", 1, 4, 1, [300], [(0, 0)], 10)
    L = gpu_layer(w, 0)
    q = wl.queries(w, 0, 1, "cuda")[:, 0].contiguous()
    run_decode(L, q, 256, 0.1)
    assert L.err.item() & kvq.KVQ_DEVERR_MAXLEN


def test_decode_is_repeatable_and_lse_consistent():
    w = wl.Workload("t", "decode", 2, 8, 2, [777, 4096], [(1, 0)], 12)
    L = gpu_layer(w, 0)
    q = wl.queries(w, 0, 1, "cuda")[:, 0].contiguous()
    o1, l1 = run_decode(L, q, 4096, 0.1)
    o2, l2 = run_decode(L, q, 4096, 0.1)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_workspace_reused_across_calls_and_geometries():
    """The ticket counters return to zero: one zeroed workspace serves many
    calls of different shapes, including grids larger than the unit count."""
    cases = [wl.Workload("a", "decode", 3, 8, 2, [5000, 17, 300], [(2, 1)], 40),
             wl.Workload("b", "decode", 1, 4, 4, [20], [(1, 1)], 41),
             wl.Workload("c", "decode", 7, 16, 2, [1, 2, 3, 40, 0, 700, 16], [(0, 2)], 42),
             wl.Workload("d", "decode", 2, 4, 2, [3, 1], [(2, 0)], 43)]
    # case d: max_len far above the lengths, so the grid exceeds the unit count
    max_lens = [max(w.lens) for w in cases[:3]] + [cases[3].capacity]
    big = max(kvq.attn_decode_workspace(gpu_layer(w, 0), ml) for w, ml in zip(cases, max_lens))
    ws = torch.zeros(big, dtype=torch.uint8, device="cuda")
    for rep in range(2):
        for w, ml in zip(cases, max_lens):
            L = gpu_layer(w, 0)
            q = wl.queries(w, 0, 1, "cuda")[:, 0].contiguous()
            out = torch.empty_like(q)
            lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
            kvq.attn_decode(L, q, 0.1, out, lse, ml, ws)
            torch.cuda.synchronize()
            groups = [(s, h) for s in range(w.n_seqs) for h in range(w.n_kv) if w.lens[s] > 0]
            check_against_oracle(w, 0, L, q, out, lse, 0.1, groups=groups)
            for s in range(w.n_seqs):
                if w.lens[s] == 0:
                    assert torch.all(out[s] == 0) and torch.all(torch.isneginf(lse[s]))
    assert torch.count_nonzero(ws[:64]) == 0     # tickets back to zero


@pytest.mark.parametrize("ck,cv", [(2, 2), (1, 0)])
def test_query_rows_only_8_byte_aligned(ck, cv):
    """q at an 8-byte (not 16-byte) offset takes the direct-load path for the
    query rows; it must give the same bits as 16-byte aligned rows, and both
    must match the oracle.  Many short streams put several segments (so
    several query-row copies, double-buffered) into each CTA."""
    lens = [40, 700, 33, 512, 1, 95, 300, 64, 129, 250]
    w = wl.Workload("t", "decode", len(lens), 16, 2, lens, [(ck, cv)], 300 + ck)
    L = gpu_layer(w, 0)
    q = wl.queries(w, 0, 1, "cuda")[:, 0].contiguous()
    raw = torch.empty(q.numel() + 4, dtype=torch.float16, device="cuda")
    q8 = raw[4:].view(q.shape)
    q8.copy_(q)
    assert q.data_ptr() % 16 == 0 and q8.data_ptr() % 16 == 8
    scale = 1 / math.sqrt(128)
    out, lse = run_decode(L, q, max(lens), scale)
    out8, lse8 = run_decode(L, q8, max(lens), scale)
    assert torch.equal(out, out8) and torch.equal(lse, lse8)
    check_against_oracle(w, 0, L, q, out, lse, scale)
