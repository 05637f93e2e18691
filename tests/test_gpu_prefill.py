"""Chunked-prefill attention on the GPU (tcgen05) against the fp64 oracle.

Bar: max |out - oracle| <= 2e-3 * max |V^| over the attended values, lse
within 1e-3.  The prefill path rounds each dequantized key and value to fp16
once (the tensor-core operand type) and P to fp16; both errors are far inside
the bar (see the error budget in the design notes)."""
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


def run_prefill(L, seq, q_start, q, scale):
    out = torch.full_like(q, float("nan"))
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    ws = torch.empty(kvq.attn_prefill_workspace(L, q_start, q.shape[0]), dtype=torch.uint8,
                     device=q.device)
    kvq.attn_prefill_chunk(L, seq, q_start, q, scale, out, lse, ws)
    torch.cuda.synchronize()
    return out, lse


def check_prefill(w, L, seq, q_start, q, out, lse, scale, rows=None, kv_heads=None):
    G = w.n_q // w.n_kv
    ck, cv = w.codecs[0]
    n_tok = q.shape[0]
    T = q_start + n_tok
    rows = list(range(n_tok)) if rows is None else rows
    qn, on, ln = q.cpu().numpy(), out.float().cpu().numpy(), lse.cpu().numpy()
    for h in (range(w.n_kv) if kv_heads is None else kv_heads):
        ok_, ov_ = oracle_stream(w, 0, seq, h, T)
        ro, rl = oracle.prefill_chunk(ck, cv, ok_, ov_, 1, G, w.capacity, 0, q_start,
                                      np.ascontiguousarray(qn[:, h * G:(h + 1) * G]), scale,
                                      rows=rows)
        vmax = np.abs(oracle.dequant_stream(cv, 1, ov_, 1, w.capacity, 0, 0, T)).max()
        got = on[rows][:, h * G:(h + 1) * G]
        err = np.abs(got - ro[rows]).max()
        assert np.isfinite(got).all(), f"kvh {h}: non-finite output"
        assert err <= 2e-3 * vmax, f"kvh {h}: err {err:.3g} > {2e-3 * vmax:.3g}"
        assert np.abs(ln[rows][:, h * G:(h + 1) * G] - rl[rows]).max() < 1e-3


@pytest.mark.parametrize("ck,cv,G,q_start,n_tok", [
    (1, 1, 2, 0, 40),        # first chunk, one partial query block, one key tile
    (0, 2, 4, 100, 300),     # unaligned start: diagonal spans two key tiles
    (2, 1, 1, 256, 128),     # aligned start, exactly one query block
    (2, 2, 8, 1000, 200),
    (0, 0, 4, 37, 1),        # a single query row
    (1, 0, 5, 500, 129),     # GQA 5
    (3, 3, 4, 300, 200),     # turbo4 on both sides (un-rotated in the pre-pass)
    (3, 1, 2, 0, 64),
    (2, 3, 4, 64, 100),
])
def test_prefill_small(ck, cv, G, q_start, n_tok):
    n_kv = 2
    w = wl.Workload("t", "prefill", 1, G * n_kv, n_kv, [q_start], [(ck, cv)], 50 + ck * 3 + cv,
                    append_new=n_tok)
    L = gpu_layer(w, 0, lens=[q_start + n_tok])
    q = wl.queries(w, 0, n_tok, "cuda")[0].contiguous()
    out, lse = run_prefill(L, 0, q_start, q, 1 / math.sqrt(128))
    assert L.err.item() == 0
    check_prefill(w, L, 0, q_start, q, out, lse, 1 / math.sqrt(128))


def test_prefill_second_sequence_and_seqlen_check():
    w = wl.Workload("t", "prefill", 2, 8, 2, [300, 64], [(1, 1)], 61, append_new=64)
    L = gpu_layer(w, 0, lens=[300, 64 + 64])
    q = wl.queries(w, 0, 64, "cuda")[1].contiguous()
    out, lse = run_prefill(L, 1, 64, q, 0.1)
    assert L.err.item() == 0
    check_prefill(w, L, 1, 64, q, out, lse, 0.1)
    # a chunk whose keys were not appended sets the error bit
    run_prefill(L, 1, 128, q, 0.1)
    assert L.err.item() & kvq.KVQ_DEVERR_SEQLEN


def test_prefill_q8_32k_plus_2k_full_size_sampled_rows():
    """The benchmark workload: 32768 cached keys + a 2048-token ubatch appended
    through the append kernel, then the chunk's causal attention."""
    w = wl.get("prefill_q8_32k_plus_2k")
    L = gpu_layer(w, 0, lens=w.lens)
    kn = wl.kv_rows(w, 0, 0, 0, w.lens[0], w.append_new, "cuda")[None].contiguous()
    vn = wl.kv_rows(w, 0, 1, 0, w.lens[0], w.append_new, "cuda")[None].contiguous()
    kvq.kv_append_quantize(L, kn, vn, torch.tensor([w.append_new], dtype=torch.int32,
                                                   device="cuda"))
    q = wl.queries(w, 0, w.append_new, "cuda")[0].contiguous()
    out, lse = run_prefill(L, 0, w.lens[0], q, 1 / math.sqrt(128))
    assert L.err.item() == 0
    assert torch.isfinite(out).all()
    # every head, on 258 rows: every 8th row plus rows 1 and 2047
    rows = sorted(set([1, 2047] + list(range(0, 2048, 8))))
    check_prefill(w, L, 0, w.lens[0], q, out, lse, 1 / math.sqrt(128), rows=rows)
