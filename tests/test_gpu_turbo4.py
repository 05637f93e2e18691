"""turbo4 (Walsh-Hadamard-rotated 4-bit rows) on the GPU: appended bytes
bit-exact against the oracle (the rotation is fixed to the definition's
fp32 operation order), and decode attention, which runs in the rotated space
(query rotated once, output rotated back once), within the bar of the other
codecs: max |out - oracle| <= 2e-3 * max |V^|.

The one extra rounding of the rotated path is the query H (s * q) / 16 taken
to fp16 for the tensor cores (relative 2^-12 per element), which moves each
score by about 2^-12 * scale * |q| |k| / sqrt(128): a few 1e-4 of a logit
for the workloads' N(0,1) rows, well inside the bar."""
import math

import numpy as np
import pytest
import torch

import attention_quantized_kv_gb300 as kvq
from attention_quantized_kv_gb300 import workloads as wl

import oracle
from tests._helpers import gpu_layer, gpu_stream_bytes, oracle_stream
from tests.test_gpu_decode import check_against_oracle, run_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from attention_quantized_kv_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.mark.parametrize("G", [1, 5, 12])
def test_turbo4_gqa_and_partial_head_groups(G):
    lens = [300, 33, 1]
    w = wl.Workload("t", "decode", 3, 2 * G, 2, lens, [(3, 3)], 70 + G, outlier_frac=0.01,
                    outlier_scale=8.0)
    L = gpu_layer(w, 0)
    q = wl.queries(w, 0, 1, "cuda")[:, 0].contiguous()
    out, lse = run_decode(L, q, max(lens), 1 / math.sqrt(128))
    check_against_oracle(w, 0, L, q, out, lse, 1 / math.sqrt(128))


def test_turbo4_many_splits_bytes_and_attention():
    w = wl.Workload("t", "decode", 1, 16, 4, [20000], [(3, 3)], 77, outlier_frac=0.01,
                    outlier_scale=8.0)
    L = gpu_layer(w, 0)
    for side in (0, 1):
        for h in (0, 3):
            assert np.array_equal(gpu_stream_bytes(L, side, 0, h),
                                  oracle_stream(w, 0, 0, h, 20000)[side])
    q = wl.queries(w, 0, 1, "cuda")[:, 0].contiguous()
    out, lse = run_decode(L, q, 20000, 1 / math.sqrt(128))
    check_against_oracle(w, 0, L, q, out, lse, 1 / math.sqrt(128))


def test_append_decode_turbo4_ctx32k_full_size_sampled():
    w = wl.get("append_decode_turbo4_ctx32k")
    L = gpu_layer(w, 0, lens=w.final_lens())
    q = wl.queries(w, 0, 1, "cuda")[:, 0].contiguous()
    out, lse = run_decode(L, q, max(w.final_lens()), 1 / math.sqrt(128))
    assert L.err.item() == 0
    for side in (0, 1):
        assert np.array_equal(gpu_stream_bytes(L, side, 0, 5),
                              oracle_stream(w, 0, 0, 5, w.final_lens()[0])[side])
    check_against_oracle(w, 0, L, q, out, lse, 1 / math.sqrt(128), groups=[(0, 0), (0, 5)],
                         lens=w.final_lens())


def test_turbo4_rows_decode_to_the_oracle_values_through_the_degrade():
    """turbo4 -> f16 through the library is the oracle's x^ rounded to fp16:
    the un-rotation on the GPU is exact in fp32."""
    n_seqs, n_kv, cap = 2, 2, 512
    lens = [257, 31]
    rng = np.random.default_rng(78)
    rows = rng.standard_normal((n_seqs, max(lens), n_kv, 128)).astype(np.float16)
    for side in (0, 1):
        c = np.zeros(oracle.cache_bytes(3, n_seqs, n_kv, cap), np.uint8)
        oracle.append_side(3, side, c, n_seqs, n_kv, cap, [0] * n_seqs, lens, rows)
        ck, cv = (3, 0) if side == 0 else (0, 3)
        L = kvq.KVLayer(n_seqs, n_kv, 2 * n_kv, cap, ck, cv,
                        k_cache=torch.zeros(kvq.kvq_cache_bytes(ck, n_seqs, n_kv, cap),
                                            dtype=torch.uint8, device="cuda"),
                        v_cache=torch.zeros(kvq.kvq_cache_bytes(cv, n_seqs, n_kv, cap),
                                            dtype=torch.uint8, device="cuda"))
        x = torch.from_numpy(rows).cuda()
        kvq.kv_append_quantize(L, x, x, torch.tensor(lens, dtype=torch.int32, device="cuda"))
        kvq.degrade(L, side, 0)
        torch.cuda.synchronize()
        assert L.err.item() == 0
        got = (L.k_cache if side == 0 else L.v_cache).cpu().numpy()
        for s in range(n_seqs):
            for h in range(n_kv):
                want = oracle.dequant_stream(3, side, c, n_kv, cap, s, h, lens[s])
                g = oracle.dequant_stream(0, side, got, n_kv, cap, s, h, lens[s])
                assert np.array_equal(g, want.astype(np.float16).astype(np.float64))
