"""attn_decode_noalloc through the C ABI: the same results as attn_decode with
a caller workspace, on two calls in a row, for a caller that allocates no
device memory for scratch (the library's fixed device array is used).

Kept in a file of its own that pytest collects last."""
import ctypes
import math

import numpy as np
import pytest
import torch

import attention_quantized_kv_gb300 as kvq
from attention_quantized_kv_gb300 import _abi
from attention_quantized_kv_gb300 import workloads as wl

import oracle
from tests._helpers import gpu_layer, oracle_stream

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from attention_quantized_kv_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _noalloc(L, q, scale, out, lse, max_len):
    d = L.desc()
    stream = torch.cuda.current_stream().cuda_stream
    return _abi.load().attn_decode_noalloc(ctypes.byref(d), q.data_ptr(), float(scale),
                                           out.data_ptr(), lse.data_ptr(), int(max_len), stream)


def test_noalloc_matches_workspace_decode_on_two_calls():
    lens = [3000, 17, 640, 1]
    w = wl.Workload("na", "decode", 4, 16, 4, lens, [(1, 2)], 77)
    L = gpu_layer(w, 0)
    q = wl.queries(w, 0, 1, "cuda")[:, 0].contiguous()
    scale = 1 / math.sqrt(128)
    ref = torch.empty_like(q)
    ref_lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    ws = torch.zeros(kvq.attn_decode_workspace(L, max(lens)), dtype=torch.uint8, device="cuda")
    kvq.attn_decode(L, q, scale, ref, ref_lse, max(lens), ws)
    torch.cuda.synchronize()
    vmax = max(np.abs(oracle.dequant_stream(2, 1, oracle_stream(w, 0, s, h, lens[s])[1], 1,
                                            w.capacity, 0, 0, lens[s])).max()
               for s in range(4) for h in range(4))
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc(L, q, scale, out, lse, max(lens)) == 0
        torch.cuda.synchronize()
        err = (out.float() - ref.float()).abs().max().item()
        assert err <= 2e-3 * vmax, f"call {call}: {err}"
        assert (lse - ref_lse).abs().max().item() < 1e-3
    assert L.err.item() == 0


def test_noalloc_refuses_layers_beyond_the_scratch():
    # 1000 sequences x 16 kv heads of 4096-key contexts need far more than 8 MiB;
    # the call is refused before anything reads the (placeholder) buffers.
    d = _abi.kvq_layer()
    d.n_seqs, d.n_kv_heads, d.n_q_heads, d.head_dim, d.capacity = 1000, 16, 16, 128, 4096
    d.codec_k, d.codec_v, d.reserved = 1, 1, 0
    buf = torch.empty(256, dtype=torch.uint8, device="cuda")
    d.k_cache = d.v_cache = buf.data_ptr()
    d.seq_lens = buf.data_ptr()
    d.err = 0
    q = torch.empty(64, dtype=torch.uint8, device="cuda")
    st = _abi.load().attn_decode_noalloc(ctypes.byref(d), q.data_ptr(), 0.1, q.data_ptr(), None,
                                         4096, torch.cuda.current_stream().cuda_stream)
    assert st == _abi.KVQ_EWORKSPACE
