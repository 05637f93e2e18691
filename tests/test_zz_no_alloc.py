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


def _paged_copy(w, L, seed):
    """The same layer over a page pool: every page a sequence uses on a
    distinct pool page in shuffled order, units moved as they are."""
    rng = np.random.default_rng(seed)
    pps = w.capacity // 256
    need = [(n + 255) // 256 for n in w.lens]
    n_pages = sum(need) + 3
    pages = rng.permutation(n_pages)
    table = -np.ones((w.n_seqs, pps), np.int32)
    k = 0
    for s in range(w.n_seqs):
        table[s, :need[s]] = pages[k:k + need[s]]
        k += need[s]
    ck, cv = w.codecs[0]
    kp = oracle.to_pool(ck, L.k_cache.cpu().numpy(), w.n_seqs, w.n_kv, w.capacity, table,
                        n_pages)
    vp = oracle.to_pool(cv, L.v_cache.cpu().numpy(), w.n_seqs, w.n_kv, w.capacity, table,
                        n_pages)
    P = kvq.KVLayer(w.n_seqs, w.n_kv, w.n_q, w.capacity, ck, cv, n_pages=n_pages,
                    block_table=torch.from_numpy(table).cuda(),
                    k_cache=torch.from_numpy(kp).cuda(), v_cache=torch.from_numpy(vp).cuda())
    P.seq_lens.copy_(L.seq_lens)
    return P


@pytest.mark.parametrize("ck,cv,paged", [(1, 2, False), (0, 1, False), (2, 2, True),
                                         (3, 1, False)])
def test_noalloc_matches_workspace_decode_on_two_calls(ck, cv, paged):
    """Bit-identical to attn_decode (the same plan and kernel; only the
    scratch differs) on two calls in a row, and within the attention bar of
    the oracle."""
    lens = [3000, 17, 640, 1]
    w = wl.Workload("na", "decode", 4, 16, 4, lens, [(ck, cv)], 77)
    L = gpu_layer(w, 0)
    if paged:
        L = _paged_copy(w, L, 5)
    q = wl.queries(w, 0, 1, "cuda")[:, 0].contiguous()
    scale = 1 / math.sqrt(128)
    ref = torch.empty_like(q)
    ref_lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    ws = torch.zeros(kvq.attn_decode_workspace(L, max(lens)), dtype=torch.uint8, device="cuda")
    kvq.attn_decode(L, q, scale, ref, ref_lse, max(lens), ws)
    torch.cuda.synchronize()
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc(L, q, scale, out, lse, max(lens)) == 0
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"call {call}: output differs from attn_decode"
        assert torch.equal(lse, ref_lse), f"call {call}: lse differs from attn_decode"
    assert L.err.item() == 0
    # and against the oracle directly
    G = w.n_q // w.n_kv
    on, ln = out.float().cpu().numpy(), lse.cpu().numpy()
    qn = q.cpu().numpy()
    for s in range(w.n_seqs):
        for h in range(w.n_kv):
            kc, vc = oracle_stream(w, 0, s, h, lens[s])
            ro, rl = oracle.decode_layer(ck, cv, kc, vc, 1, 1, G, w.capacity, [lens[s]],
                                         qn[s, h * G:(h + 1) * G], scale)
            vmax = oracle.stream_absmax(cv, 1, vc, 1, w.capacity, 0, 0, lens[s])
            err = np.abs(on[s, h * G:(h + 1) * G] - ro[0]).max()
            assert err <= 2e-3 * vmax, (s, h, err, 2e-3 * vmax)
            assert np.abs(ln[s, h * G:(h + 1) * G] - rl[0]).max() < 1e-3


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
