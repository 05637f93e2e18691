"""The C ABI without a GPU: the library builds, loads, exports every symbol
the header declares, and rejects bad arguments on the host (no launches)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from attention_quantized_kv_gb300 import build, _abi
    build.build()
    return _abi.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    return sorted(set(re.findall(r"^KVQ_API\s+[\w\s\*]*?\b(\w+)\s*\(", src, re.M)))


def test_header_declares_the_binding_exports():
    from attention_quantized_kv_gb300 import _abi
    assert _declared_functions() == sorted(_abi.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    import subprocess
    from attention_quantized_kv_gb300 import _abi
    out = subprocess.run(["nm", "-D", "--defined-only", _abi.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    for name in _declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)
    # nothing else leaks out of the library's own code
    assert exported == set(_declared_functions())


def test_row_and_cache_bytes(lib):
    assert [lib.kvq_row_bytes(c, 128) for c in (0, 1, 2)] == [256, 136, 72]
    assert lib.kvq_row_bytes(1, 64) == -1 and lib.kvq_row_bytes(7, 128) == -1
    assert lib.kvq_cache_bytes(1, 2, 4, 512, 128) == 2 * 4 * 512 * 136
    assert lib.kvq_cache_bytes(2, 1, 1, 300, 128) == -1       # not a multiple of 256
    assert lib.kvq_status_str(4).decode().startswith("KVQ_EALIGN")


def _layer(**kw):
    from attention_quantized_kv_gb300._abi import kvq_layer
    d = kvq_layer()
    vals = dict(n_seqs=1, n_kv_heads=2, n_q_heads=8, head_dim=128, capacity=4096, codec_k=1,
                codec_v=1, reserved=0, k_cache=0x100000, v_cache=0x200000, seq_lens=0x300000,
                err=0)
    vals.update(kw)
    for k, v in vals.items():
        setattr(d, k, v)
    return d


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=64), 2), (dict(codec_k=5), 2), (dict(n_q_heads=7), 1),
    (dict(capacity=1000), 4), (dict(k_cache=0x100008), 4), (dict(seq_lens=0), 1),
    (dict(n_seqs=0), 1), (dict(reserved=1), 1),
])
def test_layer_validation(lib, kw, status):
    d = _layer(**kw)
    n = ctypes.c_size_t(0)
    assert lib.attn_decode(ctypes.byref(d), 0x400000, 0.1, 0x500000, None, 16, 0x600000,
                           1 << 20, None) == status
    assert lib.kv_append_quantize(ctypes.byref(d), 0x400000, 0x500000, 0x600000, 1, 1,
                                  None) == status
    assert lib.attn_prefill_workspace(ctypes.byref(d), 0, 16, ctypes.byref(n)) == status


def test_call_argument_validation(lib):
    d = _layer()
    assert lib.attn_decode(None, 0x400000, 0.1, 0x500000, None, 16, 0x600000, 1, None) == 1
    assert lib.attn_decode(ctypes.byref(d), None, 0.1, 0x500000, None, 16, 0x600000, 1, None) == 1
    assert lib.attn_decode(ctypes.byref(d), 0x400000, 0.1, 0x500000, None, 0, 0x600000, 1, None) == 1
    assert lib.attn_decode(ctypes.byref(d), 0x400000, 0.1, 0x500000, None, 5000, 0x600000, 1,
                           None) == 3
    assert lib.attn_decode(ctypes.byref(d), 0x400002, 0.1, 0x500000, None, 16, 0x600000, 1,
                           None) == 4
    assert lib.attn_decode(ctypes.byref(d), 0x400000, 0.1, 0x500000, None, 16, None, 1, None) == 5
    assert lib.kv_append_quantize(ctypes.byref(d), 0x400000, 0x500000, None, 1, 1, None) == 1
    assert lib.kv_append_quantize(ctypes.byref(d), 0x400000, 0x500000, 0x600000, 5000, 1,
                                  None) == 3
    assert lib.attn_prefill_chunk(ctypes.byref(d), 1, 0, 16, 0x400000, 0.1, 0x500000, None,
                                  0x600000, 1 << 30, None) == 1      # seq out of range
    assert lib.attn_prefill_chunk(ctypes.byref(d), 0, 4090, 16, 0x400000, 0.1, 0x500000, None,
                                  0x600000, 1 << 30, None) == 3
    n = ctypes.c_size_t(0)
    assert lib.attn_prefill_workspace(ctypes.byref(d), 0, 2048, ctypes.byref(n)) == 0
    assert n.value > 0
    assert lib.attn_prefill_chunk(ctypes.byref(d), 0, 0, 2048, 0x400000, 0.1, 0x500000, None,
                                  0x600000, n.value - 1, None) == 5


def test_oracle_and_library_share_no_code():
    """The oracle is independent of the CUDA path: neither includes nor imports the other."""
    csrc = os.path.join(ROOT, "attention_quantized_kv_gb300", "csrc")
    for f in os.listdir(csrc):
        txt = open(os.path.join(csrc, f)).read()
        assert "kvq_oracle" not in txt and "oracle" not in txt.lower(), f
    for f in os.listdir(os.path.join(ROOT, "attention_quantized_kv_gb300")):
        if f.endswith(".py"):
            txt = open(os.path.join(ROOT, "attention_quantized_kv_gb300", f)).read()
            assert "import oracle" not in txt and "from oracle" not in txt, f
    otxt = open(os.path.join(ROOT, "oracle", "kvq_oracle.c")).read()
    assert "#include \"" not in otxt and "kvq.h" not in otxt


def test_ladder_planner_and_aggregate_match_the_oracle():
    """Host logic of the library (no GPU involved) against the oracle."""
    import oracle
    import attention_quantized_kv_gb300 as kvq
    rng = np.random.default_rng(12)
    for _ in range(200):
        n = int(rng.integers(1, 12))
        codecs = [int(c) for c in rng.integers(0, 3, n)]
        order = [int(t) for t in rng.permutation(n)[:int(rng.integers(0, n + 1))]]
        floor = float(rng.choice([0.0, 4.5, 8.5, 10.0, 16.0, float(rng.uniform(4, 16))]))
        assert kvq.aggregate_bpv(codecs) == oracle.aggregate_bpv(codecs)
        assert kvq.ladder_next(codecs, floor, order) == oracle.ladder_next(codecs, order, floor)
        assert kvq.ladder_next(codecs, floor) == oracle.ladder_next(codecs, list(range(n)), floor)


def test_fused_decode_step_argument_validation(lib):
    """attn_decode_append validates on the host before any device call: layer,
    missing rows, max_len, alignment and workspace, like attn_decode."""
    d = _layer()
    f = lib.attn_decode_append
    args = dict(k=0x700000, v=0x780000, q=0x400000, out=0x500000, max_len=16, ws=0x600000,
                ws_bytes=1 << 20)

    def call(layer=ctypes.byref(d), **kw):
        a = dict(args, **kw)
        return f(layer, a["k"], a["v"], a["q"], 0.1, a["out"], None, a["max_len"], a["ws"],
                 a["ws_bytes"], None)

    assert call(layer=None) == 1
    assert call(layer=ctypes.byref(_layer(head_dim=64))) == 2
    assert call(k=None) == 1
    assert call(v=None) == 1
    assert call(q=None) == 1
    assert call(max_len=0) == 1
    assert call(max_len=5000) == 3
    assert call(k=0x700004) == 4
    assert call(v=0x780002) == 4
    assert call(q=0x400002) == 4
    assert call(ws=None) == 5
    assert call(ws=0x600008) == 4


def test_paged_block_table_alignment_is_checked_by_every_decode_entry(lib):
    """A paged layer whose block table is not 4-byte aligned is refused on the
    host (KVQ_EALIGN) by attn_decode and attn_decode_noalloc alike: both run
    the same validation before any device call."""
    d = _layer(pages_per_seq=16, n_pages=40, block_table=0x700002)
    assert lib.attn_decode(ctypes.byref(d), 0x400000, 0.1, 0x500000, None, 16, 0x600000,
                           1 << 20, None) == 4
    assert lib.attn_decode_noalloc(ctypes.byref(d), 0x400000, 0.1, 0x500000, None, 16,
                                   None) == 4
    # the no-alloc entry point rejects the other bad arguments attn_decode rejects
    for kw, status in [(dict(head_dim=64), 2), (dict(capacity=1000), 4),
                       (dict(pages_per_seq=16, n_pages=0, block_table=0x700000), 1),
                       (dict(n_q_heads=7), 1)]:
        dd = _layer(**kw)
        assert lib.attn_decode_noalloc(ctypes.byref(dd), 0x400000, 0.1, 0x500000, None, 16,
                                       None) == status, kw
    assert lib.attn_decode_noalloc(ctypes.byref(_layer()), 0x400002, 0.1, 0x500000, None, 16,
                                   None) == 4
    assert lib.attn_decode_noalloc(ctypes.byref(_layer()), 0x400000, 0.1, 0x500000, None, 5000,
                                   None) == 3
