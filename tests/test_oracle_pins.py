"""Pins for the CPU oracle: checks against what the pages and mathematics fix.

These tests never touch the CUDA library.  Each pin is chosen so that a
plausible slip in the oracle (a wrong rounding mode, a dropped scale, a
transposed layout, a wrong softmax normaliser or an off-by-one key limit)
fails at least one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- fp16 helpers

def test_half_to_float_exhaustive_matches_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.half_to_float(int(b)) for b in bits], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_float_to_half_matches_numpy_round_to_nearest_even():
    rng = np.random.default_rng(11)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(20000) * 1e-5).astype(np.float32),   # subnormal half range
        (rng.standard_normal(5000) * 3e4).astype(np.float32),     # near overflow
        np.array([65504, 65519.996, 65520, -65520, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                  2.0 ** -14, 2.0 ** -14 * (1 - 2.0 ** -12), 0.0, -0.0, 1e-30, -1e-30,
                  1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, np.inf, -np.inf], np.float32),
    ])
    # halfway points between adjacent halves exercise ties-to-even
    h = rng.integers(0, 0x7bff, 5000).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    vals = np.concatenate([vals, ((lo + hi) / 2).astype(np.float32)])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.float_to_half_bits(float(v)) for v in vals], np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- sizes (pages)

def test_row_bytes_follow_the_codec_table():
    g = _golden("codec_sizes.json")
    for name, codec in (("f16", oracle.F16), ("q8_0", oracle.Q8_0), ("q4_0", oracle.Q4_0)):
        bpv = g["bits_per_value"][name]
        assert oracle.ROW_BYTES[codec] * 8 == bpv * g["head_dim"]
        x = np.zeros((1, 128), np.float16)
        assert oracle.encode_rows(codec, x).shape == (1, g["derived"]["row_bytes"][name])


def test_kv_bytes_per_token_worked_examples():
    g = _golden("kv_bytes_per_token.json")
    L, H = g["geometry"]["layers"], g["geometry"]["kv_heads"]
    per_tok = lambda ck, cv: L * H * (oracle.ROW_BYTES[ck] + oracle.ROW_BYTES[cv])
    assert per_tok(oracle.F16, oracle.Q8_0) / 1024 == g["kib_per_token"]["k_f16_v_q8_0"]
    assert per_tok(oracle.F16, oracle.F16) / 1024 == g["kib_per_token"]["k_f16_v_f16"]
    ex = g["slots_example"]
    gib = ex["slots"] * ex["tokens_per_slot"] * per_tok(oracle.F16, oracle.Q8_0) / 2 ** 30
    assert round(gib, 1) == ex["gib_rounded_1dp"]


# ---------------------------------------------------------------- codecs: hand-derived blocks

@pytest.mark.parametrize("fixture,codec", [("q8_0_blocks.json", oracle.Q8_0),
                                            ("q4_0_blocks.json", oracle.Q4_0)])
def test_hand_derived_blocks(fixture, codec):
    for case in _golden(fixture)["cases"]:
        x = np.array(case["x"], np.float16)
        row = np.tile(x, 4)[None, :]          # the same block four times along head_dim
        got = oracle.encode_rows(codec, row)[0]
        bb = 34 if codec == oracle.Q8_0 else 18
        d16 = int(case["d16_hex"], 16)
        q = np.array(case["q"], np.int64)
        if codec == oracle.Q8_0:
            want = np.concatenate([[d16 & 0xff, d16 >> 8], q.astype(np.int8).view(np.uint8)])
        else:
            want = np.concatenate([[d16 & 0xff, d16 >> 8], q[:16] | (q[16:] << 4)])
        for b in range(4):
            assert np.array_equal(got[b * bb:(b + 1) * bb], want.astype(np.uint8)), case["name"]


def _random_blocks(rng, n):
    kinds = [
        lambda: rng.standard_normal(32),
        lambda: rng.standard_normal(32) * 1e-4,            # small scales, subnormal d16
        lambda: rng.standard_normal(32) * 300,
        lambda: np.where(rng.random(32) < 0.1, rng.standard_normal(32) * 8, rng.standard_normal(32)),
        lambda: rng.integers(-3, 4, 32).astype(np.float64),  # many ties in |x|
    ]
    return np.stack([kinds[i % len(kinds)]() for i in range(n)]).astype(np.float16)


def test_q8_0_properties_nearest_integer_and_error_bound():
    rng = np.random.default_rng(5)
    x16 = _random_blocks(rng, 4000)
    rows = oracle.encode_rows(oracle.Q8_0, x16.reshape(-1, 128)).reshape(-1, 34)
    x = x16.astype(np.float64)
    d16 = rows[:, :2].copy().view(np.uint16)[:, 0].view(np.float16).astype(np.float64)
    q = rows[:, 2:].view(np.int8).astype(np.float64)
    amax = np.abs(x).max(1)
    d = (amax.astype(np.float32) / np.float32(127)).astype(np.float64)
    # the stored scale is the fp16 rounding of amax/127 (within half an fp16 ulp)
    assert np.all(np.abs(d16 - amax / 127) <= np.maximum(np.abs(amax / 127) * 2 ** -11, 2 ** -25) + 1e-12)
    nz = d > 0
    t = x[nz] / d[nz, None]
    # q is a nearest integer of x/d (fp32 division adds at most one fp32 ulp)
    assert np.all(np.abs(t - q[nz]) <= 0.5 + 1e-5)
    assert np.all(np.abs(q) <= 127)
    # ties go away from zero: wherever |x/d| is (very nearly) k + 1/2, |q| = k + 1
    frac = np.abs(t) - np.floor(np.abs(t))
    tie = np.abs(frac - 0.5) < 1e-9
    assert np.all(np.abs(q[nz][tie]) == np.floor(np.abs(t[tie])) + 1)
    # reconstruction error: |x - d16 q| <= d/2 + |q| |d - d16| (+ rounding slack)
    err = np.abs(x - d16[:, None] * q)
    bound = d[:, None] / 2 + np.abs(q) * np.abs(d - d16)[:, None] + 1e-6 * amax[:, None] + 1e-12
    assert np.all(err <= bound)
    assert np.all(q[~nz] == 0)


def test_q4_0_properties():
    rng = np.random.default_rng(6)
    x16 = _random_blocks(rng, 4000)
    rows = oracle.encode_rows(oracle.Q4_0, x16.reshape(-1, 128)).reshape(-1, 18)
    x = x16.astype(np.float64)
    d16 = rows[:, :2].copy().view(np.uint16)[:, 0].view(np.float16).astype(np.float64)
    nib = np.concatenate([rows[:, 2:] & 0xf, rows[:, 2:] >> 4], axis=1).astype(np.float64)
    jmax = np.argmax(np.abs(x), axis=1)               # numpy argmax: first occurrence
    m = x[np.arange(len(x)), jmax]
    d = (m.astype(np.float32) / np.float32(-8)).astype(np.float64)
    assert np.all(np.abs(d16 - m / -8) <= np.maximum(np.abs(m / 8) * 2 ** -11, 2 ** -25) + 1e-12)
    # the element holding the block maximum always encodes to nibble 0 (x^ = -8 d = m)
    assert np.all(nib[np.arange(len(x)), jmax][d != 0] == 0)
    nz = d != 0
    t = x[nz] / d[nz, None]
    unclamped = t + 8.5 < 16
    # q - 8 = floor(t + 1/2) where not clamped: a nearest integer, ties upward
    assert np.all(np.abs(t - (nib[nz] - 8))[unclamped] <= 0.5 + 1e-5)
    assert np.all(nib[nz][~unclamped] == 15)
    assert np.all(nib[~nz] == 8)
    err = np.abs(x - d16[:, None] * (nib - 8))[nz]
    bound = (np.abs(d[nz, None]) / 2 + np.abs(nib[nz] - 8) * np.abs(d - d16)[nz, None]
             + 1e-6 * np.abs(m[nz, None]) + 1e-12)
    assert np.all(err[unclamped] <= bound[unclamped])
    # clamped values (x/d > 7.5: opposite sign, within d/2 of |m|) err by at most |d|
    cbound = np.broadcast_to(np.abs(d[nz, None]) + np.abs(d - d16)[nz, None] * 8
                             + 1e-6 * np.abs(m[nz, None]), err.shape)
    assert np.all(err[~unclamped] <= cbound[~unclamped])


def _fl32(r: Fraction) -> Fraction:
    """Nearest binary32 to a rational (ties to even), by exact arithmetic."""
    if r == 0:
        return Fraction(0)
    s = -1 if r < 0 else 1
    a = abs(r)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    ulp = Fraction(2) ** (e - 23)
    k = a / ulp
    fl = math.floor(k)
    rem = k - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return s * fl * ulp


def test_q8_0_exact_rational_rounding_on_sampled_blocks():
    """The two fp32 divisions of the formula, redone in exact rational arithmetic."""
    rng = np.random.default_rng(8)
    x16 = _random_blocks(rng, 60)
    rows = oracle.encode_rows(oracle.Q8_0, x16.reshape(-1, 128)).reshape(-1, 34)
    for blk, row in zip(x16, rows):
        xs = [Fraction(float(v)) for v in blk.astype(np.float64)]
        amax = max(abs(v) for v in xs)
        d = _fl32(amax / 127)
        for j, xv in enumerate(xs):
            if d == 0:
                want = 0
            else:
                t = _fl32(xv / d)
                want = int(math.floor(abs(t) + Fraction(1, 2))) * (1 if t >= 0 else -1)
            assert int(np.int8(row[2 + j].astype(np.int8))) == want


# ---------------------------------------------------------------- cache layout

@pytest.mark.parametrize("codec", [oracle.F16, oracle.Q8_0, oracle.Q4_0, oracle.TURBO4])
@pytest.mark.parametrize("side", [oracle.SIDE_K, oracle.SIDE_V])
def test_unit_layout_is_a_bijection(codec, side):
    tab = oracle.unit_offset_table(codec, side)
    ub = 16 * oracle.ROW_BYTES[codec]
    assert tab.min() == 0 and tab.max() == ub - 1
    assert np.array_equal(np.sort(tab.ravel()), np.arange(ub))


@pytest.mark.parametrize("codec", [oracle.F16, oracle.Q8_0, oracle.Q4_0, oracle.TURBO4])
def test_append_then_dequant_round_trip_in_pieces(codec):
    rng = np.random.default_rng(3)
    n_seqs, n_kv, cap = 2, 3, 64
    x = rng.standard_normal((n_seqs, 40, n_kv, 128)).astype(np.float16)
    for side in (oracle.SIDE_K, oracle.SIDE_V):
        cache_a = np.zeros(oracle.cache_bytes(codec, n_seqs, n_kv, cap), np.uint8)
        cache_b = np.zeros_like(cache_a)
        lens = np.array([0, 5], np.int32)
        # one append of all rows versus three ragged appends
        oracle.append_side(codec, side, cache_a, n_seqs, n_kv, cap, lens, [40, 33], x)
        pos = lens.copy()
        for piece in ([7, 1], [16, 17], [17, 15]):
            piece = np.array(piece, np.int32)
            xs = np.zeros((n_seqs, int(piece.max()), n_kv, 128), np.float16)
            for s in range(n_seqs):
                off = int(pos[s] - lens[s])
                xs[s, :piece[s]] = x[s, off:off + piece[s]]
            oracle.append_side(codec, side, cache_b, n_seqs, n_kv, cap, pos, piece, xs)
            pos += piece
        assert np.array_equal(cache_a, cache_b)
        for s, n in ((0, 40), (1, 33)):
            for h in range(n_kv):
                got = oracle.dequant_stream(codec, side, cache_a, n_kv, cap, s, h, lens[s] + n)
                want = oracle.decode_rows(codec, oracle.encode_rows(codec, x[s, :n, h]))
                assert np.array_equal(got[lens[s]:], want)
                if codec == oracle.F16:
                    assert np.array_equal(got[lens[s]:], x[s, :n, h].astype(np.float64))


def test_append_rejects_capacity_overflow():
    cache = np.zeros(oracle.cache_bytes(oracle.Q8_0, 1, 1, 16), np.uint8)
    x = np.zeros((1, 4, 1, 128), np.float16)
    with pytest.raises(ValueError):
        oracle.append_side(oracle.Q8_0, 0, cache, 1, 1, 16, [14], [4], x)


# ---------------------------------------------------------------- attention

def _softmax_attn_numpy(q, K, V, scale):
    s = (q.astype(np.float64) @ K.T) * scale
    m = s.max(axis=-1, keepdims=True)
    p = np.exp(s - m)
    z = p.sum(axis=-1, keepdims=True)
    return (p / z) @ V, (m + np.log(z))[..., 0]


def test_zero_query_gives_mean_of_values():
    rng = np.random.default_rng(1)
    T = 37
    K = rng.standard_normal((T, 128))
    V = rng.standard_normal((T, 128))
    q = np.zeros((3, 128), np.float16)
    out, lse = oracle.attend_rows(q, K, V, T, 1 / math.sqrt(128))
    assert np.allclose(out, V.mean(0), rtol=0, atol=1e-12)
    assert np.allclose(lse, math.log(T), atol=1e-12)


def test_dominant_score_selects_one_value_row():
    rng = np.random.default_rng(2)
    T, star = 50, 17
    q = np.zeros((1, 128), np.float16)
    q[0, 0] = 1.0
    K = rng.standard_normal((T, 128)) * 0.01
    K[star, 0] = 100.0 * math.sqrt(128)      # score 100 above every other key
    V = rng.standard_normal((T, 128))
    out, _ = oracle.attend_rows(q, K, V, T, 1 / math.sqrt(128))
    assert np.allclose(out[0], V[star], rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_four_token_contexts(seed):
    rng = np.random.default_rng(100 + seed)
    q = rng.standard_normal((5, 128)).astype(np.float16)
    K = rng.standard_normal((4, 128)).astype(np.float16).astype(np.float64)
    V = rng.standard_normal((4, 128)).astype(np.float16).astype(np.float64)
    scale = 1 / math.sqrt(128)
    out, lse = oracle.attend_rows(q, K, V, 4, scale)
    ref_o, ref_l = _softmax_attn_numpy(q, K, V, scale)
    assert np.allclose(out, ref_o, rtol=0, atol=1e-13)
    assert np.allclose(lse, ref_l, rtol=0, atol=1e-13)
    # each prefix length against explicit per-token sums
    for L in range(1, 5):
        o, l = oracle.attend_rows(q[:1], K, V, L, scale)
        s = [float(np.dot(q[0].astype(np.float64), K[t])) * scale for t in range(L)]
        w = [math.exp(v - max(s)) for v in s]
        ref = sum(wi * V[t] for t, wi in enumerate(w)) / sum(w)
        assert np.allclose(o[0], ref, rtol=0, atol=1e-13)
        assert abs(l[0] - (max(s) + math.log(sum(w)))) < 1e-13


def test_f16_codec_attention_matches_torch_float64():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(4)
    T = 29
    q = rng.standard_normal((4, 128)).astype(np.float16)
    kv16 = rng.standard_normal((2, T, 128)).astype(np.float16)
    K, V = kv16.astype(np.float64)
    out, _ = oracle.attend_rows(q, K, V, T, 0.0883883)
    qt = torch.from_numpy(q.astype(np.float64))
    p = torch.softmax(qt @ torch.from_numpy(K).T * 0.0883883, dim=-1)
    ref = (p @ torch.from_numpy(V)).numpy()
    assert np.allclose(out, ref, rtol=0, atol=1e-12)


def test_lse_merge_of_split_keys_equals_unsplit():
    rng = np.random.default_rng(9)
    T = 301
    q = rng.standard_normal((2, 128)).astype(np.float16)
    K = rng.standard_normal((T, 128))
    V = rng.standard_normal((T, 128))
    scale = 1 / math.sqrt(128)
    full_o, full_l = oracle.attend_rows(q, K, V, T, scale)
    cuts = [0, 64, 65, 200, T]
    parts = [oracle.attend_rows(q, K[a:b], V[a:b], b - a, scale) for a, b in zip(cuts, cuts[1:])]
    L = np.stack([p[1] for p in parts])
    M = L.max(0)
    w = np.exp(L - M)
    merged = sum(wi[:, None] * p[0] for wi, p in zip(w, parts)) / w.sum(0)[:, None]
    assert np.allclose(merged, full_o, rtol=0, atol=1e-12)
    assert np.allclose(M + np.log(w.sum(0)), full_l, rtol=0, atol=1e-12)


def test_empty_context_gives_zero_and_minus_inf():
    q = np.ones((1, 128), np.float16)
    out, lse = oracle.attend_rows(q, np.zeros((0, 128)), np.zeros((0, 128)), 0, 1.0)
    assert np.all(out == 0) and np.isneginf(lse[0])


def _fill_layer(rng, ck, cv, n_seqs, n_kv, cap, lens):
    caches = []
    xs = []
    for codec, side in ((ck, oracle.SIDE_K), (cv, oracle.SIDE_V)):
        c = np.zeros(oracle.cache_bytes(codec, n_seqs, n_kv, cap), np.uint8)
        x = rng.standard_normal((n_seqs, max(lens), n_kv, 128)).astype(np.float16)
        oracle.append_side(codec, side, c, n_seqs, n_kv, cap, [0] * n_seqs, lens, x)
        caches.append(c)
        xs.append(x)
    return caches, xs


def test_decode_layer_gqa_mapping_and_ragged_lengths():
    rng = np.random.default_rng(12)
    n_seqs, n_kv, n_q, cap = 3, 2, 6, 48
    lens = [5, 33, 1]
    ck, cv = oracle.Q8_0, oracle.Q4_0
    (cache_k, cache_v), (xk, xv) = _fill_layer(rng, ck, cv, n_seqs, n_kv, cap, lens)
    q = rng.standard_normal((n_seqs, n_q, 128)).astype(np.float16)
    out, lse = oracle.decode_layer(ck, cv, cache_k, cache_v, n_seqs, n_kv, n_q, cap, lens, q, 0.1)
    G = n_q // n_kv
    for s in range(n_seqs):
        for h in range(n_q):
            kv = h // G
            K = oracle.decode_rows(ck, oracle.encode_rows(ck, xk[s, :lens[s], kv]))
            V = oracle.decode_rows(cv, oracle.encode_rows(cv, xv[s, :lens[s], kv]))
            ro, rl = _softmax_attn_numpy(q[s, h][None], K, V, 0.1)
            assert np.allclose(out[s, h], ro[0], rtol=0, atol=1e-12)
            assert abs(lse[s, h] - rl[0]) < 1e-12


def test_prefill_chunk_is_causal_over_cached_plus_new_keys():
    rng = np.random.default_rng(13)
    n_kv, n_q, cap, cached, n_tok = 2, 4, 64, 20, 9
    ck = cv = oracle.Q8_0
    (cache_k, cache_v), (xk, xv) = _fill_layer(rng, ck, cv, 1, n_kv, cap, [cached + n_tok])
    q = rng.standard_normal((n_tok, n_q, 128)).astype(np.float16)
    out, lse = oracle.prefill_chunk(ck, cv, cache_k, cache_v, n_kv, n_q, cap, 0, cached, q, 0.125)
    for i in range(n_tok):
        for h in range(n_q):
            kv = h // (n_q // n_kv)
            L = cached + i + 1
            K = oracle.decode_rows(ck, oracle.encode_rows(ck, xk[0, :L, kv]))
            V = oracle.decode_rows(cv, oracle.encode_rows(cv, xv[0, :L, kv]))
            ro, rl = _softmax_attn_numpy(q[i, h][None], K, V, 0.125)
            assert np.allclose(out[i, h], ro[0], rtol=0, atol=1e-12)
    sub_o, _ = oracle.prefill_chunk(ck, cv, cache_k, cache_v, n_kv, n_q, cap, 0, cached, q, 0.125,
                                    rows=[0, 8])
    assert np.array_equal(sub_o[[0, 8]], out[[0, 8]]) and np.isnan(sub_o[1]).all()


# --------------------------------------------------------------------------- degrade ladder

_VBR = json.load(open(os.path.join(GOLDEN, "vbr_ladder.json")))


def test_bits_per_value_follow_the_codec_table():
    sizes = json.load(open(os.path.join(GOLDEN, "codec_sizes.json")))["bits_per_value"]
    assert oracle.bits_per_value(oracle.F16) == sizes["f16"]
    assert oracle.bits_per_value(oracle.Q8_0) == sizes["q8_0"]
    assert oracle.bits_per_value(oracle.Q4_0) == sizes["q4_0"]


def test_aggregate_bpv_reproduces_the_pages_first_two_steps():
    # the pages' 15.75 then 15.51 for 32 tensors fit a rung of 8.125 bits (two
    # decimals); the mean itself is checked with exact rationals, and with q8_0
    # the same two steps give the derived values.
    for k, printed in enumerate(_VBR["facts"]["qwen35_example"]["first_aggregates"], start=1):
        exact = Fraction((32 - k) * 16, 1) + k * Fraction(65, 8)
        assert round(float(exact / 32), 2) == printed
    want = _VBR["derived"]["q8_0_first_two_aggregates_32_tensors"]
    assert oracle.aggregate_bpv([0] * 31 + [1]) == want[0]
    assert oracle.aggregate_bpv([0] * 30 + [1, 1]) == want[1]
    rng = np.random.default_rng(5)
    for _ in range(20):
        c = rng.integers(0, 3, rng.integers(1, 40))
        brute = sum(Fraction(oracle.ROW_BYTES[int(x)] * 8, 128) for x in c) / len(c)
        assert oracle.aggregate_bpv(c) == float(brute)


def _run_ladder(codecs, order, floor):
    codecs = list(codecs)
    steps = []
    while True:
        st = oracle.ladder_next(codecs, order, floor)
        if st is None:
            return codecs, steps
        t, k = st
        assert k == codecs[t] + 1 or (codecs[t] == 0 and k == 1)  # one rung at a time
        codecs[t] = k
        steps.append(st)


def test_ladder_is_banded_and_has_tensors_times_rungs_steps():
    n = _VBR["facts"]["qwen35_example"]["tensors"]
    order = list(np.random.default_rng(6).permutation(n))
    final, steps = _run_ladder([0] * n, order, oracle.bits_per_value(oracle.Q4_0))
    assert len(steps) == _VBR["derived"]["classic_steps_32_tensors"] == 2 * n
    assert final == [2] * n
    # banded: the first n steps take every tensor to q8_0, in price order
    assert steps[:n] == [(t, 1) for t in order]
    assert steps[n:] == [(t, 2) for t in order]


def test_ladder_stops_at_the_floor_and_never_moves_pinned_tensors():
    n = 32
    final, steps = _run_ladder([0] * n, list(range(n)), 15.7)
    assert steps == [(0, 1)]  # 15.765625 >= 15.7 > 15.53125
    # the floor is inclusive
    final, steps = _run_ladder([0] * n, list(range(n)), 15.53125)
    assert steps == [(0, 1), (1, 1)]
    # tensors missing from the order (pinned) keep their codec
    order = [t for t in range(n) if t % 2 == 1]
    final, steps = _run_ladder([0] * n, order, 0.0)
    assert all(final[t] == 0 for t in range(0, n, 2))
    assert all(final[t] == 2 for t in order) and len(steps) == 2 * len(order)
    # a tensor already below f16 starts where it is
    final, steps = _run_ladder([1, 0, 2, 0], [0, 1, 2, 3], 0.0)
    assert steps == [(1, 1), (3, 1), (0, 2), (1, 2), (3, 2)]


def _cache_from_rows(codec, side, rows16, n_seqs, n_kv, capacity, lens):
    cache = np.zeros(oracle.cache_bytes(codec, n_seqs, n_kv, capacity), np.uint8)
    oracle.append_side(codec, side, cache, n_seqs, n_kv, capacity, [0] * n_seqs, lens, rows16)
    return cache


@pytest.mark.parametrize("side", [0, 1])
@pytest.mark.parametrize("dst", [1, 2, 3])
def test_requantize_from_f16_equals_appending_the_same_rows(side, dst):
    n_seqs, n_kv, capacity, lens = 2, 2, 256, [40, 17]
    rng = np.random.default_rng(7 + side + 2 * dst)
    rows = (rng.standard_normal((n_seqs, max(lens), n_kv, 128)) * 3).astype(np.float16)
    src = _cache_from_rows(0, side, rows, n_seqs, n_kv, capacity, lens)
    got = oracle.requantize_side(0, dst, side, src, n_seqs, n_kv, capacity, lens)
    want = _cache_from_rows(dst, side, rows, n_seqs, n_kv, capacity, lens)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("side", [0, 1])
def test_requantize_q8_to_q4_equals_q4_of_fp16_exact_values(side):
    # q8_0 blocks with power-of-two scales and small quants decode to values
    # that fp16 holds exactly, so q8_0 -> q4_0 must equal appending those fp16
    # values with q4_0.
    n_seqs, n_kv, capacity, lens = 1, 2, 256, [33]
    rng = np.random.default_rng(8 + side)
    q = rng.integers(-127, 128, (n_seqs, 33, n_kv, 128))
    q[..., ::32] = 127  # amax 127 per block, so d = 2^e exactly
    e = rng.integers(-8, 2, (n_seqs, 33, n_kv, 4))
    vals = (q.reshape(n_seqs, 33, n_kv, 4, 32) * (2.0 ** e)[..., None]).reshape(q.shape)
    vals16 = vals.astype(np.float16)
    assert np.array_equal(vals16.astype(np.float64), vals)  # exact in fp16
    src = _cache_from_rows(1, side, vals16, n_seqs, n_kv, capacity, lens)
    back = oracle.dequant_stream(1, side, src, n_kv, capacity, 0, 0, 33)
    assert np.array_equal(back, vals[0, :, 0].astype(np.float64))
    got = oracle.requantize_side(1, 2, side, src, n_seqs, n_kv, capacity, lens)
    want = _cache_from_rows(2, side, vals16, n_seqs, n_kv, capacity, lens)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("src_codec", [1, 2, 3])
def test_requantize_to_f16_rounds_the_decoded_values(src_codec):
    n_seqs, n_kv, capacity, lens = 1, 1, 256, [20]
    rng = np.random.default_rng(9)
    rows = rng.standard_normal((1, 20, 1, 128)).astype(np.float16)
    src = _cache_from_rows(src_codec, 1, rows, n_seqs, n_kv, capacity, lens)
    got = oracle.requantize_side(src_codec, 0, 1, src, n_seqs, n_kv, capacity, lens)
    dec = oracle.dequant_stream(src_codec, 1, src, n_kv, capacity, 0, 0, 20)
    f16 = oracle.dequant_stream(0, 1, got, n_kv, capacity, 0, 0, 20)
    assert np.array_equal(f16, dec.astype(np.float16).astype(np.float64))  # numpy RN
    # tokens past the length stay untouched (zero)
    assert not got[oracle.cache_bytes(0, 1, 1, 32):].any()


# --------------------------------------------------------------------------- paged layout

def test_paged_unit_address_hand_example():
    # 2 sequences x 2 pages, 3 kv heads; sequence 1's first page is pool page 0
    table = np.array([[3, 1], [0, -1]], np.int32)
    n_kv, n_pages = 3, 4
    # unit j of stream (s, h) -> (table[s][j // 16] * n_kv + h) * 16 + j % 16
    assert oracle.paged_unit(0, 0, 0, n_kv, table, n_pages) == (3 * 3 + 0) * 16
    assert oracle.paged_unit(0, 2, 17, n_kv, table, n_pages) == (1 * 3 + 2) * 16 + 1
    assert oracle.paged_unit(1, 1, 15, n_kv, table, n_pages) == (0 * 3 + 1) * 16 + 15
    assert oracle.paged_unit(1, 0, 16, n_kv, table, n_pages) == -1   # unmapped page
    assert oracle.paged_unit(0, 0, 32, n_kv, table, n_pages) == -1   # past pages_per_seq


@pytest.mark.parametrize("codec", [0, 1, 2])
def test_pool_with_one_kv_head_and_identity_table_is_the_contiguous_cache(codec):
    n_seqs, n_kv, pps = 3, 1, 2
    cap = pps * 256
    rng = np.random.default_rng(40 + codec)
    cache = rng.integers(0, 256, oracle.cache_bytes(codec, n_seqs, n_kv, cap)).astype(np.uint8)
    table = np.arange(n_seqs * pps, dtype=np.int32).reshape(n_seqs, pps)
    pool = oracle.to_pool(codec, cache, n_seqs, n_kv, cap, table, n_seqs * pps)
    assert np.array_equal(pool, cache)


@pytest.mark.parametrize("codec", [0, 1, 2, 3])
def test_pool_round_trip_under_a_shuffled_table(codec):
    n_seqs, n_kv, pps, n_pages = 3, 2, 3, 11
    cap = pps * 256
    rng = np.random.default_rng(50 + codec)
    cache = rng.integers(0, 256, oracle.cache_bytes(codec, n_seqs, n_kv, cap)).astype(np.uint8)
    pages = rng.permutation(n_pages)[:n_seqs * pps].astype(np.int32)
    table = pages.reshape(n_seqs, pps).copy()
    table[2, 2] = -1  # an unmapped page: its units do not survive the round trip
    pool = oracle.to_pool(codec, cache, n_seqs, n_kv, cap, table, n_pages)
    back = oracle.from_pool(codec, pool, n_seqs, n_kv, cap, table, n_pages)
    ub = 16 * oracle.ROW_BYTES[codec]
    units = cap // 16
    want = cache.copy().reshape(n_seqs, n_kv, units, ub)
    want[2, :, 32:48] = 0
    assert np.array_equal(back.reshape(n_seqs, n_kv, units, ub), want)
    # every pool unit that a mapped page covers holds exactly one source unit
    used = {int(p) for p in table.flatten() if p >= 0}
    assert not pool.reshape(n_pages, n_kv * 16, ub)[[p for p in range(n_pages)
                                                      if p not in used]].any()


# --------------------------------------------------------------------------- probe-scored eviction

def _probe_cache(rng, codec, n_seqs, n_kv, cap, lens, scale_rows=1.0):
    rows = (rng.standard_normal((n_seqs, max(lens), n_kv, 128)) * scale_rows).astype(np.float16)
    c = np.zeros(oracle.cache_bytes(codec, n_seqs, n_kv, cap), np.uint8)
    oracle.append_side(codec, 0, c, n_seqs, n_kv, cap, [0] * n_seqs, lens, rows)
    return c, rows


def test_probe_mass_sums_to_the_head_count_and_is_flat_for_a_zero_query():
    n_seqs, n_kv, n_q, cap, lens = 2, 2, 6, 256, [50, 7]
    rng = np.random.default_rng(80)
    c, _ = _probe_cache(rng, 1, n_seqs, n_kv, cap, lens)
    q = rng.standard_normal((n_seqs, n_q, 128)).astype(np.float16)
    m = oracle.probe_mass(1, c, n_seqs, n_kv, n_q, cap, lens, q, 0.1)
    for s in range(n_seqs):
        assert m[s, :lens[s]].sum() == pytest.approx(n_q, rel=1e-12)
        assert not m[s, lens[s]:].any()
    m0 = oracle.probe_mass(1, c, n_seqs, n_kv, n_q, cap, lens, np.zeros_like(q), 0.1)
    for s in range(n_seqs):
        assert np.allclose(m0[s, :lens[s]], n_q / lens[s], rtol=1e-12)


def test_probe_mass_of_a_dominant_key_and_the_gqa_mapping():
    # f16 keys: query head j of kv head h sees keys of kv head h only
    n_seqs, n_kv, n_q, cap, T = 1, 2, 4, 256, 9
    K = np.zeros((1, T, n_kv, 128), np.float16)
    K[0, 3, 0, 0] = 8.0   # kv head 0: key 3 dominates for q e_0
    K[0, 6, 1, 1] = 8.0   # kv head 1: key 6 dominates for q e_1
    c = np.zeros(oracle.cache_bytes(0, 1, n_kv, cap), np.uint8)
    oracle.append_side(0, 0, c, 1, n_kv, cap, [0], [T], K)
    q = np.zeros((1, n_q, 128), np.float16)
    q[0, 0:2, 0] = 8.0    # query heads 0, 1 -> kv head 0
    q[0, 2:4, 1] = 8.0    # query heads 2, 3 -> kv head 1
    m = oracle.probe_mass(0, c, 1, n_kv, n_q, cap, [T], q, 1.0)
    w = 1.0 / (1.0 + (T - 1) * math.exp(-64.0))  # softmax weight of the dominant key
    assert m[0, 3] == pytest.approx(2 * w, rel=1e-12)
    assert m[0, 6] == pytest.approx(2 * w, rel=1e-12)
    assert m[0, :T].sum() == pytest.approx(n_q, rel=1e-12)


def test_evict_select_against_brute_force_and_protection():
    rng = np.random.default_rng(81)
    for _ in range(300):
        length = int(rng.integers(0, 60))
        sink, recent, n_ev = (int(rng.integers(0, 6)), int(rng.integers(0, 6)),
                              int(rng.integers(0, 20)))
        sc = rng.integers(0, 8, length).astype(np.float32)  # many ties
        got = oracle.evict_select(sc, length, sink, recent, n_ev)
        mid = list(range(sink, max(sink, length - recent)))
        want = sorted(sorted(mid, key=lambda t: (sc[t], t))[:n_ev])
        assert list(got) == want
        assert all(sink <= t < length - recent for t in got)


@pytest.mark.parametrize("codec", [0, 1, 2, 3])
@pytest.mark.parametrize("side", [0, 1])
def test_compaction_equals_appending_the_kept_rows(codec, side):
    n_seqs, n_kv, cap, lens = 2, 2, 256, [40, 17]
    rng = np.random.default_rng(82 + codec + 3 * side)
    rows = rng.standard_normal((n_seqs, max(lens), n_kv, 128)).astype(np.float16)
    c = np.zeros(oracle.cache_bytes(codec, n_seqs, n_kv, cap), np.uint8)
    oracle.append_side(codec, side, c, n_seqs, n_kv, cap, [0] * n_seqs, lens, rows)
    evict = [[1, 2, 17, 39], [0, 16]]
    got = oracle.compact_side(codec, side, c, n_seqs, n_kv, cap, lens, evict)
    kept_lens = [lens[s] - len(evict[s]) for s in range(n_seqs)]
    kept = np.zeros((n_seqs, max(kept_lens), n_kv, 128), np.float16)
    for s in range(n_seqs):
        keep = [t for t in range(lens[s]) if t not in evict[s]]
        kept[s, :len(keep)] = rows[s, keep]
    want = np.zeros_like(c)
    oracle.append_side(codec, side, want, n_seqs, n_kv, cap, [0] * n_seqs, kept_lens, kept)
    assert np.array_equal(got, want)


# --------------------------------------------------------------------------- turbo4 (rotated 4-bit)

def test_splitmix64_published_outputs():
    g = _golden("splitmix64.json")
    assert oracle.splitmix64(g["seed"], len(g["outputs"])) == [int(v) for v in g["outputs"]]


def test_turbo_signs_are_bit_63_of_the_generator():
    outs = oracle.splitmix64(0x4B5651, 128)
    want = np.array([-1 if (v >> 63) else 1 for v in outs], np.int32)
    got = oracle.turbo_signs()
    assert np.array_equal(got, want)
    assert 40 < (got > 0).sum() < 88  # sign flips, not a constant


def test_fwht_is_the_sylvester_hadamard_matrix():
    from scipy.linalg import hadamard
    H = hadamard(128).astype(np.float64)
    rng = np.random.default_rng(90)
    xi = rng.integers(-1000, 1000, 128).astype(np.float64)  # exact in fp32 and fp64
    assert np.array_equal(oracle.fwht128(xi), H @ xi)
    assert np.array_equal(oracle.fwht128(xi.astype(np.float32), np.float32), (H @ xi).astype(np.float32))
    x = rng.standard_normal(128)
    assert np.allclose(oracle.fwht128(x), H @ x, rtol=0, atol=1e-12)
    assert np.allclose(oracle.fwht128(oracle.fwht128(x)), 128 * x, rtol=0, atol=1e-11)


def test_turbo4_hand_derived_rows():
    g = _golden("turbo4_rows.json")
    s = oracle.turbo_signs()
    assert s[0] == 1
    for r in g["rows"]:
        x = np.zeros(128) if r["x"] == "e0" else s.astype(np.float64)
        if r["x"] == "e0":
            x[0] = 1.0
        row = oracle.encode_rows(oracle.TURBO4, x.astype(np.float16)[None])[0]
        assert row.tobytes().hex() == r["bytes_hex"], r["name"]
        dec = oracle.decode_rows(oracle.TURBO4, row[None])[0]
        assert np.array_equal(dec, x), r["name"]


def test_turbo4_round_trip_and_quantisation_bound():
    """y = H(s x)/8 recomputed with the Hadamard matrix in fp64; the stored
    y^ = d16 (q - 8) is within d16/2 (+ the fp16 rounding of d) of y except
    for values clamped to 15 (within |d|); x^ = s H y^ / 16 exactly, and
    ||x^ - x|| = ||y^ - y|| / sqrt(2) (the rotation is orthogonal up to the
    exact factors)."""
    from scipy.linalg import hadamard
    H = hadamard(128).astype(np.float64)
    s = oracle.turbo_signs().astype(np.float64)
    rng = np.random.default_rng(91)
    x = rng.standard_normal((400, 128))
    x[:, [3, 77]] *= 8.0  # outlier channels
    x[:100] *= 1e-3
    x = x.astype(np.float16)
    rows = oracle.encode_rows(oracle.TURBO4, x)
    dec = oracle.decode_rows(oracle.TURBO4, rows)
    for i in range(len(x)):
        xd = x[i].astype(np.float64)
        y = H @ (s * xd) / 8
        yh = oracle.turbo4_rotated(rows[i])
        d16 = oracle.half_to_float(int(rows[i][0]) | (int(rows[i][1]) << 8))
        jm = int(np.argmax(np.abs(y)))
        d = np.float32(y[jm]) / np.float32(-8.0)
        q = np.round(yh / d16 + 8).astype(int)
        err = np.abs(y - yh)
        clamped = q == 15
        bound = abs(d16) / 2 + np.abs(q - 8) * abs(float(d) - d16) + 1e-6 * abs(d16)
        assert (err[~clamped] <= bound[~clamped]).all()
        assert (err[clamped] <= abs(d16) * 1.0001 + 1e-6 * abs(d16)).all()
        assert np.array_equal(dec[i], s * (H @ yh) / 16)
        assert np.linalg.norm(dec[i] - xd) == pytest.approx(np.linalg.norm(yh - y) / math.sqrt(2),
                                                            rel=1e-9)


def test_turbo4_bits_per_value_follow_the_codec_table():
    g = _golden("codec_sizes.json")
    assert oracle.bits_per_value(oracle.TURBO4) == g["bits_per_value"]["turbo4"]
    assert oracle.ROW_BYTES[oracle.TURBO4] == g["derived"]["row_bytes"]["turbo4"]


def test_turbo4_attention_equals_attention_over_decoded_rows():
    """decode_layer over a turbo4 cache is softmax attention over x^ (the
    oracle never attends in the rotated space), and q . x^ = (H s q / 16) . y^."""
    from scipy.linalg import hadamard
    H = hadamard(128).astype(np.float64)
    s = oracle.turbo_signs().astype(np.float64)
    rng = np.random.default_rng(92)
    n_kv, n_q, cap, T = 1, 2, 256, 30
    k = rng.standard_normal((1, T, n_kv, 128)).astype(np.float16)
    v = rng.standard_normal((1, T, n_kv, 128)).astype(np.float16)
    ck = np.zeros(oracle.cache_bytes(3, 1, n_kv, cap), np.uint8)
    cv = np.zeros_like(ck)
    oracle.append_side(3, 0, ck, 1, n_kv, cap, [0], [T], k)
    oracle.append_side(3, 1, cv, 1, n_kv, cap, [0], [T], v)
    q = rng.standard_normal((1, n_q, 128)).astype(np.float16)
    out, lse = oracle.decode_layer(3, 3, ck, cv, 1, n_kv, n_q, cap, [T], q, 0.1)
    K = oracle.dequant_stream(3, 0, ck, n_kv, cap, 0, 0, T)
    V = oracle.dequant_stream(3, 1, cv, n_kv, cap, 0, 0, T)
    ro, rl = _softmax_attn_numpy(q[0], K, V, 0.1)
    assert np.allclose(out[0], ro, rtol=0, atol=1e-12)
    assert np.allclose(lse[0], rl, rtol=0, atol=1e-12)
    rows = oracle.encode_rows(3, k[0, :, 0])
    qr = H @ (s * q[0, 0].astype(np.float64)) / 16
    for t in range(T):
        assert float(q[0, 0].astype(np.float64) @ K[t]) == pytest.approx(
            float(qr @ oracle.turbo4_rotated(rows[t])), rel=1e-12, abs=1e-12)


# ---------------------------------------------------------------- q4_0 decoder, by hand

def _q4_0_row_by_hand():
    """One canonical q4_0 row (four 18-byte blocks) and its values worked out
    by hand from x^ = d16 * (q - 8), low nibble = element j, high nibble =
    element j + 16 (byte layout of the q4_0 row of the "Codecs" table's
    4.5-bit format: fp16 scale, then 16 bytes of two nibbles each)."""
    row, want = [], []
    # block 0: d16 = 0x3C00 (1.0); byte j = j | (15 - j) << 4
    row += [0x00, 0x3C] + [j | ((15 - j) << 4) for j in range(16)]
    want += [j - 8.0 for j in range(16)] + [7.0 - j for j in range(16)]
    # block 1: d16 = 0xB000 (-0.125); every byte 0x0F: low nibble 15, high 0
    row += [0x00, 0xB0] + [0x0F] * 16
    want += [-0.125 * 7] * 16 + [-0.125 * -8] * 16
    # block 2: d16 = 0x4000 (2.0); every byte 0x88: both nibbles 8 -> 0
    row += [0x00, 0x40] + [0x88] * 16
    want += [0.0] * 32
    # block 3: d16 = 0x0001 (2^-24, the smallest subnormal); bytes 0xF0, 0x1E
    row += [0x01, 0x00] + [0xF0, 0x1E] * 8
    lo = [0 - 8, 14 - 8] * 8
    hi = [15 - 8, 1 - 8] * 8
    want += [v * 2.0 ** -24 for v in lo] + [v * 2.0 ** -24 for v in hi]
    return np.array(row, np.uint8), np.array(want, np.float64)


def test_q4_0_decoder_hand_derived_values():
    row, want = _q4_0_row_by_hand()
    assert row.size == 72
    got = oracle.decode_rows(oracle.Q4_0, row)[0]
    assert np.array_equal(got, want)
    # a swapped nibble order or 8 - q instead of q - 8 moves these values
    assert got[0] == -8.0 and got[16] == 7.0 and got[32] == -0.875 and got[48] == 1.0


@pytest.mark.parametrize("side", [0, 1])
def test_q4_0_dequant_stream_hand_derived_values(side):
    """The same row placed at token 21 of a stream (unit 1, row 5) by the
    layout's offsets and read back through the stream dequantizer."""
    row, want = _q4_0_row_by_hand()
    cap = 256
    cache = np.zeros(oracle.cache_bytes(oracle.Q4_0, 1, 1, cap), np.uint8)
    unit = cache[16 * 72:32 * 72]
    for cb in range(72):
        unit[oracle.unit_offset(oracle.Q4_0, side, 5, cb)] = row[cb]
    got = oracle.dequant_stream(oracle.Q4_0, side, cache, 1, cap, 0, 0, 22)
    assert np.array_equal(got[21], want)
    # every other row of the stream decodes from zero bytes: d16 = 0
    assert not np.any(got[:21])


# ---------------------------------------------------------------- unit layout, by hand

# (codec, side, token row r, canonical byte cb, unit offset), each worked out
# by hand from the placement formulas of the library's public header
# (g = r & 7, rh = r >> 3, tig = (r & 7) >> 1, par = r & 1):
_UNIT_OFFSETS_BY_HAND = [
    # f16 K: d = cb >> 1, k = cb & 1; b=d>>5 h=(d>>4)&1 w=(d>>2)&3 i=d&3
    #        -> (2b+rh)*512 + (4g+w)*16 + h*8 + i*2 + k
    (0, 0, 0, 0, 0),
    (0, 0, 11, 154, 2802),   # d 77: b2 h0 w3 i1; g3 rh1 -> 5*512 + 15*16 + 2
    (0, 0, 5, 45, 349),      # d 22 k1: b0 h1 w1 i2; g5 -> 21*16 + 8 + 4 + 1
    (0, 0, 15, 255, 4095),   # the unit's last byte
    # f16 V: mt=d>>4 gq=(d&15)>>1 s=d&1 -> mt*512 + (4gq+tig)*16 + (rh*4+s*2+par)*2 + k
    (0, 1, 11, 154, 2462),   # d 77: mt4 gq6 s1; tig1 par1 rh1 -> 2048 + 25*16 + 7*2
    (0, 1, 6, 11, 181),      # d 5 k1: mt0 gq2 s1; tig3 par0 -> 11*16 + 2*2 + 1
    (0, 1, 15, 255, 4095),
    # q8_0 K: b = cb // 34, o = cb % 34; scale byte o < 2 -> 2048 + g*16 + rh*8 + b*2 + o;
    #         quant e = o - 2: h=e>>4 w=(e>>2)&3 i=e&3 -> b*512 + (4g+w)*16 + (2rh+h)*4 + i
    (1, 0, 0, 0, 2048),
    (1, 0, 9, 35, 2075),     # block 1 scale byte 1; g1 rh1 -> 2048 + 16 + 8 + 2 + 1
    (1, 0, 9, 91, 1117),     # block 2, e 21: h1 w1 i1 -> 1024 + 5*16 + 3*4 + 1
    (1, 0, 15, 135, 2047),   # block 3, e 31 -> 1536 + 31*16 + 3*4 + 3
    (1, 0, 15, 103, 2175),   # block 3 scale byte 1: the unit's last byte
    # q8_0 V: quant of dim d = 32b + e: mt=d>>4 gq=(d&15)>>1 s=d&1
    #         -> (mt>>1)*512 + (4gq+tig)*16 + ((mt&1)*2+rh)*4 + par*2 + s;
    #         scale byte k -> 2048 + tig*32 + b*8 + rh*4 + par*2 + k
    (1, 1, 0, 2, 0),
    (1, 1, 11, 91, 1183),    # d 85: mt5 gq2 s1; tig1 par1 rh1 -> 1024 + 9*16 + 3*4 + 3
    (1, 1, 11, 35, 2095),    # block 1 scale byte 1 -> 2048 + 32 + 8 + 4 + 2 + 1
    (1, 1, 14, 1, 2149),     # block 0 scale byte 1; tig3 par0 rh1 -> 2048 + 96 + 4 + 1
    (1, 1, 15, 103, 2175),
    # q4_0 K: b = cb // 18, o = cb % 18; scale -> 1024 + g*16 + rh*8 + b*2 + o;
    #         byte jc = o - 2: w=jc>>2 i=jc&3 -> (b>>1)*512 + (4g+w)*16 + ((b&1)*2+rh)*4 + i
    (2, 0, 0, 2, 0),
    (2, 0, 13, 70, 894),     # block 3 jc 14: w3 i2; g5 rh1 -> 512 + 23*16 + 3*4 + 2
    (2, 0, 13, 19, 1115),    # block 1 scale byte 1 -> 1024 + 80 + 8 + 2 + 1
    (2, 0, 2, 43, 657),      # block 2 jc 5: w1 i1; g2 rh0 -> 512 + 9*16 + 1
    (2, 0, 15, 71, 1023),
    # q4_0 V: byte jc of block b: mt=2b+(jc>>3) gq=jc&7
    #         -> (mt>>2)*512 + (4gq+tig)*16 + (mt&3)*4 + par*2 + rh;
    #         scale byte k -> 1024 + tig*32 + b*8 + rh*4 + par*2 + k
    (2, 1, 0, 2, 0),
    (2, 1, 13, 70, 943),     # block 3 jc 14: mt7 gq6; tig2 par1 rh1 -> 512 + 26*16 + 12 + 2 + 1
    (2, 1, 13, 19, 1103),    # block 1 scale byte 1 -> 1024 + 64 + 8 + 4 + 2 + 1
    (2, 1, 4, 29, 108),      # block 1 jc 9: mt3 gq1; tig2 par0 rh0 -> 6*16 + 3*4
    (2, 1, 15, 71, 1023),
    # turbo4: scale bytes cb < 2 (K: 1024 + g*4 + rh*2 + cb; V: 1024 + tig*8 + rh*4 + par*2 + cb);
    #         group byte cb = 2 + 16b + jc sits at q4_0's place of byte jc of block b
    (3, 0, 13, 1, 1047),     # g5 rh1 -> 1024 + 20 + 2 + 1
    (3, 0, 13, 64, 894),     # group 3 byte 14: as the q4_0 K case above
    (3, 0, 15, 1, 1055),     # the unit's last byte (1056 bytes)
    (3, 1, 13, 0, 1046),     # tig2 rh1 par1 -> 1024 + 16 + 4 + 2
    (3, 1, 13, 64, 943),     # as the q4_0 V case above
]


@pytest.mark.parametrize("codec,side,r,cb,want", _UNIT_OFFSETS_BY_HAND)
def test_unit_offset_hand_worked_examples(codec, side, r, cb, want):
    assert oracle.unit_offset(codec, side, r, cb) == want


# ---------------------------------------------------------------- threading does not change results

def test_decode_layer_is_identical_on_one_thread_and_on_all():
    """Rows are attended independently in a fixed order, so the thread count
    and the batching of groups change nothing, bit for bit."""
    rng = np.random.default_rng(77)
    n_seqs, n_kv, n_q, cap = 3, 2, 6, 512
    lens = [300, 0, 511]
    caches = []
    for side, codec in ((0, oracle.Q4_0), (1, oracle.Q8_0)):
        c = np.zeros(oracle.cache_bytes(codec, n_seqs, n_kv, cap), np.uint8)
        x = rng.standard_normal((n_seqs, max(lens), n_kv, 128)).astype(np.float16)
        oracle.append_side(codec, side, c, n_seqs, n_kv, cap, [0] * n_seqs, lens, x)
        caches.append(c)
    q = rng.standard_normal((n_seqs, n_q, 128)).astype(np.float16)
    with oracle.threads(1):
        o1, l1 = oracle.decode_layer(oracle.Q4_0, oracle.Q8_0, *caches, n_seqs, n_kv, n_q, cap,
                                     lens, q, 0.088)
    on, ln = oracle.decode_layer(oracle.Q4_0, oracle.Q8_0, *caches, n_seqs, n_kv, n_q, cap,
                                 lens, q, 0.088)
    assert np.array_equal(o1, on) and np.array_equal(l1, ln)
    # one group at a time gives the same rows
    for s in range(n_seqs):
        for h in range(n_kv):
            sel = np.zeros((n_seqs, n_kv), bool)
            sel[s, h] = True
            og, lg = oracle.decode_layer(oracle.Q4_0, oracle.Q8_0, *caches, n_seqs, n_kv, n_q,
                                         cap, lens, q, 0.088, sel=sel)
            rows = slice(h * 3, h * 3 + 3)
            assert np.array_equal(og[s, rows], on[s, rows])
            assert np.array_equal(lg[s, rows], ln[s, rows])
    assert np.all(on[1] == 0) and np.all(ln[1] == -np.inf)


def test_stream_absmax_is_the_largest_decoded_magnitude():
    rng = np.random.default_rng(78)
    cap = 256
    for side, codec in ((0, oracle.F16), (1, oracle.Q8_0), (1, oracle.Q4_0), (0, oracle.TURBO4)):
        c = np.zeros(oracle.cache_bytes(codec, 1, 2, cap), np.uint8)
        x = (rng.standard_normal((1, 200, 2, 128)) * 3).astype(np.float16)
        oracle.append_side(codec, side, c, 1, 2, cap, [0], [200], x)
        for h in range(2):
            want = np.abs(oracle.dequant_stream(codec, side, c, 2, cap, 0, h, 200)).max()
            assert oracle.stream_absmax(codec, side, c, 2, cap, 0, h, 200) == want
        assert oracle.stream_absmax(codec, side, c, 2, cap, 0, 1, 0) == 0.0


def test_append_is_identical_on_one_thread_and_on_all():
    rng = np.random.default_rng(79)
    cap = 512
    x = rng.standard_normal((2, 400, 3, 128)).astype(np.float16)
    for codec in (0, 1, 2, 3):
        a = np.zeros(oracle.cache_bytes(codec, 2, 3, cap), np.uint8)
        b = np.zeros_like(a)
        with oracle.threads(1):
            oracle.append_side(codec, 1, a, 2, 3, cap, [5, 0], [395, 400], x)
        oracle.append_side(codec, 1, b, 2, 3, cap, [5, 0], [395, 400], x)
        assert np.array_equal(a, b)


def test_requantize_compact_and_probe_are_identical_on_one_thread_and_on_all():
    """Rows, streams and tokens are independent in these three: the bytes (and
    the probe mass, whose normaliser is summed on one thread in token order)
    must not depend on the thread count."""
    rng = np.random.default_rng(83)
    cap, n_kv, n_seqs = 512, 2, 2
    lens = [400, 137]
    x = rng.standard_normal((n_seqs, 400, n_kv, 128)).astype(np.float16)
    for src, dst in ((0, 1), (1, 2), (2, 3), (3, 0)):
        c = np.zeros(oracle.cache_bytes(src, n_seqs, n_kv, cap), np.uint8)
        oracle.append_side(src, 0, c, n_seqs, n_kv, cap, [0, 0], lens, x)
        with oracle.threads(1):
            a = oracle.requantize_side(src, dst, 0, c, n_seqs, n_kv, cap, lens)
        b = oracle.requantize_side(src, dst, 0, c, n_seqs, n_kv, cap, lens)
        assert np.array_equal(a, b)
        ev = [np.sort(rng.choice(lens[s], lens[s] // 4, replace=False)).astype(np.int32)
              for s in range(n_seqs)]
        with oracle.threads(1):
            ca = oracle.compact_side(src, 0, c, n_seqs, n_kv, cap, lens, ev)
        cb = oracle.compact_side(src, 0, c, n_seqs, n_kv, cap, lens, ev)
        assert np.array_equal(ca, cb)
        q = rng.standard_normal((n_seqs, 8, 128)).astype(np.float16)
        with oracle.threads(1):
            ma = oracle.probe_mass(src, c, n_seqs, n_kv, 8, cap, lens, q, 0.088)
        mb = oracle.probe_mass(src, c, n_seqs, n_kv, 8, cap, lens, q, 0.088)
        assert np.array_equal(ma, mb)
