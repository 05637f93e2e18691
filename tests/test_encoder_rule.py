"""The division-free rule of the GPU row encoders, checked against the oracle.

The kernels take the quotient x/d of the q8_0 and q4_0 (and turbo4) encoders
as t = RN(x * RN(1/d)) and read the integer from t (nearest integer of t for
q8_0, floor of u = RN(t + 8.5) for q4_0) wherever t is more than a margin away
from the encoder's rounding boundary (2^-14 from a half-integer for q8_0, u
2^-17 from an integer for q4_0), and divide exactly elsewhere.  This test
restates that rule in numpy float32 (IEEE round-to-nearest, like the GPU's
__fmul_rn / __fadd_rn / __frcp_rn) and checks that it gives exactly the codes
of the oracle's encoder (the written formula with IEEE divisions) on rows
whose quotients sit on or next to the boundaries, and on random rows.
"""
import numpy as np
import pytest

import oracle
from tests._helpers import boundary_rows

F32 = np.float32
MAGIC = F32(12582912.0)  # 1.5 * 2^23


def _rule_q8(x, d):
    r = (F32(1) / d).astype(F32)
    t = (x * r).astype(F32)
    tm = (t + MAGIC).astype(F32)
    dist = np.abs((t - (tm - MAGIC).astype(F32)).astype(F32))
    fast = np.abs((dist - F32(0.5)).astype(F32)) > F32(2.0 ** -14)
    q_fast = tm.view(np.int32).astype(np.int64) - 0x4B400000
    q_exact = (x / d).astype(F32).astype(np.float64)
    q_exact = (np.sign(q_exact) * np.floor(np.abs(q_exact) + 0.5)).astype(np.int64)
    return np.where(fast, q_fast, q_exact), fast


def _rule_q4(x, d):
    r = (F32(1) / d).astype(F32)
    u = ((x * r).astype(F32) + F32(8.5)).astype(F32)
    fm = ((u - F32(0.5)).astype(F32) + MAGIC).astype(F32)
    fr = (u - (fm - MAGIC).astype(F32)).astype(F32)
    fast = (fr > F32(2.0 ** -17)) & (fr < F32(1) - F32(2.0 ** -17))
    q_fast = fm.view(np.int32).astype(np.int64) - 0x4B400000
    q_exact = np.trunc(((x / d).astype(F32) + F32(8.5)).astype(F32)).astype(np.int64)
    return np.minimum(np.where(fast, q_fast, q_exact), 15), fast


def _oracle_codes(codec, rows):
    """Block scales (fp32) and codes of the oracle's canonical row bytes."""
    by = oracle.encode_rows(codec, rows).reshape(len(rows), 4, -1)
    d = by[:, :, 0:2].copy().view(np.float16).astype(np.float32)[:, :, 0]
    if codec == 1:
        q = by[:, :, 2:34].view(np.int8).astype(np.int64)
    else:
        b = by[:, :, 2:18].astype(np.int64)
        q = np.concatenate([b & 0xF, b >> 4], axis=2)
    return d, q


@pytest.mark.parametrize("codec", [1, 2])
@pytest.mark.parametrize("kind", ["boundary", "random"])
def test_division_free_rule_matches_the_oracle(codec, kind):
    rng = np.random.default_rng(70 + codec + (kind == "random"))
    if kind == "boundary":
        rows = boundary_rows(codec, 96, rng)
    else:
        rows = (rng.standard_normal((512, 128)) * 10.0 ** rng.uniform(-4, 3, (512, 1))
                ).astype(np.float16)
    x = rows.astype(np.float32).reshape(-1, 4, 32)
    # the encoder's fp32 scale d (before its fp16 rounding), as the kernels compute it
    if codec == 1:
        d = (np.abs(x).max(axis=2, keepdims=True) / F32(127)).astype(F32)
    else:
        m = np.take_along_axis(x, np.argmax(np.abs(x), axis=2)[:, :, None], axis=2)
        d = (m / F32(-8)).astype(F32)
    ok = d[:, :, 0] != 0
    xx, dd = x[ok], np.broadcast_to(d, x.shape)[ok]
    q, fast = (_rule_q8 if codec == 1 else _rule_q4)(xx, dd)
    d16, q_ref = _oracle_codes(codec, rows)
    assert np.array_equal(q, q_ref[ok]), "rule and oracle disagree"
    assert np.array_equal(d.astype(np.float16).astype(np.float32)[:, :, 0], d16)
    if kind == "boundary":
        assert (~fast).sum() > 100, "boundary rows must exercise the exact-division path"
