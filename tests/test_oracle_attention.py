"""Pins for the oracle's sparse decode attention.

Checks: a single selected row returns that row, identical rows return the
row, a zero query averages the rows, two rows with a known logit gap follow
the closed-form logistic weight, -1 padding is skipped, and pure-Python loops
agree on a tiny case."""

import math

import numpy as np

from oracle import codecs as C
from oracle.attention import sparse_attn_decode
from synth import decode_case, to_bf16_bits

SCALE = 1.0 / math.sqrt(512.0)


def _rows(n, seed):
    case = decode_case(n, seed)
    return C.pack_kv_rows(case["kv_in"]), case["q_attn"]


def test_single_row_returns_the_row():
    rows, q = _rows(50, 1)
    v = C.unpack_kv_rows(rows[17:18])[0]
    out, exact, lse = sparse_attn_decode(rows, [17], q, SCALE)
    assert np.array_equal(out, np.tile(C.bf16_round(v), (64, 1)))
    q64 = C.bf16_decode(q)
    np.testing.assert_allclose(lse, (q64 @ v) * SCALE, rtol=1e-14)


def test_identical_rows_return_the_row():
    rows, q = _rows(5, 2)
    rep = np.tile(rows[3:4], (9, 1))
    v = C.unpack_kv_rows(rows[3:4])[0]
    _, exact, lse = sparse_attn_decode(rep, np.arange(9), q, SCALE)
    # 9 * (v / 9) is v only up to fp64 rounding, so compare before the bf16
    # rounding (an FP16 RoPE value can sit exactly on a bf16 midpoint)
    np.testing.assert_allclose(exact, np.tile(v, (64, 1)), rtol=1e-14, atol=0)
    q64 = C.bf16_decode(q)
    np.testing.assert_allclose(lse, (q64 @ v) * SCALE + math.log(9), rtol=1e-13)


def test_zero_query_is_the_mean():
    rows, _ = _rows(40, 3)
    sel = [0, 5, 9, 39, 22]
    out, exact, _ = sparse_attn_decode(rows, sel, np.zeros((64, 512), np.uint16), SCALE)
    mean = C.unpack_kv_rows(rows[sel]).mean(axis=0)
    np.testing.assert_allclose(exact, np.tile(mean, (64, 1)), rtol=1e-14, atol=1e-15)


def test_two_rows_closed_form():
    rows, q = _rows(8, 4)
    v = C.unpack_kv_rows(rows[[2, 6]])
    q64 = C.bf16_decode(q)
    gap = (q64 @ (v[0] - v[1])) * SCALE
    p0 = 1.0 / (1.0 + np.exp(-gap))
    _, exact, _ = sparse_attn_decode(rows, [2, 6], q, SCALE)
    ref = p0[:, None] * v[0] + (1.0 - p0)[:, None] * v[1]
    np.testing.assert_allclose(exact, ref, rtol=1e-12, atol=1e-14)


def test_padding_is_skipped():
    rows, q = _rows(30, 5)
    a = sparse_attn_decode(rows, [4, -1, 11, -1], q, SCALE)
    b = sparse_attn_decode(rows, [4, 11], q, SCALE)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[2], b[2])


def test_loops_tiny():
    rows, _ = _rows(6, 6)
    rng = np.random.default_rng(0)
    q = to_bf16_bits(rng.standard_normal((2, 512)).astype(np.float32))
    sel = [5, 0, 3]
    v = C.unpack_kv_rows(rows[sel])
    qd = C.bf16_decode(q)
    out, exact, lse = sparse_attn_decode(rows, sel, q, SCALE)
    for h in range(2):
        logits = [math.fsum(float(qd[h, d]) * float(v[j, d]) for d in range(512)) * SCALE for j in range(3)]
        m = max(logits)
        e = [math.exp(x - m) for x in logits]
        z = math.fsum(e)
        for d in range(0, 512, 37):
            o = math.fsum(e[j] * float(v[j, d]) for j in range(3)) / z
            assert abs(o - exact[h, d]) <= 1e-12 * max(1.0, abs(o))
        assert abs(lse[h] - (m + math.log(z))) < 1e-12
