"""Pins for the oracle's dense (HCA) decode attention and the split-KV
log-sum-exp combine.

Dense attention: one row returns the row; identical rows return the row with
lse = logit + log n; a zero query gives the mean of all rows; two rows follow
the closed-form logistic weight; a pure-Python loop agrees on a tiny case;
the sparse attention selecting every row (written separately) agrees; no rows
give zeros and -inf.  Combine: splitting the rows into tiles (some empty) and
combining the tiles' normalised outputs and LSEs reproduces the whole softmax,
the identity that makes score-split attention exact."""

import math

import numpy as np
import pytest

from oracle import codecs as C
from oracle.attention import dense_attn_decode, lse_combine, sparse_attn_decode
from synth import decode_case

SCALE = 1.0 / math.sqrt(512.0)


def _rows(n, seed):
    case = decode_case(n, seed)
    return C.pack_kv_rows(case["kv_in"]), case["q_attn"]


def test_dense_single_row():
    rows, q = _rows(1, 21)
    v = C.unpack_kv_rows(rows)[0]
    out, exact, lse = dense_attn_decode(rows, 1, q, SCALE)
    assert np.array_equal(out, np.tile(C.bf16_round(v), (64, 1)))
    np.testing.assert_allclose(lse, (C.bf16_decode(q) @ v) * SCALE, rtol=1e-14)


def test_dense_identical_rows():
    rows, q = _rows(4, 22)
    rep = np.tile(rows[1:2], (37, 1))
    v = C.unpack_kv_rows(rows[1:2])[0]
    _, exact, lse = dense_attn_decode(rep, 37, q, SCALE)
    np.testing.assert_allclose(exact, np.tile(v, (64, 1)), rtol=1e-13, atol=0)
    np.testing.assert_allclose(lse, (C.bf16_decode(q) @ v) * SCALE + math.log(37), rtol=1e-13)


def test_dense_zero_query_is_the_mean():
    rows, _ = _rows(300, 23)
    _, exact, lse = dense_attn_decode(rows, 300, np.zeros((64, 512), np.uint16), SCALE)
    mean = C.unpack_kv_rows(rows).mean(axis=0)
    np.testing.assert_allclose(exact, np.tile(mean, (64, 1)), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, np.full(64, math.log(300)), rtol=1e-14)


def test_dense_two_rows_closed_form():
    rows, q = _rows(2, 24)
    v = C.unpack_kv_rows(rows)
    gap = (C.bf16_decode(q) @ (v[0] - v[1])) * SCALE
    p0 = 1.0 / (1.0 + np.exp(-gap))
    _, exact, _ = dense_attn_decode(rows, 2, q, SCALE)
    ref = p0[:, None] * v[0] + (1.0 - p0)[:, None] * v[1]
    np.testing.assert_allclose(exact, ref, rtol=1e-12, atol=1e-13)


def test_dense_loops_tiny():
    rows, q = _rows(3, 25)
    v = C.unpack_kv_rows(rows)
    qd = C.bf16_decode(q)
    _, exact, lse = dense_attn_decode(rows, 3, q, SCALE)
    for h in (0, 17, 63):
        logits = [SCALE * sum(float(qd[h, d]) * float(v[t, d]) for d in range(512)) for t in range(3)]
        m = max(logits)
        ws = [math.exp(x - m) for x in logits]
        s = sum(ws)
        for d in (0, 100, 447, 448, 511):
            ref = sum(ws[t] * float(v[t, d]) for t in range(3)) / s
            assert abs(exact[h, d] - ref) <= 1e-12 * max(1.0, abs(ref))
        assert abs(lse[h] - (m + math.log(s))) <= 1e-12 * max(1.0, abs(lse[h]))


def test_dense_equals_sparse_over_every_row():
    rows, q = _rows(700, 26)
    out_d, exact_d, lse_d = dense_attn_decode(rows, 650, q, SCALE)  # rows past n are not read
    out_s, exact_s, lse_s = sparse_attn_decode(rows, np.arange(650), q, SCALE)
    np.testing.assert_allclose(exact_d, exact_s, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse_d, lse_s, rtol=1e-13)


def test_dense_no_rows():
    rows, q = _rows(5, 27)
    out, exact, lse = dense_attn_decode(rows, 0, q, SCALE)
    assert np.all(out == 0) and np.all(exact == 0) and np.all(np.isneginf(lse))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_lse_combine_split_identity(seed):
    n = 3000
    rows, q = _rows(n, 30 + seed)
    _, whole, lse_whole = dense_attn_decode(rows, n, q, SCALE)
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.choice(np.arange(1, n), size=11, replace=False))
    bounds = [0, *cuts.tolist(), cuts[-1], n]  # one empty tile (cuts[-1] twice)
    parts = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        _, o, l = sparse_attn_decode(rows, np.arange(a, b), q, SCALE)
        parts.append((o, l))
    o, lse = lse_combine(parts)
    np.testing.assert_allclose(o, whole, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lse, lse_whole, rtol=1e-13)


def test_lse_combine_degenerate():
    rows, q = _rows(40, 40)
    _, o, l = dense_attn_decode(rows, 40, q, SCALE)
    o1, l1 = lse_combine([(o, l)])
    np.testing.assert_allclose(o1, o, rtol=1e-15)
    np.testing.assert_allclose(l1, l, rtol=1e-15)
    empty = (np.zeros_like(o), np.full(64, -np.inf))
    o2, l2 = lse_combine([empty, (o, l), empty])
    np.testing.assert_allclose(o2, o, rtol=1e-15)
    np.testing.assert_allclose(l2, l, rtol=1e-15)
    o3, l3 = lse_combine([empty, empty])
    assert np.all(o3 == 0) and np.all(np.isneginf(l3))
