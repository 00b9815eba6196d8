"""Pins for the oracle's indexer score and exact top-k.

Checks: brute-force pure-Python loops on tiny inputs, one-hot special cases
that read the score straight from the decoded row, the all-zero query (every
score 0, so the tie break alone decides), constant keys, and top-k against a
full Python sort on random and adversarial orders."""

import math

import numpy as np
import pytest

from oracle import codecs as C
from oracle import indexer as I
from synth import decode_case, to_bf16_bits


def _loops_score(idx_rows, q_bits, w):
    """Score by explicit loops over rows, heads and elements, decoding each
    nibble and scale byte by hand with the pinned element tables."""
    e2m1 = [float(v) for v in C.e2m1_decode(np.arange(16))]
    q = C.bf16_decode(q_bits)
    out = []
    for row in idx_rows:
        k = []
        for j in range(128):
            b = int(row[j // 2])
            code = (b & 0xF) if j % 2 == 0 else (b >> 4)
            k.append(e2m1[code] * 2.0 ** (int(row[64 + j // 32]) - 127))
        s = 0.0
        for h in range(q.shape[0]):
            d = math.fsum(float(q[h, j]) * k[j] for j in range(128))
            s += float(w[h]) * max(0.0, d)
        out.append(s)
    return np.array(out)


def test_score_matches_loops():
    case = decode_case(12, 5)
    rows = C.pack_idx_rows(case["idx_in"])
    got = I.score_rows(rows, case["q_idx"], case["w"])
    ref = _loops_score(rows, case["q_idx"], case["w"])
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-13)


def test_one_hot_reads_the_row():
    case = decode_case(64, 6)
    rows = C.pack_idx_rows(case["idx_in"])
    k = C.unpack_idx_rows(rows)
    for j in (0, 1, 31, 32, 77, 127):
        q = np.zeros((64, 128), dtype=np.float32)
        q[3, j] = 1.0
        w = np.zeros(64, dtype=np.float32)
        w[3] = 1.0
        s = I.score_rows(rows, to_bf16_bits(q), w)
        assert np.array_equal(s, np.maximum(k[:, j], 0.0))
    # a negative one-hot query flips the sign before the ReLU
    q = np.zeros((64, 128), dtype=np.float32)
    q[0, 5] = -2.0
    w = np.zeros(64, dtype=np.float32)
    w[0] = 0.5
    s = I.score_rows(rows, to_bf16_bits(q), w)
    assert np.array_equal(s, 0.5 * np.maximum(-2.0 * k[:, 5], 0.0))


def test_zero_query_ties_break_to_lower_index():
    case = decode_case(2000, 7)
    rows = C.pack_idx_rows(case["idx_in"])
    idx, val, s = I.score_topk(rows, np.zeros((64, 128), np.uint16), case["w"], 512)
    assert np.all(s == 0)
    assert np.array_equal(idx, np.arange(512))


def test_constant_keys_all_equal():
    row = np.random.default_rng(1).standard_normal(128).astype(np.float32)
    rows = C.pack_idx_rows(np.tile(row, (700, 1)))
    case = decode_case(1, 8)
    idx, val, s = I.score_topk(rows, case["q_idx"], case["w"], 512)
    assert np.all(s == s[0])
    assert np.array_equal(idx, np.arange(512))


def _sort_topk(scores, k):
    order = sorted(range(len(scores)), key=lambda t: (-scores[t], t))[:k]
    return order + [-1] * (k - len(order))


@pytest.mark.parametrize("kind", ["random", "ascending", "descending", "equal", "few_values"])
def test_topk_against_full_sort(kind):
    rng = np.random.default_rng(2)
    n = 3000
    s = {"random": rng.standard_normal(n),
         "ascending": np.arange(n, dtype=np.float64),
         "descending": -np.arange(n, dtype=np.float64),
         "equal": np.full(n, 1.5),
         "few_values": rng.integers(0, 4, n).astype(np.float64)}[kind]
    for k in (1, 7, 512):
        idx, val = I.topk(s, k)
        assert list(idx) == _sort_topk(list(s), k)
        assert np.array_equal(val, s[idx])


def test_topk_fewer_rows_than_k_pads():
    s = np.array([0.5, 2.0, 2.0, -1.0])
    idx, val = I.topk(s, 6)
    assert list(idx) == [1, 2, 0, 3, -1, -1]
    assert np.isnan(val[4]) and np.isnan(val[5])
