"""Pins for the oracle's decode attention over the selected compressed rows
plus the raw sliding window (the next widening row).

w = 0 is the sparse attention (written separately); no selected rows is the
dense attention over the window in logical order; the whole is the
log-sum-exp merge of the two parts (the pinned combine); rotating the ring's
physical storage (and its newest slot with it) changes nothing; a window
that wraps past slot 0 reads the right slots; one window row alone returns
that row; nothing selected and an empty window give zeros and -inf."""

import math

import numpy as np

from oracle import codecs as C
from oracle.attention import dense_attn_decode, lse_combine, sparse_attn_decode, window_sparse_attn_decode
from synth import decode_case

SCALE = 1.0 / math.sqrt(512.0)
R = 256


def _case(seed, n=900):
    a = decode_case(n, seed)
    b = decode_case(R, seed + 100)
    rows = C.pack_kv_rows(a["kv_in"])
    ring = C.pack_kv_rows(b["kv_in"])
    rng = np.random.default_rng(seed)
    idx = rng.choice(n, size=512, replace=False).astype(np.int64)
    return rows, ring, idx, a["q_attn"]


def _logical(ring, pos, w):
    return ring[[(pos - j) % R for j in range(w)]]


def test_no_window_is_the_sparse_attention():
    rows, ring, idx, q = _case(1)
    out, exact, lse = window_sparse_attn_decode(rows, idx, ring, 17, 0, q, SCALE)
    out_s, exact_s, lse_s = sparse_attn_decode(rows, idx, q, SCALE)
    np.testing.assert_allclose(exact, exact_s, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, lse_s, rtol=1e-13)


def test_no_selected_rows_is_the_dense_window():
    rows, ring, _, q = _case(2)
    pos, w = 200, 128
    _, exact, lse = window_sparse_attn_decode(rows, np.full(512, -1), ring, pos, w, q, SCALE)
    _, exact_d, lse_d = dense_attn_decode(_logical(ring, pos, w), w, q, SCALE)
    np.testing.assert_allclose(exact, exact_d, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, lse_d, rtol=1e-13)


def test_union_is_the_lse_merge_of_the_parts():
    rows, ring, idx, q = _case(3)
    pos, w = 40, 200
    _, exact, lse = window_sparse_attn_decode(rows, idx, ring, pos, w, q, SCALE)
    _, o_s, l_s = sparse_attn_decode(rows, idx, q, SCALE)
    _, o_w, l_w = dense_attn_decode(_logical(ring, pos, w), w, q, SCALE)
    o, l = lse_combine([(o_s, l_s), (o_w, l_w)])
    np.testing.assert_allclose(exact, o, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lse, l, rtol=1e-13)


def test_ring_rotation_changes_nothing():
    rows, ring, idx, q = _case(4)
    pos, w = 100, 256
    _, exact, lse = window_sparse_attn_decode(rows, idx, ring, pos, w, q, SCALE)
    for r in (1, 77, 255):
        rot = np.roll(ring, r, axis=0)  # slot s moves to s + r
        _, e2, l2 = window_sparse_attn_decode(rows, idx, rot, (pos + r) % R, w, q, SCALE)
        np.testing.assert_allclose(e2, exact, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(l2, lse, rtol=1e-13)


def test_window_wraps_past_slot_zero():
    rows, ring, idx, q = _case(5)
    pos, w = 3, 10  # slots 3, 2, 1, 0, 255, ..., 250
    _, exact, lse = window_sparse_attn_decode(rows, np.full(512, -1), ring, pos, w, q, SCALE)
    explicit = ring[[3, 2, 1, 0, 255, 254, 253, 252, 251, 250]]
    _, exact_d, lse_d = dense_attn_decode(explicit, 10, q, SCALE)
    np.testing.assert_allclose(exact, exact_d, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, lse_d, rtol=1e-13)


def test_one_window_row_alone_is_that_row():
    rows, ring, _, q = _case(6)
    out, _, lse = window_sparse_attn_decode(rows, np.full(512, -1), ring, 9, 1, q, SCALE)
    v = C.unpack_kv_rows(ring[9:10])[0]
    assert np.array_equal(out, np.tile(C.bf16_round(v), (64, 1)))
    np.testing.assert_allclose(lse, (C.bf16_decode(q) @ v) * SCALE, rtol=1e-14)


def test_nothing_at_all():
    rows, ring, _, q = _case(7)
    out, exact, lse = window_sparse_attn_decode(rows, np.full(512, -1), ring, 0, 0, q, SCALE)
    assert np.all(out == 0) and np.all(exact == 0) and np.all(np.isneginf(lse))
