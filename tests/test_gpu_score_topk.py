"""ds4x_index_score_topk vs the oracle's score + exact top-k."""

import numpy as np
import pytest

from gpu_path import pack, require_gpu, score_topk
from oracle import codecs as C
from oracle import indexer as I
from parity import check_topk
from synth import decode_case, to_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,k", [(4096, 512), (1, 512), (511, 512), (512, 512), (513, 512),
                                 (4097, 512), (10037, 512), (20000, 1), (20000, 7), (3000, 100)])
def test_score_topk_parity(n, k):
    require_gpu()
    case = decode_case(n, 2000 + n)
    idx_rows, _ = pack(idx_in=case["idx_in"])
    gi, gs = score_topk(idx_rows, n, case["q_idx"], case["w"], k)
    rows = C.pack_idx_rows(case["idx_in"])
    s = I.score_rows(rows, case["q_idx"], case["w"])
    check_topk(gi, gs, s, k)


def test_zero_query_breaks_ties_by_index():
    require_gpu()
    n = 5000
    case = decode_case(n, 11)
    idx_rows, _ = pack(idx_in=case["idx_in"])
    gi, gs = score_topk(idx_rows, n, np.zeros((64, 128), np.uint16), case["w"], 512)
    assert np.array_equal(gi, np.arange(512))
    assert np.all(gs == 0)


def test_constant_keys_tie_break():
    require_gpu()
    row = np.random.default_rng(1).standard_normal(128).astype(np.float32)
    idx_in = np.tile(row, (3000, 1))
    case = decode_case(1, 12)
    idx_rows, _ = pack(idx_in=idx_in)
    gi, gs = score_topk(idx_rows, 3000, case["q_idx"], case["w"], 512)
    assert np.array_equal(gi, np.arange(512))
    assert np.all(gs == gs[0])


@pytest.mark.parametrize("order", ["ascending", "descending"])
def test_adversarial_orders(order):
    """Rows sorted by score (every row a new candidate, or none after the first)."""
    require_gpu()
    n = 30000
    case = decode_case(n, 13)
    rows = C.pack_idx_rows(case["idx_in"])
    s = I.score_rows(rows, case["q_idx"], case["w"])
    perm = np.argsort(s, kind="stable")
    if order == "descending":
        perm = perm[::-1]
    idx_in = np.ascontiguousarray(case["idx_in"][perm])
    idx_rows, _ = pack(idx_in=idx_in)
    gi, gs = score_topk(idx_rows, n, case["q_idx"], case["w"], 512)
    check_topk(gi, gs, s[perm], 512)


def test_one_hot_query_and_negative_weights():
    require_gpu()
    n = 6000
    case = decode_case(n, 14)
    q = np.zeros((64, 128), dtype=np.float32)
    q[7, 100] = 1.0
    q[8, 3] = -0.5
    w = np.zeros(64, dtype=np.float32)
    w[7] = 1.0
    w[8] = -2.0  # negative scores must order correctly too
    qb = to_bf16_bits(q)
    idx_rows, _ = pack(idx_in=case["idx_in"])
    gi, gs = score_topk(idx_rows, n, qb, w, 512)
    rows = C.pack_idx_rows(case["idx_in"])
    check_topk(gi, gs, I.score_rows(rows, qb, w), 512)
