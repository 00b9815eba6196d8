"""Chunked-prefill scoring: the query quantiser (bit-exact) and the per-query
causal top-k against the oracle."""

import numpy as np
import pytest
import torch

from gpu_path import dev, new_ws, pack, require_gpu
from oracle import codecs as C
from oracle import prefill as P
from parity import check_topk
from synth import prefill_case

pytestmark = pytest.mark.gpu


def _quantize(q):
    B = require_gpu()
    q = np.ascontiguousarray(q, dtype=np.float32)
    n = q.size // 128
    codes = torch.empty(n * 128, dtype=torch.uint8, device="cuda")
    scales = torch.empty(n * 4, dtype=torch.uint8, device="cuda")
    B.ds4x_quantize_query_e4m3(dev(q), codes, scales)
    torch.cuda.synchronize()
    return codes.cpu().numpy().reshape(*q.shape[:-1], 128), scales.cpu().numpy().reshape(*q.shape[:-1], 4)


def test_query_quantiser_bit_exact():
    case = prefill_case(T=64, n=16, causal_base=0)
    gc, gs = _quantize(case["q"])
    oc, os_ = P.quantize_query_e4m3(case["q"])
    assert np.array_equal(gc, oc)
    assert np.array_equal(gs, os_)


def test_query_quantiser_special_blocks():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((6, 128)).astype(np.float32)
    q[0, :32] = 0.0                                        # all-zero block: scale byte 127
    q[1, 32:64] = -1e-30                                   # tiny negatives keep their sign
    q[2, :] *= np.float32(2.0 ** 40)                       # large scale
    q[3, 64:96] = np.float32(448.0)                        # exactly emax
    grid = C.e4m3_decode(np.arange(0x7f, dtype=np.uint8))
    mids = (grid[1:] + grid[:-1]) / 2                      # rounding midpoints (ties to even)
    q[4, :] = np.resize(mids[-60:], 128).astype(np.float32)
    q[5, :] = -np.resize(mids[:64], 128).astype(np.float32) * np.float32(2.0 ** -20)
    gc, gs = _quantize(q)
    oc, os_ = P.quantize_query_e4m3(q)
    assert np.array_equal(gc, oc)
    assert np.array_equal(gs, os_)


@pytest.mark.parametrize("T,n,base,k", [(24, 6000, 5000, 512), (70, 3000, 400, 512), (5, 2000, 2500, 100)])
def test_prefill_topk_parity(T, n, base, k):
    B = require_gpu()
    case = prefill_case(T=T, n=n, causal_base=base)
    idx_rows, _ = pack(idx_in=case["idx_in"])
    codes, scales = P.quantize_query_e4m3(case["q"])
    out_idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    out_score = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ws = new_ws(B.ds4x_index_score_topk_prefill_workspace(n, T, k))
    B.ds4x_index_score_topk_prefill(idx_rows, n, dev(codes), dev(scales), dev(case["w"]), T, base, k, out_idx,
                                    out_score, ws)
    torch.cuda.synchronize()
    assert B.ds4x_workspace_status(ws) == 0
    gi, gs = out_idx.cpu().numpy(), out_score.cpu().numpy()
    rows = C.pack_idx_rows(case["idx_in"])
    s = P.prefill_scores(rows, codes, scales, case["w"], base)
    for i in range(T):
        vis = int(np.sum(np.isfinite(s[i])))
        assert vis == min(n, base + i)
        check_topk(gi[i], gs[i], s[i, :vis], k)


def _score_prefill(idx_rows, n, codes, scales, w, T, base, k):
    B = require_gpu()
    out_idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    out_score = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ws = new_ws(B.ds4x_index_score_topk_prefill_workspace(n, T, k))
    B.ds4x_index_score_topk_prefill(idx_rows, n, dev(codes), dev(scales), dev(w), T, base, k, out_idx, out_score, ws)
    torch.cuda.synchronize()
    assert B.ds4x_workspace_status(ws) == 0
    return out_idx.cpu().numpy(), out_score.cpu().numpy()


def test_prefill_all_scores_equal_lowest_rows_win():
    """20,000 copies of one row: every visible score of a query is the same,
    more than the top-k kernel holds in shared memory, so the tie is broken
    by the index-order pass: rows 0..k-1 exactly."""
    require_gpu()
    n, T, base, k = 20000, 5, 19998, 512
    case = prefill_case(T=T, n=1, causal_base=0)
    idx_in = np.tile(case["idx_in"][:1], (n, 1))
    idx_rows, _ = pack(idx_in=idx_in)
    codes, scales = P.quantize_query_e4m3(case["q"])
    gi, gs = _score_prefill(idx_rows, n, codes, scales, case["w"], T, base, k)
    s = P.prefill_scores(C.pack_idx_rows(idx_in[:1]), codes, scales, case["w"], 1)[:, 0]
    for i in range(T):
        assert np.array_equal(gi[i], np.arange(k)), i
        assert np.all(gs[i] == gs[i, 0])
        np.testing.assert_allclose(gs[i, 0], s[i], rtol=2e-5)


def test_prefill_one_hot_queries_wide_buckets():
    """One-hot queries (code 1.0 at one element of one head, one-hot weights):
    every score is one E2M1 key value times a power of two, so thousands of
    rows share the k-th score; the histogram passes narrow to it and the
    index-order pass breaks the tie.  The scores are exact in fp32, so the
    lists must equal the oracle's, order included."""
    require_gpu()
    n, T, base, k = 30000, 6, 29995, 512
    case = prefill_case(T=T, n=n, causal_base=base)
    idx_rows, _ = pack(idx_in=case["idx_in"])
    codes = np.zeros((T, 64, 128), dtype=np.uint8)
    scales = np.full((T, 64, 4), 127, dtype=np.uint8)
    w = np.zeros((T, 64), dtype=np.float32)
    for i in range(T):
        h, e = (5 * i + 3) % 64, (37 * i + 11) % 128
        codes[i, h, e] = 0x38  # 1.0
        w[i, h] = 1.0 if i % 2 == 0 else 0.25
        if i == 3:  # a negative weight: most scores zero or below
            w[i, h] = -1.0
    gi, gs = _score_prefill(idx_rows, n, codes, scales, w, T, base, k)
    rows = C.pack_idx_rows(case["idx_in"])
    o_idx, o_val, s = P.prefill_topk(rows, codes, scales, w, base, k)
    for i in range(T):
        vis = min(n, base + i)
        check_topk(gi[i], gs[i], s[i, :vis], k)
        assert np.array_equal(gi[i], o_idx[i]), i
        assert np.array_equal(gs[i].astype(np.float64), o_val[i]), i
