"""Parity at the full decode sizes, through the C ABI against the oracle.

The scorer's grid has one CTA per SM, each streaming a contiguous range of
128-row tiles.  Only at these sizes does every CTA stream enough tiles for
the paths that small cases never reach:

* mid decode, 131,072 rows (seed 1001): 7 tiles per CTA;
* long decode, 1,048,576 rows (seed 1002): 54 tiles per CTA, so the
  stage, A and accumulator rings wrap many times in the two-piece (hi + lo)
  query mode;
* 2**21 rows (indexer only, seed 1005): 108 tiles per CTA, past the 64-tile
  chunk, so the chunk-end carry and cut run; with adversarial row orders,
  constant keys and a one-hot query with a negative weight the boundary
  buckets hold thousands of keys, so the exact selections (a carried set
  beyond 1,024 keys, a candidate bucket beyond the candidate array) and the
  exact fallback merge run too.

Checks: packed rows bit-exact; the top-512 set equal to the oracle's except
rows within 1e-5 relative of the 512th oracle score (exactly equal, order
included, where every score is exact in fp32); attention over the GPU's own
list (R18) within max |diff| 2e-3 and rel-L2 1e-3 of the bf16-rounded
oracle.
"""

import numpy as np
import pytest
import torch

from gpu_path import attention, fallback_merges, new_ws, pack, require_gpu, score_topk
from oracle import attention as A
from oracle import codecs as C
from oracle import indexer as I
from parity import SOFTMAX_SCALE, check_attention, check_topk
from synth import indexer_case, to_bf16_bits, workload

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

BIG_N = 1 << 21
BIG_SEED = 1005


def _decode_parity(name):
    require_gpu()
    case = workload(name)
    n = case["n"]
    idx_rows, kv_rows = pack(idx_in=case["idx_in"], kv_in=case["kv_in"])
    rows_o = C.pack_idx_rows(case["idx_in"])
    assert np.array_equal(idx_rows.cpu().numpy().reshape(n, 68), rows_o), "packed indexer rows differ"
    # KV rows: every row at the mid size, a strided sample (plus the last rows) at the long size
    stride = 1 if n <= 131072 else 7
    sample = np.unique(np.concatenate([np.arange(0, n, stride), np.arange(n - 64, n)]))
    kv_o = C.pack_kv_rows(case["kv_in"][sample])
    kv_g = kv_rows.view(n, 583)[torch.from_numpy(sample).cuda()].cpu().numpy()
    assert np.array_equal(kv_g, kv_o), "packed KV rows differ"

    s = I.score_rows(rows_o, case["q_idx"], case["w"])
    gi, gs = score_topk(idx_rows, n, case["q_idx"], case["w"], 512)
    check_topk(gi, gs, s, 512)

    # attention over the GPU's own list, the oracle packing those rows itself
    out, lse, ws = attention(kv_rows, n, gi, case["q_attn"], SOFTMAX_SCALE)
    B = require_gpu()
    assert B.ds4x_workspace_status(ws) == 0
    sel_o = C.pack_kv_rows(case["kv_in"][gi])
    ref_out, _, ref_lse = A.sparse_attn_decode(sel_o, np.arange(512), case["q_attn"], SOFTMAX_SCALE)
    check_attention(out, ref_out)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-5, atol=1e-5)


def test_mid_decode_131072_rows():
    _decode_parity("mid")


def test_long_decode_1048576_rows():
    _decode_parity("long")


@pytest.fixture(scope="module")
def big():
    """2**21 packed indexer rows on the GPU and in the oracle."""
    require_gpu()
    case = indexer_case(BIG_N, BIG_SEED)
    idx_rows, _ = pack(idx_in=case["idx_in"])
    rows_o = C.pack_idx_rows(case["idx_in"])
    assert np.array_equal(idx_rows.cpu().numpy().reshape(BIG_N, 68), rows_o), "packed indexer rows differ"
    s = I.score_rows(rows_o, case["q_idx"], case["w"])
    return {"case": case, "rows": idx_rows, "rows_o": rows_o, "s": s}


def _permuted(big, perm):
    """The same packed rows in another order, on the GPU; row t of the
    result is row perm[t] of the original (the oracle's scores follow)."""
    rows = big["rows"].view(BIG_N, 68)[torch.from_numpy(perm).cuda()].contiguous().view(-1)
    return rows, big["s"][perm]


def test_chunk_carry_2m_rows(big):
    """108 tiles per CTA: two chunks, the first cut carried into the second."""
    c = big["case"]
    gi, gs = score_topk(big["rows"], BIG_N, c["q_idx"], c["w"], 512)
    check_topk(gi, gs, big["s"], 512)


@pytest.mark.parametrize("k", [1, 100])
def test_chunk_carry_2m_rows_small_k(big, k):
    c = big["case"]
    gi, gs = score_topk(big["rows"], BIG_N, c["q_idx"], c["w"], k)
    check_topk(gi, gs, big["s"], k)


@pytest.mark.parametrize("order", ["ascending", "descending"])
def test_adversarial_orders_2m_rows(big, order):
    """Rows sorted by score: ascending puts every winner in the last CTA's
    range (its bound beats the k-th key: the exact fallback merge);
    descending puts them all in the first."""
    perm = np.argsort(big["s"], kind="stable")
    if order == "descending":
        perm = perm[::-1].copy()
    rows, s = _permuted(big, perm)
    c = big["case"]
    gi, gs, ws = score_topk(rows, BIG_N, c["q_idx"], c["w"], 512, return_ws=True)
    check_topk(gi, gs, s, 512)
    # one CTA holds every winner: its bound beats the k-th candidate
    assert fallback_merges(ws) == 1


def test_constant_keys_2m_rows():
    """Every row the same: every key of a chunk lands in one bucket, so the
    carried set exceeds 1,024 keys and is cut exactly, and the candidate
    bucket exceeds the candidate array (exact top-M); the tie break by
    index then gives rows 0..511 exactly."""
    require_gpu()
    c = indexer_case(1, BIG_SEED + 1)
    row = torch.from_numpy(c["idx_in"]).cuda()
    B = require_gpu()
    idx_rows = torch.zeros(BIG_N * 68, dtype=torch.uint8, device="cuda")
    B.ds4x_cache_append(None, idx_rows, 0, None, row.expand(BIG_N, 128).contiguous())
    one_o = C.pack_idx_rows(c["idx_in"])
    assert np.array_equal(idx_rows.view(BIG_N, 68)[:: 4099].cpu().numpy(), np.repeat(one_o, (BIG_N + 4098) // 4099, 0))
    s1 = I.score_rows(one_o, c["q_idx"], c["w"])[0]
    gi, gs = score_topk(idx_rows, BIG_N, c["q_idx"], c["w"], 512)
    assert np.array_equal(gi, np.arange(512))
    assert np.all(gs == gs[0])
    np.testing.assert_allclose(gs[0], s1, rtol=2e-5)


def test_one_hot_query_negative_weight_2m_rows(big):
    """Scores max(0, k_t[100]) - 2 max(0, -0.5 k_t[3]): most are <= 0 (one
    histogram bucket) and the positive ones take few distinct values, so the
    boundary buckets are wide.  Every score is exact in fp32, so the GPU
    list must equal the oracle's top-512, order and ties included."""
    q = np.zeros((64, 128), dtype=np.float32)
    q[7, 100] = 1.0
    q[8, 3] = -0.5
    w = np.zeros(64, dtype=np.float32)
    w[7] = 1.0
    w[8] = -2.0
    qb = to_bf16_bits(q)
    s = I.score_rows(big["rows_o"], qb, w)
    o_idx, o_val = I.topk(s, 512)
    gi, gs = score_topk(big["rows"], BIG_N, qb, w, 512)
    check_topk(gi, gs, s, 512)
    assert np.array_equal(gi, o_idx)
    assert np.array_equal(gs.astype(np.float64), o_val)


def test_scorer_workspace_reused_across_sizes(big):
    """One workspace, calls of growing and shrinking size in a row (the
    exchange words of each call are cleared for the next one)."""
    B = require_gpu()
    c = big["case"]
    ws = new_ws(B.ds4x_index_score_topk_workspace(BIG_N, 512))
    out_idx = torch.empty(512, dtype=torch.int32, device="cuda")
    out_score = torch.empty(512, dtype=torch.float32, device="cuda")
    from gpu_path import bf16_dev, dev

    q, w = bf16_dev(c["q_idx"]), dev(c["w"])
    for n in (BIG_N, 5000, 700_000, BIG_N, 129):
        B.ds4x_index_score_topk(big["rows"], n, q, w, 512, out_idx, out_score, ws)
        torch.cuda.synchronize()
        check_topk(out_idx.cpu().numpy(), out_score.cpu().numpy(), big["s"][:n], 512)
    assert B.ds4x_workspace_status(ws) == 0
