"""The micro-batched decode and the chunked prefill at their full sizes.

* 16 sessions with lengths uniform on [8192, 65536] (seed 1003, about
  590,000 rows in all): one batched scorer launch and one batched attention
  launch; every session's top-512 and attention against the oracle (the
  attention over the GPU's own list, reading R18).
* A prefill chunk of 2048 query tokens over 65,536 rows, query i seeing
  rows t < 63488 + i (seed 1004): the query quantiser bit-exact on every
  vector; the per-query exact top-512 of every query computed on the GPU and
  checked for a seeded sample of 32 queries (the first and the last among
  them); the per-query attention over the GPU's lists for the same sample.
  Each score CTA streams a query pair's ~496 visible tiles, and each query's
  top-k runs over ~64K scores: the histogram passes, not the in-memory path.
"""

import numpy as np
import pytest
import torch

from gpu_path import bf16_dev, bf16_host_bits, dev, new_ws, pack, require_gpu
from oracle import attention as A
from oracle import codecs as C
from oracle import indexer as I
from oracle import prefill as P
from parity import SOFTMAX_SCALE, check_attention, check_topk
from synth import prefill_case, sessions_case

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _ptrs(ts):
    return torch.tensor([t.data_ptr() for t in ts], dtype=torch.int64, device="cuda")


def test_sixteen_sessions_full_lengths():
    B = require_gpu()
    sess = sessions_case(n_sess=16)
    assert all(8192 <= s["n"] <= 65536 for s in sess)
    idx_rows, kv_rows = [], []
    for s in sess:
        i, kv = pack(idx_in=s["idx_in"], kv_in=s["kv_in"])
        idx_rows.append(i)
        kv_rows.append(kv)
    n = torch.tensor([s["n"] for s in sess], dtype=torch.int64, device="cuda")
    q = bf16_dev(np.stack([s["q_idx"] for s in sess]))
    w = dev(np.stack([s["w"] for s in sess]))
    k = 512
    out_idx = torch.empty((16, k), dtype=torch.int32, device="cuda")
    out_score = torch.empty((16, k), dtype=torch.float32, device="cuda")
    ws = new_ws(B.ds4x_index_score_topk_batched_workspace(16, k))
    qa = np.stack([s["q_attn"] for s in sess])
    out = torch.empty((16, 64, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((16, 64), dtype=torch.float32, device="cuda")
    ws_a = new_ws(B.ds4x_sparse_attn_decode_workspace(k))
    for _ in range(2):  # the second step reuses both workspaces
        B.ds4x_index_score_topk_batched(_ptrs(idx_rows), n, q, w, k, out_idx, out_score, ws)
        B.ds4x_sparse_attn_decode_batched(_ptrs(kv_rows), n, out_idx, k, bf16_dev(qa), SOFTMAX_SCALE, out, lse, ws_a)
        torch.cuda.synchronize()
        assert B.ds4x_workspace_status(ws) == 0
        assert B.ds4x_workspace_status(ws_a) == 0
        gi, gs = out_idx.cpu().numpy(), out_score.cpu().numpy()
        got, got_lse = bf16_host_bits(out), lse.cpu().numpy()
        for j, s in enumerate(sess):
            rows_o = C.pack_idx_rows(s["idx_in"])
            assert np.array_equal(idx_rows[j].cpu().numpy().reshape(s["n"], 68), rows_o), j
            check_topk(gi[j], gs[j], I.score_rows(rows_o, s["q_idx"], s["w"]), k)
            sel_o = C.pack_kv_rows(s["kv_in"][gi[j]])
            ref_out, _, ref_lse = A.sparse_attn_decode(sel_o, np.arange(k), s["q_attn"], SOFTMAX_SCALE)
            check_attention(got[j], ref_out)
            np.testing.assert_allclose(got_lse[j], ref_lse, rtol=1e-5, atol=1e-5)


def test_prefill_chunk_2048_queries_65536_rows():
    B = require_gpu()
    case = prefill_case()
    T, n, base, k = case["T"], case["n"], case["causal_base"], 512
    assert (T, n, base) == (2048, 65536, 63488)
    idx_rows, kv_rows = pack(idx_in=case["idx_in"], kv_in=case["kv_in"])
    rows_o = C.pack_idx_rows(case["idx_in"])
    assert np.array_equal(idx_rows.cpu().numpy().reshape(n, 68), rows_o)

    q = dev(case["q"])
    codes = torch.empty(T * 64 * 128, dtype=torch.uint8, device="cuda")
    scales = torch.empty(T * 64 * 4, dtype=torch.uint8, device="cuda")
    B.ds4x_quantize_query_e4m3(q, codes, scales)
    oc, os_ = P.quantize_query_e4m3(case["q"])
    assert np.array_equal(codes.cpu().numpy().reshape(T, 64, 128), oc)
    assert np.array_equal(scales.cpu().numpy().reshape(T, 64, 4), os_)

    out_idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    out_score = torch.empty((T, k), dtype=torch.float32, device="cuda")
    ws = new_ws(B.ds4x_index_score_topk_prefill_workspace(n, T, k))
    B.ds4x_index_score_topk_prefill(idx_rows, n, codes, scales, dev(case["w"]), T, base, k, out_idx, out_score, ws)
    out = torch.empty((T, 64, 512), dtype=torch.bfloat16, device="cuda")
    ws_a = new_ws(B.ds4x_sparse_attn_decode_workspace(k))
    B.ds4x_sparse_attn_prefill(kv_rows, n, out_idx, T, k, bf16_dev(case["q_attn"]), SOFTMAX_SCALE, out, None, ws_a)
    torch.cuda.synchronize()
    assert B.ds4x_workspace_status(ws) == 0
    assert B.ds4x_workspace_status(ws_a) == 0

    rng = np.random.default_rng(2048)
    queries = np.unique(np.concatenate([[0, T - 1], rng.choice(T, size=30, replace=False)]))
    o_idx, o_val, s = P.prefill_topk(rows_o, oc, os_, case["w"], base, k, queries=queries)
    gi, gs = out_idx.cpu().numpy(), out_score.cpu().numpy()
    got = bf16_host_bits(out)
    for r, i in enumerate(queries):
        vis = base + int(i)
        assert np.all(np.isfinite(s[r, :vis])) and np.all(np.isneginf(s[r, vis:]))
        check_topk(gi[i], gs[i], s[r, :vis], k)
        sel_o = C.pack_kv_rows(case["kv_in"][gi[i]])
        ref_out, _, _ = A.sparse_attn_decode(sel_o, np.arange(k), case["q_attn"][i], SOFTMAX_SCALE)
        check_attention(got[i], ref_out)
