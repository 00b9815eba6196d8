"""Micro-batched decode (ragged independent sessions, one launch each for
scoring and attention) and prefill attention (one launch over many query
tokens) against the oracle, session by session / query by query."""

import numpy as np
import pytest
import torch

from gpu_path import bf16_dev, bf16_host_bits, dev, new_ws, pack, require_gpu
from oracle import attention as A
from oracle import codecs as C
from oracle import indexer as I
from parity import SOFTMAX_SCALE, check_attention, check_topk
from synth import prefill_case, sessions_case

pytestmark = pytest.mark.gpu


def _pack_sessions(sess):
    idx_rows, kv_rows = [], []
    for s in sess:
        i, kv = pack(idx_in=s["idx_in"], kv_in=s["kv_in"])
        idx_rows.append(i)
        kv_rows.append(kv)
    return idx_rows, kv_rows


def _ptrs(ts):
    return torch.tensor([t.data_ptr() for t in ts], dtype=torch.int64, device="cuda")


@pytest.mark.parametrize("n_sess,scale,k", [(16, 0.0625, 512), (3, 0.02, 100), (1, 0.01, 512)])
def test_batched_score_topk_per_session(n_sess, scale, k):
    B = require_gpu()
    sess = sessions_case(n_sess=n_sess, scale_lengths=scale)
    idx_rows, _ = _pack_sessions(sess)
    n = torch.tensor([s["n"] for s in sess], dtype=torch.int64, device="cuda")
    q = bf16_dev(np.stack([s["q_idx"] for s in sess]))
    w = dev(np.stack([s["w"] for s in sess]))
    out_idx = torch.empty((n_sess, k), dtype=torch.int32, device="cuda")
    out_score = torch.empty((n_sess, k), dtype=torch.float32, device="cuda")
    ws = new_ws(B.ds4x_index_score_topk_batched_workspace(n_sess, k))
    for _ in range(2):  # the second call checks the per-session tickets reset
        B.ds4x_index_score_topk_batched(_ptrs(idx_rows), n, q, w, k, out_idx, out_score, ws)
        torch.cuda.synchronize()
        assert B.ds4x_workspace_status(ws) == 0
        gi, gs = out_idx.cpu().numpy(), out_score.cpu().numpy()
        for j, s in enumerate(sess):
            scores = I.score_rows(C.pack_idx_rows(s["idx_in"]), s["q_idx"], s["w"])
            check_topk(gi[j], gs[j], scores, k)


def test_batched_score_session_shorter_than_k():
    B = require_gpu()
    sess = sessions_case(n_sess=4, scale_lengths=0.01)
    sess[2] = dict(sess[2], n=300, idx_in=sess[2]["idx_in"][:300], kv_in=sess[2]["kv_in"][:300])
    idx_rows, _ = _pack_sessions(sess)
    n = torch.tensor([s["n"] for s in sess], dtype=torch.int64, device="cuda")
    q = bf16_dev(np.stack([s["q_idx"] for s in sess]))
    w = dev(np.stack([s["w"] for s in sess]))
    out_idx = torch.empty((4, 512), dtype=torch.int32, device="cuda")
    ws = new_ws(B.ds4x_index_score_topk_batched_workspace(4, 512))
    B.ds4x_index_score_topk_batched(_ptrs(idx_rows), n, q, w, 512, out_idx, None, ws)
    gi = out_idx.cpu().numpy()
    for j, s in enumerate(sess):
        scores = I.score_rows(C.pack_idx_rows(s["idx_in"]), s["q_idx"], s["w"])
        check_topk(gi[j], None, scores, 512)


def test_batched_attention_per_session():
    B = require_gpu()
    sess = sessions_case(n_sess=16, scale_lengths=0.03)
    _, kv_rows = _pack_sessions(sess)
    n = torch.tensor([s["n"] for s in sess], dtype=torch.int64, device="cuda")
    rng = np.random.default_rng(7)
    k = 512
    idx = np.stack([rng.choice(s["n"], size=k, replace=False) for s in sess]).astype(np.int32)
    q = np.stack([s["q_attn"] for s in sess])
    out = torch.empty((16, 64, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((16, 64), dtype=torch.float32, device="cuda")
    ws = new_ws(B.ds4x_sparse_attn_decode_workspace(k))
    B.ds4x_sparse_attn_decode_batched(_ptrs(kv_rows), n, dev(idx), k, bf16_dev(q), SOFTMAX_SCALE, out, lse, ws)
    torch.cuda.synchronize()
    assert B.ds4x_workspace_status(ws) == 0
    got = bf16_host_bits(out)
    got_lse = lse.cpu().numpy()
    for j, s in enumerate(sess):
        ref_out, _, ref_lse = A.sparse_attn_decode(C.pack_kv_rows(s["kv_in"]), idx[j], s["q_attn"], SOFTMAX_SCALE)
        check_attention(got[j], ref_out)
        np.testing.assert_allclose(got_lse[j], ref_lse, rtol=1e-5, atol=1e-5)


def test_prefill_attention_per_query():
    B = require_gpu()
    case = prefill_case(T=24, n=6000, causal_base=5000)
    _, kv_rows = pack(kv_in=case["kv_in"])
    rng = np.random.default_rng(8)
    T, k = case["T"], 512
    # each query's own rows, all visible to it (t < causal_base + i)
    idx = np.stack([rng.choice(case["causal_base"] + i, size=k, replace=False) for i in range(T)]).astype(np.int32)
    idx[3, 100:] = -1  # a ragged list
    out = torch.empty((T, 64, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, 64), dtype=torch.float32, device="cuda")
    ws = new_ws(B.ds4x_sparse_attn_decode_workspace(k))
    B.ds4x_sparse_attn_prefill(kv_rows, case["n"], dev(idx), T, k, bf16_dev(case["q_attn"]), SOFTMAX_SCALE, out,
                               lse, ws)
    torch.cuda.synchronize()
    assert B.ds4x_workspace_status(ws) == 0
    got = bf16_host_bits(out)
    got_lse = lse.cpu().numpy()
    packed = C.pack_kv_rows(case["kv_in"])
    for i in range(T):
        ref_out, _, ref_lse = A.sparse_attn_decode(packed, idx[i], case["q_attn"][i], SOFTMAX_SCALE)
        check_attention(got[i], ref_out)
        np.testing.assert_allclose(got_lse[i], ref_lse, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("n_sess,k", [(3, 512), (3, 333), (6, 512)])
def test_batched_attention_equals_single(n_sess, k):
    """One item runs 4 heads per cluster, a batch 8 or 16 (the fewest whose
    grid fits one wave of 2 CTAs per SM, else 16: 3 sessions take 8 and 6
    take 16 on 152 SMs): the per-head arithmetic is the same, so each
    session's output and LSE agree bit for bit."""
    B = require_gpu()
    sess = sessions_case(n_sess=n_sess, scale_lengths=0.02)
    _, kv_rows = _pack_sessions(sess)
    n = torch.tensor([s["n"] for s in sess], dtype=torch.int64, device="cuda")
    rng = np.random.default_rng(11)
    idx = np.full((n_sess, k), -1, dtype=np.int32)  # sessions shorter than k: ragged lists
    for j, s in enumerate(sess):
        m = min(k, s["n"])
        idx[j, :m] = rng.choice(s["n"], size=m, replace=False)
    idx[1, k // 2:] = -1
    q = np.stack([s["q_attn"] for s in sess])
    ws = new_ws(B.ds4x_sparse_attn_decode_workspace(k))
    out_b = torch.empty((n_sess, 64, 512), dtype=torch.bfloat16, device="cuda")
    lse_b = torch.empty((n_sess, 64), dtype=torch.float32, device="cuda")
    B.ds4x_sparse_attn_decode_batched(_ptrs(kv_rows), n, dev(idx), k, bf16_dev(q), SOFTMAX_SCALE, out_b, lse_b, ws)
    for j, s in enumerate(sess):
        out_1 = torch.empty((64, 512), dtype=torch.bfloat16, device="cuda")
        lse_1 = torch.empty(64, dtype=torch.float32, device="cuda")
        B.ds4x_sparse_attn_decode(kv_rows[j], s["n"], dev(idx[j]), k, bf16_dev(s["q_attn"]), SOFTMAX_SCALE, out_1,
                                  lse_1, ws)
        torch.cuda.synchronize()
        assert torch.equal(out_1.view(torch.int16), out_b[j].view(torch.int16)), j
        assert torch.equal(lse_1.view(torch.int32), lse_b[j].view(torch.int32)), j
    assert B.ds4x_workspace_status(ws) == 0
