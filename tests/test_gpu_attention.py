"""ds4x_sparse_attn_decode vs the oracle's exact attention (bf16 vs bf16)."""

import numpy as np
import pytest

from gpu_path import attention, pack, require_gpu
from oracle import codecs as C
from oracle import indexer as I
from oracle.attention import sparse_attn_decode
from parity import SOFTMAX_SCALE, check_attention
from synth import decode_case, to_bf16_bits

pytestmark = pytest.mark.gpu


def _run(case, idx, n=None):
    n = n or case["n"]
    _, kv_rows = pack(kv_in=case["kv_in"])
    g_out, g_lse, ws = attention(kv_rows, n, idx, case["q_attn"], SOFTMAX_SCALE)
    rows = C.pack_kv_rows(case["kv_in"])
    o_out, _, o_lse = sparse_attn_decode(rows, idx, case["q_attn"], SOFTMAX_SCALE)
    return g_out, g_lse, o_out, o_lse, ws


def test_attention_on_oracle_topk_tiny_decode():
    require_gpu()
    case = decode_case(4096, 1000)
    rows = C.pack_idx_rows(case["idx_in"])
    idx, _, _ = I.score_topk(rows, case["q_idx"], case["w"], 512)
    g_out, g_lse, o_out, o_lse, _ = _run(case, idx)
    check_attention(g_out, o_out)
    np.testing.assert_allclose(g_lse, o_lse, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("k", [1, 2, 31, 33, 100, 511, 512])
def test_attention_ragged_k(k):
    require_gpu()
    case = decode_case(3000, 30 + k)
    idx = np.random.default_rng(k).choice(3000, size=k, replace=False)
    g_out, g_lse, o_out, o_lse, _ = _run(case, idx)
    check_attention(g_out, o_out)
    np.testing.assert_allclose(g_lse, o_lse, rtol=1e-5, atol=1e-5)


def test_attention_single_row_is_the_row():
    require_gpu()
    case = decode_case(100, 41)
    g_out, _, o_out, _, _ = _run(case, [42])
    v = C.unpack_kv_rows(C.pack_kv_rows(case["kv_in"][42:43]))[0]
    expect = np.tile(C.bf16_encode(v), (64, 1))
    assert np.array_equal(g_out, expect)


def test_attention_padding_and_bad_indices():
    B = require_gpu()
    case = decode_case(500, 42)
    idx = np.full(64, -1, dtype=np.int64)
    idx[[3, 10, 40]] = [7, 499, 0]
    g_out, g_lse, o_out, o_lse, ws = _run(case, idx)
    check_attention(g_out, o_out)
    assert B.ds4x_workspace_status(ws) == 0
    # all rows skipped: zero output, -inf lse
    g2, l2, _ = attention(pack(kv_in=case["kv_in"])[1], 500, np.full(40, -1), case["q_attn"], SOFTMAX_SCALE)
    assert np.all(g2 == 0) and np.all(np.isneginf(l2))
    # out-of-range indices are skipped and flagged
    bad = idx.copy()
    bad[5] = 500
    bad[6] = -7
    g3, _, ws3 = attention(pack(kv_in=case["kv_in"])[1], 500, bad, case["q_attn"], SOFTMAX_SCALE)
    check_attention(g3, o_out)
    assert B.ds4x_workspace_status(ws3) == -7
    assert B.ds4x_workspace_status(ws3) == 0  # reading clears it


def test_attention_large_logits():
    """Scaled-up queries make the softmax nearly one-hot; the max-subtraction
    must keep it finite."""
    require_gpu()
    case = decode_case(2000, 43)
    q = C.bf16_decode(case["q_attn"]).astype(np.float32) * 40.0
    case["q_attn"] = to_bf16_bits(q)
    idx = np.arange(0, 2000, 4)[:512]
    g_out, g_lse, o_out, o_lse, _ = _run(case, idx)
    # outputs approach raw row values (|o| up to ~3.5): one bf16 ulp is 1.6e-2
    check_attention(g_out, o_out, ulp_floor=True)
    np.testing.assert_allclose(g_lse, o_lse, rtol=1e-5)
