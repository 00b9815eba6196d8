"""ds4x_dense_attn_decode (the HCA layers' attention over every compressed
row) against the oracle's dense attention, over tile edges (512-row tiles)
and the 8192 rows of a 1M-token ratio-128 layer; one tile must equal the
sparse attention over every row bit for bit."""

import numpy as np
import pytest
import torch

from gpu_path import bf16_dev, bf16_host_bits, dev, new_ws, pack, require_gpu
from oracle import codecs as C
from oracle.attention import dense_attn_decode
from parity import SOFTMAX_SCALE, check_attention
from synth import decode_case

pytestmark = pytest.mark.gpu


def _dense(B, kv_rows, n, q_bits):
    out = torch.empty((64, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(64, dtype=torch.float32, device="cuda")
    ws = new_ws(B.ds4x_dense_attn_decode_workspace(n))
    B.ds4x_dense_attn_decode(kv_rows, n, bf16_dev(q_bits), SOFTMAX_SCALE, out, lse, ws)
    torch.cuda.synchronize()
    assert B.ds4x_workspace_status(ws) == 0
    return out, lse


@pytest.mark.parametrize("n", [1, 2, 511, 512, 513, 1500, 8192])
def test_dense_attention_parity(n):
    B = require_gpu()
    case = decode_case(n, 5000 + n)
    _, kv_rows = pack(kv_in=case["kv_in"])
    out, lse = _dense(B, kv_rows, n, case["q_attn"])
    ref_out, _, ref_lse = dense_attn_decode(C.pack_kv_rows(case["kv_in"]), n, case["q_attn"], SOFTMAX_SCALE)
    check_attention(bf16_host_bits(out), ref_out)
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-5)


def test_dense_attention_reads_only_its_rows():
    """Rows past n_rows (here garbage-free but different) do not change the result."""
    B = require_gpu()
    case = decode_case(3000, 5101)
    _, kv_rows = pack(kv_in=case["kv_in"])
    out, lse = _dense(B, kv_rows, 1234, case["q_attn"])
    ref_out, _, ref_lse = dense_attn_decode(C.pack_kv_rows(case["kv_in"]), 1234, case["q_attn"], SOFTMAX_SCALE)
    check_attention(bf16_host_bits(out), ref_out)
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("n", [7, 512])
def test_one_tile_equals_sparse_over_every_row(n):
    """With one tile the finalize multiplies by e^0 = 1 and divides by 1."""
    B = require_gpu()
    case = decode_case(n, 5200 + n)
    _, kv_rows = pack(kv_in=case["kv_in"])
    out_d, lse_d = _dense(B, kv_rows, n, case["q_attn"])
    out_s = torch.empty((64, 512), dtype=torch.bfloat16, device="cuda")
    lse_s = torch.empty(64, dtype=torch.float32, device="cuda")
    ws = new_ws(B.ds4x_sparse_attn_decode_workspace(n))
    B.ds4x_sparse_attn_decode(kv_rows, n, dev(np.arange(n, dtype=np.int32)), n, bf16_dev(case["q_attn"]),
                              SOFTMAX_SCALE, out_s, lse_s, ws)
    torch.cuda.synchronize()
    assert torch.equal(out_d.view(torch.int16), out_s.view(torch.int16))
    assert torch.equal(lse_d.view(torch.int32), lse_s.view(torch.int32))
