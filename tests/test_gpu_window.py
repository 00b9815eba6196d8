"""ds4x_window_sparse_attn_decode (the selected compressed rows plus the raw
sliding window, one softmax) against the oracle; with no window it must equal
the sparse attention bit for bit."""

import numpy as np
import pytest
import torch

from gpu_path import bf16_dev, bf16_host_bits, dev, new_ws, pack, require_gpu
from oracle import codecs as C
from oracle.attention import window_sparse_attn_decode
from parity import SOFTMAX_SCALE, check_attention
from synth import decode_case

pytestmark = pytest.mark.gpu


def _case(seed, n=5000):
    a = decode_case(n, seed)
    b = decode_case(256, seed + 100)
    _, kv_rows = pack(kv_in=a["kv_in"])
    _, ring_rows = pack(kv_in=b["kv_in"])
    return a, b, kv_rows, ring_rows


def _window(B, kv_rows, n, idx, ring_rows, pos, w, q_bits):
    out = torch.empty((64, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(64, dtype=torch.float32, device="cuda")
    ws = new_ws(B.ds4x_window_sparse_attn_decode_workspace())
    B.ds4x_window_sparse_attn_decode(kv_rows, n, dev(idx), len(idx), ring_rows, pos, w, bf16_dev(q_bits),
                                     SOFTMAX_SCALE, out, lse, ws)
    torch.cuda.synchronize()
    assert B.ds4x_workspace_status(ws) == 0
    return out, lse


@pytest.mark.parametrize("k,pos,w,ragged", [(512, 200, 128, False), (512, 3, 10, False), (512, 255, 256, True),
                                            (100, 0, 1, False), (1, 77, 200, True)])
def test_window_sparse_parity(k, pos, w, ragged):
    B = require_gpu()
    a, b, kv_rows, ring_rows = _case(6000 + k + w)
    n = a["kv_in"].shape[0]
    rng = np.random.default_rng(k + w)
    idx = rng.choice(n, size=k, replace=False).astype(np.int32)
    if ragged:
        idx[k // 2:] = -1
    out, lse = _window(B, kv_rows, n, idx, ring_rows, pos, w, a["q_attn"])
    ref_out, _, ref_lse = window_sparse_attn_decode(C.pack_kv_rows(a["kv_in"]), idx, C.pack_kv_rows(b["kv_in"]), pos,
                                                    w, a["q_attn"], SOFTMAX_SCALE)
    check_attention(bf16_host_bits(out), ref_out)
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-5)


def test_no_window_equals_the_sparse_attention():
    """The empty window item has weight e^-inf = 0 in the finalize."""
    B = require_gpu()
    a, _, kv_rows, ring_rows = _case(6100)
    n = a["kv_in"].shape[0]
    idx = np.random.default_rng(3).choice(n, size=512, replace=False).astype(np.int32)
    out_w, lse_w = _window(B, kv_rows, n, idx, ring_rows, 9, 0, a["q_attn"])
    out_s = torch.empty((64, 512), dtype=torch.bfloat16, device="cuda")
    lse_s = torch.empty(64, dtype=torch.float32, device="cuda")
    ws = new_ws(B.ds4x_sparse_attn_decode_workspace(512))
    B.ds4x_sparse_attn_decode(kv_rows, n, dev(idx), 512, bf16_dev(a["q_attn"]), SOFTMAX_SCALE, out_s, lse_s, ws)
    torch.cuda.synchronize()
    assert torch.equal(out_w.view(torch.int16), out_s.view(torch.int16))
    assert torch.equal(lse_w.view(torch.int32), lse_s.view(torch.int32))
