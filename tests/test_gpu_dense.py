"""ds4x_dense_attn_decode (the HCA layers' attention over every compressed
row) against the oracle's dense attention.

The rows are cut into items of R consecutive rows (R = 128 up to 32,768 rows,
then 256, 384, 512), each run by the tensor-core attention kernel with the
one query, then a log-sum-exp combine over the items.  The cases reach: item
edges (127, 128, 129 rows); the 8192 rows of a 1M-token ratio-128 layer (64
items, one wave); more items than SMs (a CTA's later items reuse its buffers
and barrier phases) with 128-, 256- and 512-row items; rows past n_rows left
alone; blocks whose scales differ by up to 2^12 over an item's rows (the exact
regime) and by up to 2^40 (the smallest rounded below 2^-24 of their block's
largest); and one item equal to the prefill attention over the same rows bit
for bit.
"""

import numpy as np
import pytest
import torch

from gpu_path import bf16_dev, bf16_host_bits, dev, new_ws, pack, require_gpu
from oracle import codecs as C
from oracle.attention import dense_attn_decode
from parity import SOFTMAX_SCALE, bf16_ulp, check_attention
from synth import decode_case

pytestmark = pytest.mark.gpu


def _rows_per_item(n):
    return 128 * min(4, max(1, -(-n // 32768)))


def _dense(B, kv_rows, n, q_bits, scale=SOFTMAX_SCALE):
    out = torch.empty((64, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(64, dtype=torch.float32, device="cuda")
    ws = new_ws(B.ds4x_dense_attn_decode_workspace(n))
    B.ds4x_dense_attn_decode(kv_rows, n, bf16_dev(q_bits), scale, out, lse, ws)
    torch.cuda.synchronize()
    assert B.ds4x_workspace_status(ws) == 0
    return out, lse


@pytest.mark.parametrize("n", [1, 2, 127, 128, 129, 1500, 8192, 32768, 32769, 100000])
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


@pytest.mark.parametrize("spread", [6, 20])
def test_dense_attention_block_scale_spread(spread):
    """Each non-RoPE block of each row multiplied by its own 2^e, e uniform in
    [-spread, spread]: one block of an item's rows holds scales up to
    2 spread apart.  At 6 every value is exact in the kernel's fp16 operand;
    at 20 the smallest blocks round at 2^-24 of their block's largest scale
    over the item's rows.  The softmax scale shrinks by 2^spread so the
    logits stay O(1)."""
    B = require_gpu()
    n = 1000  # 8 items of 128 rows, the last ragged
    case = decode_case(n, 5300 + spread)
    rng = np.random.default_rng(60 + spread)
    e = rng.integers(-spread, spread + 1, size=(n, 7))
    kv_in = case["kv_in"].copy()
    kv_in[:, :448] = (kv_in[:, :448].reshape(-1, 7, 64) * np.ldexp(1.0, e)[:, :, None]).reshape(-1, 448)
    _, kv_rows = pack(kv_in=kv_in)
    packed = C.pack_kv_rows(kv_in)
    scale = SOFTMAX_SCALE * 2.0 ** -spread
    out, lse = _dense(B, kv_rows, n, case["q_attn"], scale=scale)
    ref_out, exact, ref_lse = dense_attn_decode(packed, n, case["q_attn"], scale)
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=1e-5, atol=1e-5)
    if spread <= 7:
        check_attention(bf16_host_bits(out), ref_out, ulp_floor=True)
        return
    # an output element is a convex combination of the items' normalised
    # outputs, each within 2^-24 * 448 * 2^(S_b - 127) of exact (S_b the largest
    # scale byte of its block over that item's rows): so within the largest
    # such room over the items, plus the usual bar
    R = _rows_per_item(n)
    s_b = np.stack([packed[i:i + R, 576:583].astype(np.int64).max(axis=0) for i in range(0, n, R)]).max(axis=0)
    room = np.concatenate([np.repeat(np.ldexp(448.0, s_b - 127 - 24), 64), np.zeros(64)])
    g = C.bf16_decode(bf16_host_bits(out)).astype(np.float64)
    assert np.all(np.abs(g - exact) <= np.maximum(2e-3, bf16_ulp(exact)) + room[None, :])


@pytest.mark.parametrize("n", [7, 128])
def test_one_item_equals_prefill_attention_over_every_row(n):
    """With one item the combine multiplies by e^0 = 1 and divides by 1, so
    the result is the prefill attention's over rows 0 .. n - 1, bit for bit."""
    B = require_gpu()
    case = decode_case(n, 5200 + n)
    _, kv_rows = pack(kv_in=case["kv_in"])
    out_d, lse_d = _dense(B, kv_rows, n, case["q_attn"])
    out_p = torch.empty((1, 64, 512), dtype=torch.bfloat16, device="cuda")
    lse_p = torch.empty((1, 64), dtype=torch.float32, device="cuda")
    ws = new_ws(B.ds4x_sparse_attn_decode_workspace(n))
    B.ds4x_sparse_attn_prefill(kv_rows, n, dev(np.arange(n, dtype=np.int32)[None, :]), 1, n,
                               bf16_dev(case["q_attn"][None]), SOFTMAX_SCALE, out_p, lse_p, ws)
    torch.cuda.synchronize()
    assert B.ds4x_workspace_status(ws) == 0
    assert torch.equal(out_d.view(torch.int16), out_p[0].view(torch.int16))
    assert torch.equal(lse_d.view(torch.int32), lse_p[0].view(torch.int32))
