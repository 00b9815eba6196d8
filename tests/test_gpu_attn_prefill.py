"""ds4x_sparse_attn_prefill (the tensor-core prefill attention) against the
oracle's exact attention, query by query, bf16 vs bf16.

The kernel runs each query's selected rows in tiles of 128, with an online
softmax whose reference maximum moves only when a tile's maximum exceeds it
by more than 8 (log2 units), and one persistent CTA per SM taking several
queries in turn.  The cases reach: k below, at and across tile boundaries;
more queries than SMs (a CTA's later queries reuse its buffers and barrier
phases); -1 padding, a list with no valid row, out-of-range indices; the
rescale of the accumulators (large logits with rows in ascending logit
order, so every tile raises the maximum); blocks whose scales differ by up
to 2^12 over a query's rows (the exact regime) and by up to 2^40 (the
smallest rounded below 2^-24 of their block's largest).
"""

import numpy as np
import pytest
import torch

from gpu_path import bf16_dev, bf16_host_bits, dev, new_ws, pack, require_gpu
from oracle import attention as A
from oracle import codecs as C
from parity import SOFTMAX_SCALE, bf16_ulp, check_attention
from synth import prefill_case, to_bf16_bits

pytestmark = pytest.mark.gpu


def _run(kv_rows, n, idx, q_bits, scale=SOFTMAX_SCALE):
    B = require_gpu()
    T, k = idx.shape
    out = torch.empty((T, 64, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, 64), dtype=torch.float32, device="cuda")
    ws = new_ws(B.ds4x_sparse_attn_decode_workspace(k))
    B.ds4x_sparse_attn_prefill(kv_rows, n, dev(idx.astype(np.int32)), T, k, bf16_dev(q_bits), scale, out, lse, ws)
    torch.cuda.synchronize()
    return bf16_host_bits(out), lse.cpu().numpy(), B.ds4x_workspace_status(ws)


def _check(packed, idx, q_bits, got, got_lse, queries=None, scale=SOFTMAX_SCALE, ulp_floor=False, lse_rtol=1e-5):
    queries = range(idx.shape[0]) if queries is None else queries
    for i in queries:
        ref_out, _, ref_lse = A.sparse_attn_decode(packed, idx[i], q_bits[i], scale)
        check_attention(got[i], ref_out, ulp_floor=ulp_floor)
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(got_lse[i]), fin), i
        np.testing.assert_allclose(got_lse[i][fin], ref_lse[fin], rtol=lse_rtol, atol=1e-5)


@pytest.fixture(scope="module")
def rows():
    require_gpu()
    case = prefill_case(T=400, n=5000, causal_base=4600)
    _, kv_rows = pack(kv_in=case["kv_in"])
    return {"case": case, "kv": kv_rows, "packed": C.pack_kv_rows(case["kv_in"])}


@pytest.mark.parametrize("k", [1, 100, 128, 129, 300, 512])
def test_prefill_attention_ragged_k(rows, k):
    c = rows["case"]
    T = 9
    rng = np.random.default_rng(100 + k)
    idx = np.stack([rng.choice(c["n"], size=k, replace=False) for _ in range(T)])
    got, got_lse, st = _run(rows["kv"], c["n"], idx, c["q_attn"][:T])
    assert st == 0
    _check(rows["packed"], idx, c["q_attn"][:T], got, got_lse)


def test_prefill_attention_more_queries_than_sms(rows):
    """400 queries: every CTA takes two or three in turn."""
    c = rows["case"]
    T, k = 400, 512
    rng = np.random.default_rng(7)
    idx = np.stack([rng.choice(c["causal_base"] + i, size=k, replace=False) for i in range(T)])
    got, got_lse, st = _run(rows["kv"], c["n"], idx, c["q_attn"])
    assert st == 0
    _check(rows["packed"], idx, c["q_attn"], got, got_lse)


def test_prefill_attention_padding_and_bad_indices(rows):
    B = require_gpu()
    c = rows["case"]
    T, k = 5, 300
    rng = np.random.default_rng(9)
    idx = np.stack([rng.choice(c["n"], size=k, replace=False) for _ in range(T)])
    idx[0, 50:] = -1         # ragged list
    idx[1, :] = -1           # no valid row: zeros and -inf
    idx[2, ::3] = -1         # holes in every tile
    idx[3, 130:260] = -1     # a whole tile of padding
    got, got_lse, st = _run(rows["kv"], c["n"], idx, c["q_attn"][:T])
    assert st == 0
    assert np.all(got[1] == 0) and np.all(np.isneginf(got_lse[1]))
    _check(rows["packed"], idx, c["q_attn"][:T], got, got_lse, queries=[0, 2, 3, 4])
    # out-of-range indices are skipped and flagged (the status word reads DS4X_EDEVICE once)
    bad = idx.copy()
    bad[4, 7] = c["n"]
    bad[4, 200] = -5
    got2, got_lse2, st2 = _run(rows["kv"], c["n"], bad, c["q_attn"][:T])
    assert st2 == -7
    skipped = bad.copy()
    skipped[4, 7] = -1
    skipped[4, 200] = -1
    _check(rows["packed"], skipped, c["q_attn"][:T], got2, got_lse2, queries=[0, 4])


def test_prefill_attention_large_logits_rescale(rows):
    """Queries scaled by 40 make the logits spread over hundreds of units;
    each list is ordered by ascending logit of its head 0, so every later
    tile raises that head's maximum by far more than 8 and the accumulators
    are rescaled at every tile."""
    c = rows["case"]
    T, k = 6, 512
    q = (C.bf16_decode(c["q_attn"][:T]).astype(np.float32) * 40.0)
    qb = to_bf16_bits(q)
    v = C.unpack_kv_rows(rows["packed"])
    rng = np.random.default_rng(12)
    idx = np.stack([rng.choice(c["n"], size=k, replace=False) for _ in range(T)])
    for i in range(T):
        lg = v[idx[i]] @ C.bf16_decode(qb[i])[0]
        idx[i] = idx[i][np.argsort(lg, kind="stable")]
    got, got_lse, st = _run(rows["kv"], c["n"], idx, qb)
    assert st == 0
    _check(rows["packed"], idx, qb, got, got_lse, ulp_floor=True)


@pytest.mark.parametrize("spread", [6, 20])
def test_prefill_attention_block_scale_spread(spread):
    """Each non-RoPE block of each row multiplied by its own 2^e, e uniform
    in [-spread, spread] (the FP16 RoPE values keep their range): one block
    of a query's rows holds scales up to 2 spread apart.  At 6 (12 binades)
    every value is exact in the kernel's fp16 operand; at 20 the smallest
    blocks round at 2^-24 of their block's largest, far below the
    tolerance.  The softmax scale shrinks by 2^spread so the logits stay
    O(1) (logits near 10^6 would lose their last units to any fp32
    accumulation)."""
    require_gpu()
    case = prefill_case(T=8, n=3000, causal_base=2900)
    rng = np.random.default_rng(50 + spread)
    e = rng.integers(-spread, spread + 1, size=(case["n"], 7))
    kv_in = case["kv_in"].copy()
    kv_in[:, :448] = (kv_in[:, :448].reshape(-1, 7, 64) * np.ldexp(1.0, e)[:, :, None]).reshape(-1, 448)
    _, kv_rows = pack(kv_in=kv_in)
    packed = C.pack_kv_rows(kv_in)
    T, k = 8, 512
    idx = np.stack([rng.choice(case["n"], size=k, replace=False) for _ in range(T)])
    scale = SOFTMAX_SCALE * 2.0 ** -spread
    got, got_lse, st = _run(kv_rows, case["n"], idx, case["q_attn"], scale=scale)
    assert st == 0
    if spread <= 7:
        _check(packed, idx, case["q_attn"], got, got_lse, scale=scale, ulp_floor=True)
        return
    # beyond 15 binades a block's small values enter the fp16 operand rounded
    # at 2^-24 of the block's largest scale; an output element (a convex
    # combination of the rows' values) is then within the usual bar (2e-3 or
    # one bf16 ulp) plus 2^-24 * 448 * 2^(S_b - 127) of the exact result,
    # S_b the largest scale byte of its block over the query's rows
    for i in range(T):
        ref_out, exact, ref_lse = A.sparse_attn_decode(packed, idx[i], case["q_attn"][i], scale)
        s_b = packed[idx[i], 576:583].astype(np.int64).max(axis=0)
        room = np.concatenate([np.repeat(np.ldexp(448.0, s_b - 127 - 24), 64), np.zeros(64)])
        g = C.bf16_decode(got[i]).astype(np.float64)
        assert np.all(np.abs(g - exact) <= np.maximum(2e-3, bf16_ulp(exact)) + room[None, :]), i
        np.testing.assert_allclose(got_lse[i], ref_lse, rtol=1e-5, atol=1e-5)


def test_prefill_attention_agrees_with_decode_kernel(rows):
    """Each query through the decode attention too: two kernels, two
    precision schemes, both within the bar of the oracle and of each other."""
    B = require_gpu()
    c = rows["case"]
    T, k = 4, 512
    rng = np.random.default_rng(13)
    idx = np.stack([rng.choice(c["n"], size=k, replace=False) for _ in range(T)]).astype(np.int32)
    got, got_lse, _ = _run(rows["kv"], c["n"], idx, c["q_attn"][:T])
    for i in range(T):
        out = torch.empty((64, 512), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(64, dtype=torch.float32, device="cuda")
        ws = new_ws(B.ds4x_sparse_attn_decode_workspace(k))
        B.ds4x_sparse_attn_decode(rows["kv"], c["n"], dev(idx[i]), k, bf16_dev(c["q_attn"][i]), SOFTMAX_SCALE, out,
                                  lse, ws)
        torch.cuda.synchronize()
        d_out = bf16_host_bits(out)
        check_attention(got[i], C.bf16_decode(d_out).astype(np.float64))
        np.testing.assert_allclose(got_lse[i], lse.cpu().numpy(), rtol=1e-5, atol=1e-5)
