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
    ws = new_ws(B.ds4x_index_score_topk_prefill_workspace(T, k))
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
