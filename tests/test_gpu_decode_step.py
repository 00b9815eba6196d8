"""ds4x_csa_decode_step (score + top-k, then attention over the selected
rows, in one call) gives exactly the results of ds4x_index_score_topk
followed by ds4x_sparse_attn_decode, and matches the oracle."""

import numpy as np
import pytest
import torch

from gpu_path import bf16_dev, bf16_host_bits, dev, new_ws, pack, require_gpu
from oracle import attention as A
from oracle import codecs as C
from oracle import indexer as I
from parity import SOFTMAX_SCALE, check_attention, check_topk
from synth import decode_case

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,k", [(4096, 512), (70000, 512), (3000, 100), (300, 512)])
def test_decode_step_equals_the_two_calls(n, k):
    B = require_gpu()
    case = decode_case(n, 5000 + n)
    idx_rows, kv_rows = pack(idx_in=case["idx_in"], kv_in=case["kv_in"])
    q, w, qa = bf16_dev(case["q_idx"]), dev(case["w"]), bf16_dev(case["q_attn"])

    def outs():
        return (torch.empty(k, dtype=torch.int32, device="cuda"), torch.empty(k, dtype=torch.float32, device="cuda"),
                torch.empty((64, 512), dtype=torch.bfloat16, device="cuda"), torch.empty(64, dtype=torch.float32, device="cuda"))

    i1, s1, o1, l1 = outs()
    ws_s = new_ws(B.ds4x_index_score_topk_workspace(n, k))
    ws_a = new_ws(B.ds4x_sparse_attn_decode_workspace(k))
    B.ds4x_index_score_topk(idx_rows, n, q, w, k, i1, s1, ws_s)
    B.ds4x_sparse_attn_decode(kv_rows, n, i1, k, qa, SOFTMAX_SCALE, o1, l1, ws_a)
    i2, s2, o2, l2 = outs()
    ws = new_ws(B.ds4x_csa_decode_step_workspace(n, k))
    for _ in range(2):  # the workspace is ready for the next step
        B.ds4x_csa_decode_step(idx_rows, kv_rows, n, q, w, k, qa, SOFTMAX_SCALE, i2, s2, o2, l2, ws)
        torch.cuda.synchronize()
        assert B.ds4x_workspace_status(ws) == 0
        assert torch.equal(i1, i2) and torch.equal(s1.view(torch.int32), s2.view(torch.int32))
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1.view(torch.int32), l2.view(torch.int32))
    gi, gs = i2.cpu().numpy(), s2.cpu().numpy()
    check_topk(gi, gs, I.score_rows(C.pack_idx_rows(case["idx_in"]), case["q_idx"], case["w"]), k)
    sel = gi[gi >= 0]
    ref_out, _, _ = A.sparse_attn_decode(C.pack_kv_rows(case["kv_in"][sel]), np.arange(sel.size), case["q_attn"],
                                         SOFTMAX_SCALE)
    check_attention(bf16_host_bits(o2), ref_out)
