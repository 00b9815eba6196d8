"""The scorer's bounded waits: when its CTA exchange can never complete,
every CTA gives up after its time limit (0.5 s of the GPU's global timer),
frees its tensor memory and returns; the workspace status word reads
DS4X_ETIMEOUT and the context stays usable.  The wait is made to run out
without any fault: the workspace header's extra-arrivals word is set to 1,
so the arrival count the CTAs wait for is one more than there are CTAs."""

import time

import numpy as np
import pytest
import torch

from gpu_path import bf16_dev, dev, new_ws, pack, require_gpu, score_topk
from oracle import codecs as C
from oracle import indexer as I
from parity import check_topk
from synth import decode_case

pytestmark = pytest.mark.gpu

ETIMEOUT = -6


def test_exchange_wait_times_out_and_recovers():
    B = require_gpu()
    n, k = 40000, 512  # more tiles than SMs: every CTA takes part in the exchange
    case = decode_case(n, 606)
    rows, _ = pack(idx_in=case["idx_in"])
    ws = new_ws(B.ds4x_index_score_topk_workspace(n, k))
    ws[12:16].view(torch.int32).fill_(1)  # one arrival that never comes
    out_idx = torch.full((k,), -7, dtype=torch.int32, device="cuda")
    q, w = bf16_dev(case["q_idx"]), dev(case["w"])
    t0 = time.time()
    B.ds4x_index_score_topk(rows, n, q, w, k, out_idx, None, ws)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert B.ds4x_workspace_status(ws) == ETIMEOUT
    assert 0.3 < elapsed < 30.0, elapsed
    assert np.all(out_idx.cpu().numpy() == -7)  # no winner is written after a time-out
    # the context is still usable and a fresh workspace gives the exact result
    gi, gs = score_topk(rows, n, case["q_idx"], case["w"], k)
    check_topk(gi, gs, I.score_rows(C.pack_idx_rows(case["idx_in"]), case["q_idx"], case["w"]), k)
