"""Packed-row checkpoints on the device path: rows written by the CUDA cache
writer are saved (ds4x_checkpoint_save), loaded back (ds4x_checkpoint_load)
into fresh device buffers, and the score + top-512, the sparse attention,
the sparse + raw-window attention and the dense (HCA) attention over the
reloaded rows are bit-identical to those over the original rows (DS4X
README, "Validation commands": the packed checkpoint round trip; the window
comes back in logical order, oldest first)."""

import numpy as np
import pytest
import torch

from gpu_path import bf16_dev, dev, new_ws, pack, require_gpu
from parity import SOFTMAX_SCALE
from synth import decode_case

pytestmark = pytest.mark.gpu


def _step(B, idx_rows, kv_rows, n, ring, ring_pos, live, hca_rows, n_hca, case):
    k = 512
    ws = new_ws(B.ds4x_index_score_topk_workspace(n, k))
    out_idx = torch.empty(k, dtype=torch.int32, device="cuda")
    out_score = torch.empty(k, dtype=torch.float32, device="cuda")
    B.ds4x_index_score_topk(idx_rows, n, bf16_dev(case["q_idx"]), dev(case["w"]), k, out_idx, out_score, ws)
    qa = bf16_dev(case["q_attn"])
    outs = {"idx": out_idx, "score": out_score}
    ws_a = new_ws(B.ds4x_sparse_attn_decode_workspace(k))
    outs["attn"] = torch.empty((64, 512), dtype=torch.bfloat16, device="cuda")
    outs["lse"] = torch.empty(64, dtype=torch.float32, device="cuda")
    B.ds4x_sparse_attn_decode(kv_rows, n, out_idx, k, qa, SOFTMAX_SCALE, outs["attn"], outs["lse"], ws_a)
    ws_w = new_ws(B.ds4x_window_sparse_attn_decode_workspace())
    outs["win"] = torch.empty((64, 512), dtype=torch.bfloat16, device="cuda")
    outs["win_lse"] = torch.empty(64, dtype=torch.float32, device="cuda")
    B.ds4x_window_sparse_attn_decode(kv_rows, n, out_idx, k, ring, ring_pos, live, qa, SOFTMAX_SCALE, outs["win"],
                                     outs["win_lse"], ws_w)
    ws_d = new_ws(B.ds4x_dense_attn_decode_workspace(n_hca))
    outs["hca"] = torch.empty((64, 512), dtype=torch.bfloat16, device="cuda")
    outs["hca_lse"] = torch.empty(64, dtype=torch.float32, device="cuda")
    B.ds4x_dense_attn_decode(hca_rows, n_hca, qa, SOFTMAX_SCALE, outs["hca"], outs["hca_lse"], ws_d)
    torch.cuda.synchronize()
    for w in (ws, ws_a, ws_w, ws_d):
        assert B.ds4x_workspace_status(w) == 0
    return {key: v.view(torch.int32) if v.dtype == torch.float32 else v.view(torch.int16) for key, v in outs.items()}


def test_checkpoint_round_trip_on_device():
    B = require_gpu()
    n, n_hca, live, ring_pos = 9000, 1300, 200, 57  # the window wraps past ring slot 0
    case = decode_case(n, 4242)
    idx_rows, kv_rows = pack(idx_in=case["idx_in"], kv_in=case["kv_in"])
    ring_src = decode_case(256, 4243)["kv_in"]
    _, ring = pack(kv_in=ring_src)
    _, hca_rows = pack(kv_in=decode_case(n_hca, 4244)["kv_in"])
    before = _step(B, idx_rows, kv_rows, n, ring, ring_pos, live, hca_rows, n_hca, case)

    layers = [
        {"ratio": 4, "ring_live": live, "ring_pos": ring_pos, "ring_rows": ring.cpu().numpy(),
         "kv_rows": kv_rows.cpu().numpy(), "idx_rows": idx_rows.cpu().numpy()},
        {"ratio": 128, "ring_live": 0, "ring_pos": 0, "ring_rows": np.zeros(256 * 583, np.uint8),
         "kv_rows": hca_rows.cpu().numpy(), "idx_rows": None},
    ]
    data = B.ds4x_checkpoint_save(layers)
    bufs = [{"ring_rows": np.zeros(256 * 583, np.uint8), "kv_rows": np.zeros(n * 583, np.uint8),
             "idx_rows": np.zeros(n * 68, np.uint8)},
            {"ring_rows": np.zeros(256 * 583, np.uint8), "kv_rows": np.zeros(n_hca * 583, np.uint8),
             "idx_rows": None}]
    B.ds4x_checkpoint_load(data, bufs)

    # fresh device buffers; the window lands in slots 0..live-1, newest at live-1
    idx2, kv2, ring2, hca2 = (dev(bufs[0]["idx_rows"]), dev(bufs[0]["kv_rows"]), dev(bufs[0]["ring_rows"]),
                              dev(bufs[1]["kv_rows"]))
    assert torch.equal(idx2, idx_rows) and torch.equal(kv2, kv_rows) and torch.equal(hca2, hca_rows)
    after = _step(B, idx2, kv2, n, ring2, live - 1, live, hca2, n_hca, case)
    for key in before:
        assert torch.equal(before[key], after[key]), key
