"""The allocation-free attention entry point (for callers that cannot
allocate device memory at decode time) must give the same output as
ds4x_sparse_attn_decode with a caller-provided workspace, call after call,
although all its calls share one static scratch array inside the library.

Collected last on purpose (file name), so that a run stopping at its first
failure has already run every other test; it also passes alone in a fresh
process."""

import math

import numpy as np
import pytest

from gpu_path import attention, bf16_dev, bf16_host_bits, dev, pack, require_gpu
from parity import SOFTMAX_SCALE, check_attention
from synth import decode_case

pytestmark = pytest.mark.gpu


def _noalloc(kv_rows, n, idx, q_bits):
    import torch

    B = require_gpu()
    idx = np.asarray(idx, dtype=np.int32)
    out = torch.empty((64, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(64, dtype=torch.float32, device="cuda")
    B.ds4x_sparse_attn_decode_noalloc(kv_rows, n, dev(idx), idx.shape[0], bf16_dev(q_bits), SOFTMAX_SCALE, out, lse)
    torch.cuda.synchronize()
    return bf16_host_bits(out), lse.cpu().numpy()


def test_noalloc_matches_workspace_entry_two_calls_in_a_row():
    require_gpu()
    case_a = decode_case(4096, 1000)
    case_b = decode_case(2500, 77)
    _, kv_a = pack(kv_in=case_a["kv_in"])
    _, kv_b = pack(kv_in=case_b["kv_in"])
    rng = np.random.default_rng(5)
    idx_a = rng.choice(4096, size=512, replace=False)  # all 16 splits
    idx_b = rng.choice(2500, size=97, replace=False)   # a different split count after it
    for kv, n, idx, q in ((kv_a, 4096, idx_a, case_a["q_attn"]), (kv_b, 2500, idx_b, case_b["q_attn"])):
        ref_out, ref_lse, _ = attention(kv, n, idx, q, SOFTMAX_SCALE)
        got_out, got_lse = _noalloc(kv, n, idx, q)
        ref_f = (ref_out.astype(np.uint32) << 16).view(np.float32)
        check_attention(got_out, ref_f)
        np.testing.assert_allclose(got_lse, ref_lse, rtol=1e-6, atol=1e-6)


def test_noalloc_rejects_k_above_512():
    import torch

    B = require_gpu()
    case = decode_case(600, 78)
    _, kv = pack(kv_in=case["kv_in"])
    out = torch.empty((64, 512), dtype=torch.bfloat16, device="cuda")
    idx = dev(np.arange(513, dtype=np.int32))
    with pytest.raises(B.Ds4xError) as ei:
        B.ds4x_sparse_attn_decode_noalloc(kv, 600, idx, 513, bf16_dev(case["q_attn"]), 1 / math.sqrt(512), out, None)
    assert ei.value.status == -1
