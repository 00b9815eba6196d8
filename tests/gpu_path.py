"""Helpers that drive the CUDA path through the C ABI (via the ctypes
binding) on numpy inputs from ``synth``; used by the ``-m gpu`` tests."""

import numpy as np
import pytest
import torch


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compressed_kv_sparse_csa_gb300 import binding

    binding.lib()  # raises loudly if the library is missing
    return binding


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def bf16_host_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def new_ws(nbytes):
    B = require_gpu()
    ws = torch.empty(int(nbytes), dtype=torch.uint8, device="cuda")
    B.ds4x_workspace_init(ws)
    return ws


def pack(idx_in=None, kv_in=None, capacity=None, chunks=1):
    """Append rows with ds4x_cache_append (in `chunks` calls); returns the
    device row arrays (None where not requested)."""
    B = require_gpu()
    n = (idx_in if idx_in is not None else kv_in).shape[0]
    cap = capacity or n
    idx_rows = torch.zeros(cap * 68, dtype=torch.uint8, device="cuda") if idx_in is not None else None
    kv_rows = torch.zeros(cap * 583, dtype=torch.uint8, device="cuda") if kv_in is not None else None
    bounds = np.linspace(0, n, chunks + 1).astype(int)
    d_idx = dev(idx_in) if idx_in is not None else None
    d_kv = dev(kv_in) if kv_in is not None else None
    for a, b in zip(bounds[:-1], bounds[1:]):
        if b <= a:
            continue
        B.ds4x_cache_append(kv_rows, idx_rows, int(a),
                            d_kv[a:b] if d_kv is not None else None,
                            d_idx[a:b] if d_idx is not None else None)
    return idx_rows, kv_rows


def score_topk(idx_rows, n, q_bits, w, k=512, return_ws=False):
    B = require_gpu()
    ws = new_ws(B.ds4x_index_score_topk_workspace(n, k))
    out_idx = torch.empty(k, dtype=torch.int32, device="cuda")
    out_score = torch.empty(k, dtype=torch.float32, device="cuda")
    B.ds4x_index_score_topk(idx_rows, n, bf16_dev(q_bits), dev(w), k, out_idx, out_score, ws)
    torch.cuda.synchronize()
    if return_ws:
        return out_idx.cpu().numpy(), out_score.cpu().numpy(), ws
    return out_idx.cpu().numpy(), out_score.cpu().numpy()


def fallback_merges(ws):
    """Scorer calls on this workspace that took the exact fallback merge
    (the u32 at bytes 8..11 of the workspace header)."""
    return int(ws[8:12].view(torch.int32).item())


def attention(kv_rows, n, idx, q_bits, scale, ws=None):
    B = require_gpu()
    idx = np.asarray(idx, dtype=np.int32)
    k = idx.shape[0]
    if ws is None:
        ws = new_ws(B.ds4x_sparse_attn_decode_workspace(k))
    out = torch.empty((64, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(64, dtype=torch.float32, device="cuda")
    B.ds4x_sparse_attn_decode(kv_rows, n, dev(idx), k, bf16_dev(q_bits), scale, out, lse, ws)
    torch.cuda.synchronize()
    return bf16_host_bits(out), lse.cpu().numpy(), ws
