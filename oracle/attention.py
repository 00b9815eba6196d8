"""Sparse (indexed) decode attention over packed KV rows -- float64 oracle.

Test infrastructure only (see ``oracle/__init__``).

For each attention head h < 64 with bf16 query q_h (dimension 512) and the
selected rows j (indices from the top-k; -1 entries are padding and skipped):

    v_j   = dequantised 583-byte row: 448 E4M3 * 2**(scale - 127), then the
            64 FP16 RoPE values (DS4X README, "Packed cache ABI")
    l_hj  = scale * (q_h . v_j)                  (scale = 1/sqrt(512))
    p_hj  = exp(l_hj - max_j l_hj) / sum_j exp(l_hj - max_j l_hj)
    o_h   = sum_j p_hj v_j                       -> rounded to bf16 (RNE)
    lse_h = max_j l_hj + log(sum_j exp(l_hj - max_j l_hj))

Keys and values are the same vector (shared KV across all heads); no mask,
no sink.  The output is rounded to bf16 because the path's output is bf16:
parity compares bf16 with bf16.
"""

from __future__ import annotations

import numpy as np

from .codecs import bf16_decode, bf16_round, unpack_kv_rows


def sparse_attn_decode(kv_rows, idx, q_bf16, scale: float):
    """Returns (out float64 [H, 512] bf16-rounded, out_exact float64 [H, 512],
    lse float64 [H]).

    kv_rows : uint8 [n, 583]
    idx     : int [k] selected row indices (-1 = skip)
    q_bf16  : uint16 [H, 512] bfloat16 bit patterns
    """
    idx = np.asarray(idx, dtype=np.int64)
    sel = idx[idx >= 0]
    q = bf16_decode(q_bf16)  # [H, 512]
    heads = q.shape[0]
    if sel.size == 0:
        zero = np.zeros((heads, q.shape[1]))
        return zero, zero, np.full(heads, -np.inf)
    v = unpack_kv_rows(np.asarray(kv_rows)[sel])  # [m, 512]
    logits = (q @ v.T) * float(scale)  # [H, m]
    mx = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - mx)
    denom = e.sum(axis=1, keepdims=True)
    out = (e / denom) @ v
    lse = mx[:, 0] + np.log(denom[:, 0])
    return bf16_round(out), out, lse
