"""Chunked-prefill (multi-query) CSA scorer and attention -- float64 oracle.

Test infrastructure only (see ``oracle/__init__``).

DS4X README, "Packed prefill implementation": batch score/top-k and
multi-token attention stay active during packed prefill over the same
68-byte indexer and 583-byte KV rows.  For a chunk of T query tokens:

* each query vector (per head, dimension 128) is quantised to E4M3 with one
  UE8M0 scale per 32 values (scale rule as for the KV rows: least e with
  amax <= 448 * 2**e), and scored from its dequantised value q^;
* query i sees only rows t < causal_base + i;
* s_it = sum_h w_ih * max(0, q^_ih . k_t) over the visible rows;
* per query: exact top-k (score descending, lower index first), then the
  decode attention of that query's bf16 attention vector over its rows.
"""

from __future__ import annotations

import numpy as np

from .attention import sparse_attn_decode
from .codecs import E4M3_MAX, e4m3_decode, e4m3_encode, quantize_blocks, ue8m0_decode, unpack_idx_rows
from .indexer import topk

Q_BLOCK = 32


def quantize_query_e4m3(q):
    """f32 [..., 128] -> (codes uint8 [..., 128], scales uint8 [..., 4])."""
    return quantize_blocks(q, Q_BLOCK, E4M3_MAX, e4m3_encode)


def dequantize_query_e4m3(codes, scales):
    codes = np.asarray(codes)
    lead = codes.shape[:-1]
    d = codes.shape[-1]
    v = e4m3_decode(codes).reshape(*lead, d // Q_BLOCK, Q_BLOCK)
    return (v * ue8m0_decode(scales)[..., None]).reshape(*lead, d)


def prefill_scores(idx_rows, q_codes, q_scales, w, causal_base: int, queries=None):
    """Scores float64 [len(queries), n]; invisible rows are -inf.

    q_codes [T, H, 128], q_scales [T, H, 4], w float32 [T, H]."""
    n = idx_rows.shape[0]
    T = q_codes.shape[0]
    queries = np.arange(T) if queries is None else np.asarray(queries)
    k = unpack_idx_rows(idx_rows)  # [n, 128]
    out = np.full((len(queries), n), -np.inf)
    for r, i in enumerate(queries):
        vis = min(n, causal_base + int(i))
        if vis <= 0:
            continue
        qh = dequantize_query_e4m3(q_codes[i], q_scales[i])  # [H, 128]
        wi = np.asarray(w[i], dtype=np.float32).astype(np.float64)
        out[r, :vis] = np.maximum(k[:vis] @ qh.T, 0.0) @ wi
    return out


def prefill_topk(idx_rows, q_codes, q_scales, w, causal_base: int, k: int = 512, queries=None):
    """Per-query exact top-k over the visible rows: (idx [Q, k], val [Q, k], scores [Q, n])."""
    s = prefill_scores(idx_rows, q_codes, q_scales, w, causal_base, queries)
    idx = np.full((s.shape[0], k), -1, dtype=np.int64)
    val = np.full((s.shape[0], k), np.nan)
    for r in range(s.shape[0]):
        vis = int(np.sum(np.isfinite(s[r])))
        i_r, v_r = topk(s[r, :vis], k)
        idx[r], val[r] = i_r, v_r
    return idx, val, s


def prefill_attention(kv_rows, idx, q_bf16, scale: float, queries=None):
    """Per-query decode attention: out float64 [Q, H, 512] (bf16-rounded).

    idx [T, k], q_bf16 uint16 [T, H, 512]."""
    T = idx.shape[0]
    queries = np.arange(T) if queries is None else np.asarray(queries)
    outs = []
    for i in queries:
        o, _, _ = sparse_attn_decode(kv_rows, idx[i], q_bf16[i], scale)
        outs.append(o)
    return np.stack(outs)
