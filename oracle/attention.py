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


def dense_attn_decode(kv_rows, n: int, q_bf16, scale: float):
    """Dense decode attention over every row [0, n) -- the HCA layers' exact
    attention over all their compressed rows (DS4X README, "Optimization
    details", the HCA bullet: exact score-split attention with no row
    ceiling).  Same definition as the sparse attention with every row
    selected; written out on its own.  Returns (out bf16-rounded, out_exact,
    lse), float64, shapes [H, 512], [H, 512], [H]; n = 0 gives zeros and -inf.
    """
    q = bf16_decode(q_bf16)
    heads, dim = q.shape
    if n <= 0:
        zero = np.zeros((heads, dim))
        return zero, zero, np.full(heads, -np.inf)
    v = unpack_kv_rows(np.asarray(kv_rows)[:n])  # [n, 512]
    logits = float(scale) * (q @ v.T)  # [H, n]
    m = logits.max(axis=1)
    w = np.exp(logits - m[:, None])
    s = w.sum(axis=1)
    out = (w @ v) / s[:, None]
    return bf16_round(out), out, m + np.log(s)


def lse_combine(parts):
    """The split-KV log-sum-exp combine of split-KV flash decoding (DS4X
    README, "Nsight Systems": the score-split finalize kernel group):
    parts is a list of (o_s [H, D] normalised within split s, lse_s [H]); an
    empty split has lse -inf.  Returns (o, lse) with
        M = max_s lse_s,  o = sum_s e^(lse_s - M) o_s / sum_s e^(lse_s - M),
        lse = M + log sum_s e^(lse_s - M).
    """
    lse = np.stack([np.asarray(p[1], dtype=np.float64) for p in parts])  # [S, H]
    o = np.stack([np.asarray(p[0], dtype=np.float64) for p in parts])  # [S, H, D]
    m = lse.max(axis=0)  # [H]
    safe_m = np.where(np.isfinite(m), m, 0.0)
    f = np.where(np.isfinite(lse), np.exp(lse - safe_m[None, :]), 0.0)  # [S, H]
    tot = f.sum(axis=0)
    out = np.where(tot[:, None] > 0, (f[:, :, None] * o).sum(axis=0) / np.where(tot > 0, tot, 1.0)[:, None], 0.0)
    return out, np.where(tot > 0, safe_m + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)


def window_sparse_attn_decode(kv_rows, idx, ring_rows, ring_pos, w: int, q_bf16, scale: float):
    """Decode attention over the selected compressed rows AND the raw
    sliding window: each layer keeps a raw KV ring of packed 583-byte rows,
    padded to 256 rows (DS4X README, "Packed cache ABI"), whose live rows are
    the most recent tokens; a checkpoint stores them in logical position
    order rather than physical ring order (ds4 README, "Disk KV Cache").
    Reading: one softmax over the union of the two row sets (equivalently
    the log-sum-exp merge of the sparse and the window attention).

    kv_rows   : uint8 [n, 583] compressed rows; idx: int [k] (-1 = skip)
    ring_rows : uint8 [R, 583] the ring in physical order
    ring_pos  : physical slot of the newest window row; the window is the w
                slots ring_pos, ring_pos - 1, ... (mod R), 0 <= w <= R
    Returns (out bf16-rounded, out_exact, lse) as sparse_attn_decode.
    """
    idx = np.asarray(idx, dtype=np.int64)
    sel = np.asarray(kv_rows)[idx[idx >= 0]]
    ring = np.asarray(ring_rows)
    slots = (int(ring_pos) - np.arange(int(w))) % ring.shape[0] if w > 0 else np.zeros(0, dtype=np.int64)
    rows = np.concatenate([sel, ring[slots]], axis=0) if (sel.shape[0] + slots.size) > 0 else sel
    q = bf16_decode(q_bf16)
    heads, dim = q.shape
    if rows.shape[0] == 0:
        zero = np.zeros((heads, dim))
        return zero, zero, np.full(heads, -np.inf)
    v = unpack_kv_rows(rows)
    logits = float(scale) * (q @ v.T)
    m = logits.max(axis=1)
    e = np.exp(logits - m[:, None])
    s = e.sum(axis=1)
    out = (e @ v) / s[:, None]
    return bf16_round(out), out, m + np.log(s)
