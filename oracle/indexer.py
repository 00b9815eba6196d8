"""CSA indexer score and exact top-k -- float64 oracle.

Test infrastructure only (see ``oracle/__init__``).

Score of compressed row t for one decode query (indexer heads h < H = 64,
dimension 128):

    s_t = sum_h w_h * max(0, sum_j q_hj * k_tj)

with k_t the dequantised 68-byte row (E2M1 code * 2**(scale byte - 127) per
32-value block).  The formula is the scorer's definition as fixed by the
decode configuration (64 heads x dim 128, bf16 query, fp32 head weights); the
page (DS4X README, "Optimization details") states that the scorer reads the
packed 68-byte rows directly.

Top-k (DS4X README, "CSA score/top-512 fusion"): the k largest rows under the
float total order of the score, the lower row index winning ties; returned in
that order (score descending, index ascending).  With fewer than k rows the
tail is padded with -1.
"""

from __future__ import annotations

import numpy as np

from .codecs import bf16_decode, unpack_idx_rows


def score_rows(idx_rows, q_bf16, w, chunk: int = 65536) -> np.ndarray:
    """Scores of every row, float64 [n].

    idx_rows : uint8 [n, 68] packed indexer rows
    q_bf16   : uint16 [H, 128] bfloat16 bit patterns of the query
    w        : float32 [H] head weights
    """
    q = bf16_decode(q_bf16)  # [H, 128] exact
    w = np.asarray(w, dtype=np.float32).astype(np.float64)
    n = idx_rows.shape[0]
    out = np.empty(n, dtype=np.float64)
    for a in range(0, n, chunk):
        k = unpack_idx_rows(idx_rows[a:a + chunk])  # [c, 128]
        dots = k @ q.T  # [c, H]: q_h . k_t
        out[a:a + chunk] = np.maximum(dots, 0.0) @ w
    return out


def topk(scores, k: int):
    """Exact top-k: (indices int64 [k], scores float64 [k]) ordered by score
    descending, ties by lower index; -1 / NaN padding when len(scores) < k."""
    scores = np.asarray(scores, dtype=np.float64)
    n = scores.shape[0]
    # lexsort sorts by the last key first: primary -score, secondary index
    order = np.lexsort((np.arange(n), -scores))[: min(k, n)]
    idx = np.full(k, -1, dtype=np.int64)
    val = np.full(k, np.nan, dtype=np.float64)
    idx[: order.shape[0]] = order
    val[: order.shape[0]] = scores[order]
    return idx, val


def score_topk(idx_rows, q_bf16, w, k: int = 512):
    """Score every row then take the exact top-k; also returns all scores."""
    s = score_rows(idx_rows, q_bf16, w)
    idx, val = topk(s, k)
    return idx, val, s
