"""Parity rules shared by the GPU tests (CUDA path through the C ABI vs the
float64 oracle on the same seeded inputs).

* packed bytes: bit-exact;
* top-k: the index sets agree on every row whose oracle score lies outside
  a relative band of 1e-5 around the k-th oracle score (rows inside the band
  are near-ties that fp32 accumulation may legitimately reorder); the GPU
  list holds k distinct valid rows (then -1 padding), ordered by its own
  scores descending with the lower index first on ties, and its scores match
  the oracle's to fp32 accumulation accuracy;
* attention: the bf16 output against the bf16-rounded oracle output with
  max |diff| <= 2e-3 and ||diff||_2 / ||oracle||_2 <= 1e-3.
"""

import math

import numpy as np

TOPK_BAND = 1e-5
ATTN_MAX_ABS = 2e-3
ATTN_REL_L2 = 1e-3
# |s_gpu - s_oracle| bound: fp32 accumulation over 64 heads x 128 products of
# O(1) terms stays well inside 1e-5 relative of the score scale
SCORE_RTOL = 2e-5


def check_topk(gpu_idx, gpu_score, oracle_scores, k, band=TOPK_BAND):
    gpu_idx = np.asarray(gpu_idx, dtype=np.int64)
    s = np.asarray(oracle_scores, dtype=np.float64)
    n = s.shape[0]
    kk = min(k, n)
    assert np.all(gpu_idx[kk:] == -1), "padding past n_rows must be -1"
    sel = gpu_idx[:kk]
    assert np.all((sel >= 0) & (sel < n)), "index out of range"
    assert np.unique(sel).size == kk, "duplicate indices"
    order = np.lexsort((np.arange(n), -s))
    o_sel = order[:kk]
    s_k = s[o_sel[-1]]
    in_band = np.abs(s - s_k) <= band * abs(s_k)
    g = np.zeros(n, bool)
    g[sel] = True
    o = np.zeros(n, bool)
    o[o_sel] = True
    bad = np.nonzero((g != o) & ~in_band)[0]
    assert bad.size == 0, f"{bad.size} rows differ outside the near-tie band, e.g. {bad[:5]} scores {s[bad[:5]]} kth {s_k}"
    if gpu_score is not None:
        gs = np.asarray(gpu_score, dtype=np.float64)[:kk]
        scale = max(1.0, float(np.max(np.abs(s[sel]))))
        np.testing.assert_allclose(gs, s[sel], rtol=SCORE_RTOL, atol=SCORE_RTOL * scale)
        # the list is ordered by the GPU's own keys: score desc, index asc
        for a in range(kk - 1):
            assert gs[a] > gs[a + 1] or (gs[a] == gs[a + 1] and sel[a] < sel[a + 1]), a
        assert np.all(np.isnan(np.asarray(gpu_score, dtype=np.float64)[kk:]))
    return int(np.sum(in_band))


def bf16_ulp(x):
    """Spacing of bfloat16 values at |x| (8 significant bits)."""
    _, e = np.frexp(np.abs(np.asarray(x, dtype=np.float64)))
    return np.ldexp(1.0, np.maximum(e - 8, -133))


def check_attention(gpu_out_bf16_bits, oracle_out, max_abs=ATTN_MAX_ABS, rel_l2=ATTN_REL_L2, ulp_floor=False):
    """ulp_floor: for outputs far above the configured workload's |o| <~ 0.4
    (e.g. a near one-hot softmax), one bf16 rounding straddle alone exceeds
    2e-3; the per-element bound is then max(max_abs, 1 bf16 ulp of the
    oracle value)."""
    g = (np.asarray(gpu_out_bf16_bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    o = np.asarray(oracle_out, dtype=np.float64).reshape(g.shape)
    diff = g - o
    if ulp_floor:
        over = np.abs(diff) > np.maximum(max_abs, bf16_ulp(o))
        assert not np.any(over), f"{int(over.sum())} elements beyond max(2e-3, 1 bf16 ulp)"
        diff = np.where(np.abs(diff) <= bf16_ulp(o), np.minimum(np.abs(diff), max_abs), diff)
    ma = float(np.max(np.abs(diff)))
    denom = float(np.linalg.norm(o))
    rl = float(np.linalg.norm(diff)) / denom if denom > 0 else float(np.linalg.norm(diff))
    assert ma <= max_abs, f"max abs {ma}"
    assert rl <= rel_l2, f"rel L2 {rl}"
    return ma, rl


SOFTMAX_SCALE = 1.0 / math.sqrt(512.0)
