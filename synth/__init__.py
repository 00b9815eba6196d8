"""Seeded synthetic inputs for the compressed-KV sparse-attention decode path.

This module only draws random numbers; it holds none of the method's
arithmetic (no quantisation, packing, scoring or attention).  Both the CUDA
path (through its C ABI) and the CPU oracle consume what it returns.

Recipe (numpy PCG64, one generator per case, draws in this order):

1. indexer keys      f32 [N, 128]  ~ N(0, 1)
2. KV non-RoPE       f32 [N, 448]  ~ N(0, 1)
3. KV RoPE           f32 [N, 64]   ~ N(0, 1)
4. indexer query     [64, 128]     ~ N(0, 1), rounded to bfloat16
5. head weights      f32 [64]      ~ U(0, 1) / 8
6. attention query   [64, 512]     ~ N(0, 1), rounded to bfloat16

Named workloads: tiny decode N = 4096 (seed 1000), mid decode N = 131072
(seed 1001), long decode N = 1048576 (seed 1002), 16 ragged sessions with
lengths uniform on [8192, 65536] (seed 1003, lengths drawn first, then each
session's arrays in the order above), chunked prefill of 2048 queries over
65536 rows (seed 1004); indexer-only cases (keys, query, weights, in that
order) for scorer checks beyond the long workload.  bfloat16 values are
carried as uint16 bit patterns.
"""

from __future__ import annotations

import numpy as np

IDX_HEADS = 64
IDX_DIM = 128
KV_NOPE = 448
KV_ROPE = 64
KV_DIM = 512
ATTN_HEADS = 64

DECODE_WORKLOADS = {
    "tiny": (4096, 1000),
    "mid": (131072, 1001),
    "long": (1048576, 1002),
}
SESSIONS_SEED = 1003
PREFILL_SEED = 1004


def to_bf16_bits(x) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even) -> uint16 bits.
    Uses torch's conversion so this module carries no rounding code."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def _normal(rng, shape):
    return rng.standard_normal(shape, dtype=np.float32)


def _draw_rows(rng, n):
    idx_in = _normal(rng, (n, IDX_DIM))
    kv = np.empty((n, KV_DIM), dtype=np.float32)
    kv[:, :KV_NOPE] = _normal(rng, (n, KV_NOPE))
    kv[:, KV_NOPE:] = _normal(rng, (n, KV_ROPE))
    return idx_in, kv


def _draw_decode_query(rng):
    q_idx = to_bf16_bits(_normal(rng, (IDX_HEADS, IDX_DIM)))
    w = (rng.random(IDX_HEADS, dtype=np.float32) / np.float32(8.0)).astype(np.float32)
    q_attn = to_bf16_bits(_normal(rng, (ATTN_HEADS, KV_DIM)))
    return q_idx, w, q_attn


def decode_case(n: int, seed: int) -> dict:
    """One batch-1 decode layer with n compressed rows."""
    rng = np.random.Generator(np.random.PCG64(seed))
    idx_in, kv_in = _draw_rows(rng, n)
    q_idx, w, q_attn = _draw_decode_query(rng)
    return {"n": n, "idx_in": idx_in, "kv_in": kv_in, "q_idx": q_idx, "w": w, "q_attn": q_attn}


def indexer_case(n: int, seed: int) -> dict:
    """Only the indexer side of a decode layer with n compressed rows (keys,
    query, head weights; same distributions as ``decode_case``), for cases
    too large to draw KV rows for."""
    rng = np.random.Generator(np.random.PCG64(seed))
    idx_in = _normal(rng, (n, IDX_DIM))
    q_idx = to_bf16_bits(_normal(rng, (IDX_HEADS, IDX_DIM)))
    w = (rng.random(IDX_HEADS, dtype=np.float32) / np.float32(8.0)).astype(np.float32)
    return {"n": n, "idx_in": idx_in, "q_idx": q_idx, "w": w}


def workload(name: str) -> dict:
    n, seed = DECODE_WORKLOADS[name]
    return decode_case(n, seed)


def sessions_case(n_sess: int = 16, lo: int = 8192, hi: int = 65536, seed: int = SESSIONS_SEED,
                  scale_lengths: float = 1.0) -> list:
    """Independent decode sessions with ragged history lengths.
    scale_lengths < 1 shrinks every length (for quick tests); the draw order
    is unchanged."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lengths = rng.integers(lo, hi + 1, size=n_sess)
    out = []
    for n in lengths:
        n = max(1, int(int(n) * scale_lengths))
        idx_in, kv_in = _draw_rows(rng, n)
        q_idx, w, q_attn = _draw_decode_query(rng)
        out.append({"n": n, "idx_in": idx_in, "kv_in": kv_in, "q_idx": q_idx, "w": w, "q_attn": q_attn})
    return out


def prefill_case(T: int = 2048, n: int = 65536, causal_base: int = 63488, seed: int = PREFILL_SEED) -> dict:
    """A chunk of T prefill queries over n history rows; query i sees rows
    t < causal_base + i."""
    rng = np.random.Generator(np.random.PCG64(seed))
    idx_in, kv_in = _draw_rows(rng, n)
    q = _normal(rng, (T, IDX_HEADS, IDX_DIM))
    w = (rng.random((T, IDX_HEADS), dtype=np.float32) / np.float32(8.0)).astype(np.float32)
    q_attn = to_bf16_bits(_normal(rng, (T, ATTN_HEADS, KV_DIM)))
    return {"n": n, "T": T, "causal_base": causal_base, "idx_in": idx_in, "kv_in": kv_in,
            "q": q, "w": w, "q_attn": q_attn}
