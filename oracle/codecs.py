"""Element codecs, block scales and packed rows -- float64 oracle.

Test infrastructure only (see ``oracle/__init__``).

Formats (DS4X README, "Packed cache ABI"; element formats as named there):

* KV row, 583 bytes = 448 E4M3 non-RoPE codes (element order)
                    + 64 FP16 RoPE values, little-endian (128 bytes)
                    + 7 UE8M0 scales, one per 64-value non-RoPE block.
* Indexer row, 68 bytes = 128 E2M1 codes, two per byte (64 bytes)
                        + 4 UE8M0 scales, one per 32-value block.

Readings where the page is silent:

* field order inside a row is the order the page lists the fields in;
* the even element of a pair sits in the low nibble of its byte;
* the block scale is 2**e with e the least integer such that
  amax <= emax * 2**e (emax = 6 for E2M1, 448 for E4M3), i.e. exactly
  ceil(log2(amax / emax)); a block with amax == 0 takes e = 0; e is
  clamped to [-127, 127]; the scale byte is e + 127;
* each element x = v * 2**-e (exact) is rounded to the nearest
  representable magnitude, ties to the even code; the sign of v is kept
  even when the magnitude rounds to zero;
* E4M3 is the "FN" variant: bias 7, subnormals m * 2**-9, max 448, no
  infinities, codes 0x7F / 0xFF are NaN and never produced.
"""

from __future__ import annotations

import numpy as np

KV_DIM = 512
KV_NOPE = 448
KV_ROPE = 64
KV_BLOCK = 64
KV_NBLOCKS = KV_NOPE // KV_BLOCK  # 7
KV_ROW_BYTES = KV_NOPE + 2 * KV_ROPE + KV_NBLOCKS  # 583

IDX_DIM = 128
IDX_BLOCK = 32
IDX_NBLOCKS = IDX_DIM // IDX_BLOCK  # 4
IDX_ROW_BYTES = IDX_DIM // 2 + IDX_NBLOCKS  # 68

E2M1_MAX = 6.0
E4M3_MAX = 448.0


# ---------------------------------------------------------------------------
# Element decoders: code -> float64 value
# ---------------------------------------------------------------------------

def e2m1_decode(codes) -> np.ndarray:
    """FP4 E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit, subnormals, no
    inf/NaN.  Magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6."""
    c = np.asarray(codes, dtype=np.int64) & 0xF
    sign = (c >> 3) & 1
    exp = (c >> 1) & 3
    man = c & 1
    mag = np.where(exp == 0, 0.5 * man, np.ldexp(1.0 + 0.5 * man, exp - 1))
    return np.where(sign == 1, -mag, mag)


def e4m3_decode(codes) -> np.ndarray:
    """FP8 E4M3 ("FN"): 1 sign, 4 exponent (bias 7), 3 mantissa bits,
    subnormals m*2**-9, no infinities, S.1111.111 is NaN."""
    c = np.asarray(codes, dtype=np.int64) & 0xFF
    sign = (c >> 7) & 1
    exp = (c >> 3) & 0xF
    man = c & 7
    mag = np.where(exp == 0, np.ldexp(man / 8.0, -6), np.ldexp(1.0 + man / 8.0, exp - 7))
    mag = np.where((exp == 15) & (man == 7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


def ue8m0_decode(codes) -> np.ndarray:
    """UE8M0 scale byte: 2**(b - 127); 255 is NaN."""
    b = np.asarray(codes, dtype=np.int64) & 0xFF
    return np.where(b == 255, np.nan, np.ldexp(1.0, b - 127))


def fp16_decode(bits) -> np.ndarray:
    """IEEE binary16 bit pattern -> value (exact)."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def bf16_decode(bits) -> np.ndarray:
    """bfloat16 bit pattern -> value (exact): the high half of a binary32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# Element encoders: nearest representable magnitude, ties to the even code
# ---------------------------------------------------------------------------

def _grid(decode, n_mag):
    """Positive magnitudes in code order (code == index); strictly ascending."""
    g = decode(np.arange(n_mag))
    assert np.all(np.diff(g) > 0)
    return g


_E2M1_GRID = None
_E4M3_GRID = None


def _nearest_code(x, grid, sign_bit):
    """Round each |x| to the nearest grid value (ties to the even index) and
    attach the sign of x.  |x| must not exceed grid[-1]."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    if np.any(a > grid[-1]):
        raise ValueError("magnitude above the format maximum")
    hi = np.searchsorted(grid, a, side="left")  # first grid value >= a
    hi = np.minimum(hi, len(grid) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - grid[lo]
    d_hi = grid[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.int64)
    neg = np.signbit(x)
    return (code | (neg.astype(np.int64) << sign_bit)).astype(np.uint8)


def e2m1_encode(x) -> np.ndarray:
    """x (already divided by the block scale, |x| <= 6) -> 4-bit code."""
    global _E2M1_GRID
    if _E2M1_GRID is None:
        _E2M1_GRID = _grid(e2m1_decode, 8)
    return _nearest_code(x, _E2M1_GRID, 3)


def e4m3_encode(x) -> np.ndarray:
    """x (already divided by the block scale, |x| <= 448) -> 8-bit code."""
    global _E4M3_GRID
    if _E4M3_GRID is None:
        _E4M3_GRID = _grid(e4m3_decode, 127)  # codes 0..126; 127 is NaN
    return _nearest_code(x, _E4M3_GRID, 7)


def fp16_encode(x) -> np.ndarray:
    """float -> IEEE binary16 bits, round to nearest even (numpy's cast)."""
    return np.asarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def bf16_round(x) -> np.ndarray:
    """Round float64 values directly to the nearest bfloat16 value (ties to
    even), returned as float64.  bfloat16 keeps 8 significant bits and the
    binary32 exponent range; its smallest subnormal is 2**-133."""
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)  # x = f * 2**e, 0.5 <= |f| < 1
    q = np.ldexp(1.0, np.maximum(e - 8, -133))  # spacing of bf16 values near x
    return np.rint(x / q) * q  # np.rint rounds half to even


def bf16_encode(x) -> np.ndarray:
    """float64 -> bfloat16 bits (direct RNE, no double rounding)."""
    r = bf16_round(x).astype(np.float32)  # exact: r is a bf16 value
    return (r.view(np.uint32) >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------
# Block scale rule
# ---------------------------------------------------------------------------

def scale_exponent(amax, emax) -> np.ndarray:
    """Least integer e with amax <= emax * 2**e, computed exactly.

    With amax = f * 2**F and emax = g * 2**G (0.5 <= f, g < 1), the answer is
    F - G when f <= g and F - G + 1 otherwise.  amax == 0 gives 0; the result
    is clamped to the UE8M0 range [-127, 127]."""
    amax = np.asarray(amax, dtype=np.float64)
    f, F = np.frexp(amax)
    g, G = np.frexp(np.float64(emax))
    e = F.astype(np.int64) - int(G) + (f > g).astype(np.int64)
    e = np.where(amax == 0, 0, e)
    return np.clip(e, -127, 127)


def quantize_blocks(v, block, emax, encode):
    """Split the last axis of v into blocks, scale each block by 2**-e and
    encode.  Returns (codes, scale_bytes) with codes in element order."""
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    lead = v.shape[:-1]
    nb = v.shape[-1] // block
    vb = v.reshape(*lead, nb, block)
    e = scale_exponent(np.max(np.abs(vb), axis=-1), emax)
    x = np.ldexp(vb, -e[..., None])  # exact power-of-two scaling
    codes = encode(x).reshape(*lead, nb * block)
    return codes, (e + 127).astype(np.uint8)


# ---------------------------------------------------------------------------
# Packed rows
# ---------------------------------------------------------------------------

def pack_idx_rows(idx_in) -> np.ndarray:
    """f32 [n, 128] -> uint8 [n, 68]: 64 code bytes then 4 scale bytes."""
    idx_in = np.asarray(idx_in, dtype=np.float32)
    n = idx_in.shape[0]
    codes, scales = quantize_blocks(idx_in, IDX_BLOCK, E2M1_MAX, e2m1_encode)
    pairs = codes.reshape(n, IDX_DIM // 2, 2).astype(np.uint8)
    packed = pairs[..., 0] | (pairs[..., 1] << 4)  # even element -> low nibble
    return np.concatenate([packed, scales], axis=1).astype(np.uint8)


def unpack_idx_rows(rows) -> np.ndarray:
    """uint8 [n, 68] -> float64 [n, 128] dequantised values."""
    rows = np.asarray(rows, dtype=np.uint8)
    n = rows.shape[0]
    b = rows[:, : IDX_DIM // 2].astype(np.int64)
    codes = np.stack([b & 0xF, b >> 4], axis=-1).reshape(n, IDX_DIM)
    vals = e2m1_decode(codes).reshape(n, IDX_NBLOCKS, IDX_BLOCK)
    scale = ue8m0_decode(rows[:, IDX_DIM // 2:])
    return (vals * scale[..., None]).reshape(n, IDX_DIM)


def pack_kv_rows(kv_in) -> np.ndarray:
    """f32 [n, 512] (448 non-RoPE then 64 RoPE) -> uint8 [n, 583]."""
    kv_in = np.asarray(kv_in, dtype=np.float32)
    n = kv_in.shape[0]
    codes, scales = quantize_blocks(kv_in[:, :KV_NOPE], KV_BLOCK, E4M3_MAX, e4m3_encode)
    rope = fp16_encode(kv_in[:, KV_NOPE:]).astype("<u2").view(np.uint8).reshape(n, 2 * KV_ROPE)
    return np.concatenate([codes, rope, scales], axis=1).astype(np.uint8)


def unpack_kv_rows(rows) -> np.ndarray:
    """uint8 [n, 583] -> float64 [n, 512] dequantised values."""
    rows = np.asarray(rows, dtype=np.uint8)
    n = rows.shape[0]
    nope = e4m3_decode(rows[:, :KV_NOPE]).reshape(n, KV_NBLOCKS, KV_BLOCK)
    scale = ue8m0_decode(rows[:, KV_NOPE + 2 * KV_ROPE:])
    nope = (nope * scale[..., None]).reshape(n, KV_NOPE)
    rope_bits = np.ascontiguousarray(rows[:, KV_NOPE:KV_NOPE + 2 * KV_ROPE]).view("<u2")
    rope = fp16_decode(rope_bits).reshape(n, KV_ROPE)
    return np.concatenate([nope, rope], axis=1)
