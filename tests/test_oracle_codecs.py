"""Pins for the oracle's element codecs, scale rule and packed rows.

Each check compares the oracle with something other than itself: torch's
independent FP8 / FP16 / E8M0 conversions, exhaustive brute force, exact
rational arithmetic, or values printed on the DS4X README."""

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import golden
from oracle import codecs as C


# ---------------------------------------------------------------------------
# A generic minifloat decoder, pinned below against torch's two FP8 formats,
# then used to pin the oracle's E2M1 table (torch has no CPU FP4 conversion).
# ---------------------------------------------------------------------------

def minifloat_value(code, ebits, mbits, bias):
    s = (code >> (ebits + mbits)) & 1
    e = (code >> mbits) & ((1 << ebits) - 1)
    m = code & ((1 << mbits) - 1)
    if e == 0:
        v = Fraction(m, 1 << mbits) * Fraction(2) ** (1 - bias)
    else:
        v = (1 + Fraction(m, 1 << mbits)) * Fraction(2) ** (e - bias)
    return -v if s else v


def _torch_fp8_values(dtype):
    t = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(dtype).to(torch.float64)
    return t.numpy()


@pytest.mark.parametrize("dtype,ebits,mbits,bias", [
    (torch.float8_e4m3fn, 4, 3, 7),
    (torch.float8_e5m2, 5, 2, 15),
])
def test_generic_minifloat_matches_torch_fp8(dtype, ebits, mbits, bias):
    ref = _torch_fp8_values(dtype)
    for c in range(256):
        if not np.isfinite(ref[c]):
            continue
        assert float(minifloat_value(c, ebits, mbits, bias)) == ref[c], c


def test_e4m3_decode_matches_torch_all_codes():
    ref = _torch_fp8_values(torch.float8_e4m3fn)
    got = C.e4m3_decode(np.arange(256))
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    fin = np.isfinite(ref)
    assert np.array_equal(ref[fin], got[fin])
    assert np.array_equal(np.signbit(ref[fin]), np.signbit(got[fin]))
    assert np.nanmax(got) == C.E4M3_MAX  # the configs' "amax/448"


def test_e2m1_decode_is_the_1_2_1_minifloat():
    got = C.e2m1_decode(np.arange(16))
    for c in range(16):
        assert got[c] == float(minifloat_value(c, 2, 1, 1))
    assert np.signbit(got[8]) and got[8] == 0.0
    assert got.max() == C.E2M1_MAX  # the configs' "amax/6"
    assert sorted(set(np.abs(got).tolist())) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_ue8m0_decode_matches_torch_e8m0():
    codes = np.arange(255)
    ref = torch.from_numpy(codes.astype(np.uint8)).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    assert np.array_equal(ref, C.ue8m0_decode(codes))
    assert np.isnan(C.ue8m0_decode(255))


def _probe_points(grid):
    """Every representable magnitude, every midpoint, and one float32 ulp on
    each side of them, with both signs and zeros."""
    pts = [0.0]
    for a, b in zip(grid[:-1], grid[1:]):
        mid = (a + b) / 2
        for p in (a, mid, b):
            p32 = np.float32(p)
            pts += [float(p32), float(np.nextafter(p32, np.float32(0))), float(np.nextafter(p32, np.float32(np.inf)))]
    pts = np.array(sorted(set(pts)))
    pts = pts[pts <= grid[-1]]
    return np.concatenate([pts, -pts, [-0.0]])


def test_e4m3_encode_matches_torch_rne():
    grid = C.e4m3_decode(np.arange(127))
    x = _probe_points(grid)
    rng = np.random.default_rng(7)
    x = np.concatenate([x, rng.uniform(-448, 448, 20000).astype(np.float32),
                        (rng.standard_normal(20000) * 0.01).astype(np.float32)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = C.e4m3_encode(x.astype(np.float64))
    bad = np.nonzero(ref != got)[0]
    assert bad.size == 0, (x[bad[:5]], ref[bad[:5]], got[bad[:5]])


def _brute_nearest_e2m1(x):
    vals = [float(minifloat_value(c, 2, 1, 1)) for c in range(8)]
    a = abs(x)
    best = None
    for c, v in enumerate(vals):
        d = abs(a - v)
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    return best[1] | (8 if math.copysign(1.0, x) < 0 else 0)


def test_e2m1_encode_brute_force():
    grid = C.e2m1_decode(np.arange(8))
    x = _probe_points(grid)
    rng = np.random.default_rng(8)
    x = np.concatenate([x, rng.uniform(-6, 6, 5000).astype(np.float32)])
    got = C.e2m1_encode(x)
    for xi, gi in zip(x, got):
        assert gi == _brute_nearest_e2m1(float(xi)), xi
    # the tie cases the scale rule relies on
    assert list(C.e2m1_encode([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])) == [0, 2, 2, 4, 4, 6, 6]
    assert C.e2m1_encode([-0.1])[0] == 0x8  # sign kept when rounding to zero


def test_fp16_encode_matches_torch():
    rng = np.random.default_rng(9)
    x = np.concatenate([rng.standard_normal(50000), rng.standard_normal(1000) * 1e-6,
                        [0.0, -0.0, 65504.0, 6.1e-5]]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ref, C.fp16_encode(x))


def _bf16_brute(x):
    """Exact nearest bfloat16 (ties to even) of a float64, by rationals."""
    fx = Fraction(x)
    if fx == 0:
        return 0.0
    e = math.frexp(abs(x))[1]
    q = Fraction(2) ** max(e - 8, -133)
    lo = (fx / q).__floor__()
    r = fx / q - lo
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return float(lo * q)


def test_bf16_round_direct_no_double_rounding():
    rng = np.random.default_rng(10)
    x = list(rng.standard_normal(3000) * 0.3)
    # float64 values just above a bf16 midpoint by less than a float32 ulp:
    # rounding through float32 first would land on the midpoint and tie down.
    for m in range(128, 140):
        mid = (m + 0.5) / 256.0
        x += [mid + 2.0 ** -40, mid - 2.0 ** -40, mid, -mid - 2.0 ** -40]
    got = C.bf16_round(np.array(x))
    for xi, gi in zip(x, got):
        assert gi == _bf16_brute(xi), xi
    # float32 inputs: agrees with torch's single-rounding conversion
    x32 = rng.standard_normal(20000).astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ref, C.bf16_round(x32.astype(np.float64)))


def _brute_exponent(amax, emax):
    if amax == 0:
        return 0
    for e in range(-400, 400):
        if Fraction(amax) <= Fraction(emax) * Fraction(2) ** e:
            return max(-127, min(127, e))
    raise AssertionError


@pytest.mark.parametrize("emax", [C.E2M1_MAX, C.E4M3_MAX])
def test_scale_exponent_brute_force(emax):
    rng = np.random.default_rng(11)
    pts = [0.0, 1.0, 2.0, 3.0, 6.0, 448.0, 224.0, 1e-30, 1e30, 1e-45, 3.4e38]
    for k in range(-140, 120, 7):
        b = np.float32(emax * 2.0 ** k)
        pts += [float(b), float(np.nextafter(b, np.float32(0))), float(np.nextafter(b, np.float32(np.inf)))]
    pts += list(np.abs(rng.standard_normal(300)).astype(np.float32) * 4)
    pts = np.array(pts, dtype=np.float32).astype(np.float64)
    got = C.scale_exponent(pts, emax)
    for a, g in zip(pts, got):
        assert g == _brute_exponent(a, emax), a


def test_scale_tightness():
    """After scaling, the block maximum lies in (emax/2, emax]."""
    rng = np.random.default_rng(12)
    v = rng.standard_normal((2000, 32)).astype(np.float32) * np.float32(2.0) ** rng.integers(-20, 20, (2000, 1)).astype(np.float32)
    for emax in (C.E2M1_MAX, C.E4M3_MAX):
        amax = np.max(np.abs(v), axis=1).astype(np.float64)
        e = C.scale_exponent(amax, emax)
        x = np.ldexp(amax, -e)
        assert np.all(x <= emax) and np.all(x > emax / 2)


def test_row_sizes_match_page():
    g = golden("packed_cache_abi.txt")
    assert C.KV_ROW_BYTES == int(g["kv_row_bytes"])
    assert C.KV_NOPE == int(g["kv_row_nope_bytes"])
    assert C.KV_ROPE == int(g["kv_row_rope_values"])
    assert C.KV_NBLOCKS == int(g["kv_row_scale_bytes"])
    assert C.IDX_ROW_BYTES == int(g["idx_row_bytes"])
    assert C.IDX_DIM == int(g["idx_row_values"])
    assert C.IDX_NBLOCKS == int(g["idx_row_scale_bytes"])
    rng = np.random.default_rng(13)
    assert C.pack_kv_rows(rng.standard_normal((3, 512))).shape == (3, 583)
    assert C.pack_idx_rows(rng.standard_normal((3, 128))).shape == (3, 68)


def test_idx_row_layout_and_roundtrip():
    """A block holding exactly representable values (with its maximum at
    6 * 2**e) round-trips exactly, and the bytes sit where the layout says."""
    vals = np.array([0.5, -1.0, 1.5, 2.0, -3.0, 4.0, 6.0, 0.0] * 4, dtype=np.float32)
    row = np.concatenate([vals * 2.0 ** -1, vals * 2.0 ** 3, -vals, vals * 2.0 ** -9]).astype(np.float32)
    packed = C.pack_idx_rows(row[None])
    assert np.array_equal(C.unpack_idx_rows(packed)[0], row.astype(np.float64))
    assert list(packed[0, 64:]) == [126, 130, 127, 118]
    # element 0 (0.25 / 2**-1 -> code 1) in the low nibble, element 1
    # (-0.5 / 2**-1 -> code 0xA) in the high nibble
    assert packed[0, 0] == (0x1 | (0xA << 4))


def test_kv_row_layout_and_roundtrip():
    rng = np.random.default_rng(14)
    grid = C.e4m3_decode(np.arange(127))
    nope = rng.choice(grid, size=448) * rng.choice([-1, 1], size=448)
    nope[::64] = 448.0  # pin every block's scale to 2**0
    nope[64:128] *= 2.0 ** -5
    rope = rng.standard_normal(64).astype(np.float16).astype(np.float32)
    row = np.concatenate([nope, rope]).astype(np.float32)
    packed = C.pack_kv_rows(row[None])
    assert np.array_equal(C.unpack_kv_rows(packed)[0], row.astype(np.float64))
    assert list(packed[0, 576:]) == [127, 122, 127, 127, 127, 127, 127]
    assert np.array_equal(packed[0, 448:576].view("<u2"), rope.astype(np.float16).view(np.uint16))


def test_zero_block_takes_scale_127():
    row = np.zeros((1, 128), dtype=np.float32)
    row[0, 40] = 1.0
    p = C.pack_idx_rows(row)
    assert list(p[0, 64:]) == [127, 125, 127, 127]
    assert np.all(p[0, :16] == 0)
