"""ds4x_cache_append vs the oracle's packer: bytes must be bit-exact."""

import numpy as np
import pytest

from gpu_path import pack, require_gpu
from oracle import codecs as C
from synth import decode_case

pytestmark = pytest.mark.gpu


def _host(t):
    return t.cpu().numpy()


@pytest.mark.parametrize("n,chunks", [(4096, 1), (1, 1), (37, 3), (1000, 7)])
def test_pack_bit_exact_synthetic(n, chunks):
    require_gpu()
    case = decode_case(n, 1000 + n)
    idx_rows, kv_rows = pack(case["idx_in"], case["kv_in"], chunks=chunks)
    assert np.array_equal(_host(idx_rows).reshape(n, 68), C.pack_idx_rows(case["idx_in"]))
    assert np.array_equal(_host(kv_rows).reshape(n, 583), C.pack_kv_rows(case["kv_in"]))


def _tie_blocks(grid, block, emax, rng, n_blocks):
    """Blocks whose scaled values hit every representable value, midpoint and
    the float32 neighbours of each, with a random power-of-two block scale and
    the block maximum pinned so the scale is known."""
    pts = []
    for a, b in zip(grid[:-1], grid[1:]):
        for p in (a, (a + b) / 2):
            p32 = np.float32(p)
            pts += [p32, np.nextafter(p32, np.float32(0)), np.nextafter(p32, np.float32(np.inf))]
    pts = np.array([p for p in pts if p <= emax], dtype=np.float32)
    out = np.empty((n_blocks, block), dtype=np.float32)
    for i in range(n_blocks):
        v = rng.choice(pts, size=block) * rng.choice(np.float32([-1, 1]), size=block)
        v[rng.integers(block)] = np.float32(emax)  # block max = emax exactly -> e = 0 before scaling
        e = int(rng.integers(-100, 100))
        out[i] = (v.astype(np.float64) * 2.0 ** e).astype(np.float32)
    return out


def test_pack_rounding_ties_and_midpoints():
    require_gpu()
    rng = np.random.default_rng(0)
    n = 512
    idx_in = _tie_blocks(C.e2m1_decode(np.arange(8)), 32, 6.0, rng, 4 * n).reshape(n, 128)
    nope = _tie_blocks(C.e4m3_decode(np.arange(127)), 64, 448.0, rng, 7 * n).reshape(n, 448)
    rope = (rng.standard_normal((n, 64)) * 10.0 ** rng.integers(-6, 4, (n, 1))).astype(np.float32)
    kv_in = np.concatenate([nope, rope], axis=1)
    idx_rows, kv_rows = pack(idx_in, kv_in)
    assert np.array_equal(_host(idx_rows).reshape(n, 68), C.pack_idx_rows(idx_in))
    assert np.array_equal(_host(kv_rows).reshape(n, 583), C.pack_kv_rows(kv_in))


def test_pack_special_values():
    """Zero blocks, negative values rounding to zero, tiny and huge scales,
    float32 subnormals."""
    require_gpu()
    n = 8
    idx_in = np.zeros((n, 128), dtype=np.float32)
    kv_in = np.zeros((n, 512), dtype=np.float32)
    idx_in[1, :32] = -1e-3
    idx_in[1, 5] = 6.0
    idx_in[2, 32:64] = np.float32(1e-40)  # float32 subnormals
    idx_in[3, 64:96] = np.float32(3e38)
    idx_in[3, 65] = -np.float32(1e30)
    idx_in[4] = -0.0
    kv_in[1, :64] = -1e-4
    kv_in[1, 3] = 448.0
    kv_in[2, 64:128] = np.float32(2e-41)
    kv_in[3, 128:192] = np.float32(3.3e38)
    kv_in[4, :] = -0.0
    kv_in[5, 448:] = np.float32([65504.0, 65520.0, 1e-8, -6e-5] * 16)
    idx_rows, kv_rows = pack(idx_in, kv_in)
    assert np.array_equal(_host(idx_rows).reshape(n, 68), C.pack_idx_rows(idx_in))
    assert np.array_equal(_host(kv_rows).reshape(n, 583), C.pack_kv_rows(kv_in))


def test_pack_one_side_only_and_offsets():
    """A layer without an indexer passes idx_rows = NULL; rows land at pos."""
    B = require_gpu()
    import torch

    case = decode_case(50, 3)
    cap = 80
    kv_rows = torch.full((cap * 583,), 0xAB, dtype=torch.uint8, device="cuda")
    B.ds4x_cache_append(kv_rows, None, 20, torch.from_numpy(case["kv_in"]).cuda(), None)
    host = kv_rows.cpu().numpy().reshape(cap, 583)
    assert np.all(host[:20] == 0xAB) and np.all(host[70:] == 0xAB)
    assert np.array_equal(host[20:70], C.pack_kv_rows(case["kv_in"]))
    idx_rows = torch.full((cap * 68,), 0xCD, dtype=torch.uint8, device="cuda")
    B.ds4x_cache_append(None, idx_rows, 79, None, torch.from_numpy(case["idx_in"][:1]).cuda())
    h2 = idx_rows.cpu().numpy().reshape(cap, 68)
    assert np.all(h2[:79] == 0xCD)
    assert np.array_equal(h2[79:], C.pack_idx_rows(case["idx_in"][:1]))
    with pytest.raises(B.Ds4xError):
        B.ds4x_cache_append(None, idx_rows, 79, None, torch.from_numpy(case["idx_in"][:2]).cuda())
