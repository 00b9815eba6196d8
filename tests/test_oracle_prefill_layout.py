"""Pins for the oracle's prefill scorer and the allocation formula.

The query quantiser is checked against torch's E4M3 conversion after the
pinned scale rule; causal scores against the decode scorer fed the
dequantised query (exact in bf16) and brute-force masking; the allocation
formula against the values printed on the DS4X README."""

import numpy as np
import torch

from conftest import golden
from oracle import codecs as C
from oracle import indexer as I
from oracle import layout as L
from oracle import prefill as P
from synth import prefill_case


def test_query_quantiser_matches_torch_e4m3():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((50, 64, 128)).astype(np.float32)
    codes, scales = P.quantize_query_e4m3(q)
    assert codes.shape == (50, 64, 128) and scales.shape == (50, 64, 4)
    e = scales.astype(np.int64) - 127
    x = np.ldexp(q.reshape(50, 64, 4, 32).astype(np.float64), -e[..., None]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy().reshape(50, 64, 128)
    assert np.array_equal(codes, ref)
    amax = np.abs(q.reshape(50, 64, 4, 32)).max(-1)
    assert np.all(amax <= 448.0 * 2.0 ** e) and np.all(amax > 224.0 * 2.0 ** e)


def test_query_dequantiser_matches_torch_e4m3_times_scale():
    """Each 32-value block decodes as torch's float8_e4m3fn value of the code
    times 2**(scale byte - 127), block b = elements 32b..32b+31 (so a wrong
    scale axis, block width or code order fails here, independently of the
    quantiser it usually feeds)."""
    rng = np.random.default_rng(21)
    codes = rng.integers(0, 256, size=(7, 64, 128), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    scales = rng.integers(100, 155, size=(7, 64, 4), dtype=np.uint8)
    # special blocks: every finite code once, extreme and unit scales, a constant block
    codes[0, 0, :126] = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)[:126]
    codes[0, 1, :] = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)[126:254]
    scales[0, 0] = [1, 127, 200, 254]
    scales[0, 1] = [127, 0, 127, 250]
    codes[1, 2, 64:96] = 0x38  # 1.0 in E4M3
    scales[1, 2, 2] = 130
    got = P.dequantize_query_e4m3(codes, scales)
    dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    factor = np.repeat(2.0 ** (scales.astype(np.float64) - 127.0), 32, axis=-1)
    ref = dec * factor
    assert got.shape == (7, 64, 128)
    assert np.array_equal(got, ref)
    assert np.all(got[1, 2, 64:96] == 8.0)


def test_prefill_scores_causal_and_consistent_with_decode():
    case = prefill_case(T=6, n=300, causal_base=290)
    rows = C.pack_idx_rows(case["idx_in"])
    codes, scales = P.quantize_query_e4m3(case["q"])
    s = P.prefill_scores(rows, codes, scales, case["w"], 290)
    for i in range(6):
        vis = min(300, 290 + i)
        assert np.all(np.isneginf(s[i, vis:])) and np.all(np.isfinite(s[i, :vis]))
        qhat = P.dequantize_query_e4m3(codes[i], scales[i])
        qbits = C.bf16_encode(qhat)
        assert np.array_equal(C.bf16_decode(qbits), qhat)  # E4M3 values are exact in bf16
        ref = I.score_rows(rows[:vis], qbits, case["w"][i])
        np.testing.assert_allclose(s[i, :vis], ref, rtol=1e-13)
    idx, val, _ = P.prefill_topk(rows, codes, scales, case["w"], 290, k=512)
    assert np.all(idx[0, 290:] == -1) and np.all(idx[0, :290] >= 0)
    assert set(idx[5, :295].tolist()) == set(range(295))


def test_allocation_formula_matches_page():
    g = golden("packed_cache_abi.txt")
    Lt = int(g["alloc_L"])
    assert L.raw_ring_bytes() == int(g["alloc_raw_rings"])
    assert L.compressed_bytes(Lt) == int(g["alloc_compressed"])
    assert L.kv_cache_bytes(Lt) == int(g["alloc_total"])
    assert L.csa_rows(Lt) == 262146
