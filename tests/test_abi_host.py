"""The C-ABI library loads, exports every symbol include/ds4x.h declares,
and its host-side argument checks reject bad calls before any CUDA call
(so these run without a GPU)."""

import ctypes
import os
import re

import pytest

from conftest import ROOT, golden

HEADER = os.path.join(ROOT, "include", "ds4x.h")


@pytest.fixture(scope="module")
def lib():
    from compressed_kv_sparse_csa_gb300 import build as B

    if not os.path.exists(B.LIB_PATH):
        B.build()
    from compressed_kv_sparse_csa_gb300 import binding

    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ds4x_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n


def test_binding_covers_every_declared_function():
    from compressed_kv_sparse_csa_gb300 import binding

    for n in declared_functions():
        assert n in binding._SIGNATURES, n


def test_host_only_calls(lib):
    assert lib.ds4x_abi_version() == 1
    assert lib.ds4x_status_str(0) == b"ok"
    assert b"workspace" in lib.ds4x_status_str(-3)
    g = golden("packed_cache_abi.txt")
    assert lib.ds4x_cache_bytes(int(g["alloc_L"])) == int(g["alloc_total"])
    assert lib.ds4x_cache_bytes(0) == int(g["alloc_raw_rings"]) + 21 * 2 * 651 + 20 * 2 * 583
    assert lib.ds4x_cache_bytes(-1) == -1
    assert lib.ds4x_index_score_topk_workspace(1 << 20, 512) >= 256
    assert lib.ds4x_sparse_attn_decode_workspace(512) >= 256


FAKE = 0x10000  # aligned, never dereferenced: every call below fails its host check first


def test_append_argument_checks(lib):
    f = lib.ds4x_cache_append
    assert f(None, None, 10, 0, FAKE, FAKE, 1, None) == -1  # no destination
    assert f(FAKE, None, 10, 0, None, None, 1, None) == -1  # kv_rows without kv_in
    assert f(FAKE + 4, None, 10, 0, FAKE, None, 1, None) == -1  # misaligned
    assert f(FAKE, FAKE, 10, 0, FAKE, FAKE, 0, None) == -1  # n < 1
    assert f(FAKE, FAKE, 10, 8, FAKE, FAKE, 3, None) == -2  # pos + n > capacity
    assert f(FAKE, FAKE, 10, -1, FAKE, FAKE, 1, None) == -2


def test_score_argument_checks(lib):
    f = lib.ds4x_index_score_topk
    ws = lib.ds4x_index_score_topk_workspace(1000, 512)
    assert f(None, 1000, FAKE, FAKE, 512, FAKE, None, FAKE, ws, None) == -1
    assert f(FAKE, 0, FAKE, FAKE, 512, FAKE, None, FAKE, ws, None) == -1
    assert f(FAKE, 1000, FAKE, FAKE, 0, FAKE, None, FAKE, ws, None) == -1
    assert f(FAKE, 1000, FAKE, FAKE, 513, FAKE, None, FAKE, ws, None) == -1
    assert f(FAKE, 1000, FAKE + 8, FAKE, 512, FAKE, None, FAKE, ws, None) == -1
    assert f(FAKE, 1000, FAKE, FAKE, 512, FAKE, None, FAKE, ws - 1, None) == -3


def test_attention_argument_checks(lib):
    f = lib.ds4x_sparse_attn_decode
    ws = lib.ds4x_sparse_attn_decode_workspace(512)
    s = ctypes.c_float(0.044)
    assert f(FAKE, 10, None, 512, FAKE, s, FAKE, None, FAKE, ws, None) == -1
    assert f(FAKE, 0, FAKE, 512, FAKE, s, FAKE, None, FAKE, ws, None) == -1
    assert f(FAKE, 10, FAKE, 600, FAKE, s, FAKE, None, FAKE, ws, None) == -1
    assert f(FAKE, 10, FAKE, 512, FAKE, s, FAKE, FAKE + 4, FAKE, ws, None) == -1
    assert f(FAKE, 10, FAKE, 512, FAKE, s, FAKE, None, FAKE, ws - 1, None) == -3


def test_copy_argument_checks(lib):
    f = lib.ds4x_copy_async
    assert f(None, FAKE, 64, None) == -1
    assert f(FAKE, None, 64, None) == -1
    assert f(FAKE + 4, FAKE + 4096, 64, None) == -1  # misaligned
    assert f(FAKE, FAKE + 32, 64, None) == -1        # overlapping
    assert f(FAKE + 32, FAKE, 64, None) == -1
    assert f(FAKE, FAKE + 4096, 0, None) == 0        # nothing to copy: no CUDA call


def test_workspace_calls_reject_null(lib):
    assert lib.ds4x_workspace_init(None, 4096, None) == -1
    assert lib.ds4x_workspace_init(FAKE, 16, None) == -1
    out = ctypes.c_int32(0)
    assert lib.ds4x_workspace_status(None, None, ctypes.byref(out)) == -1


def test_batched_and_prefill_argument_checks(lib):
    s = ctypes.c_float(0.044)
    f = lib.ds4x_index_score_topk_batched
    ws = lib.ds4x_index_score_topk_batched_workspace(16, 512)
    assert f(None, FAKE, 16, FAKE, FAKE, 512, FAKE, None, FAKE, ws, None) == -1
    assert f(FAKE, FAKE, 0, FAKE, FAKE, 512, FAKE, None, FAKE, ws, None) == -1
    assert f(FAKE, FAKE, 65, FAKE, FAKE, 512, FAKE, None, FAKE, ws, None) == -1  # beyond DS4X_MAX_SESSIONS
    assert f(FAKE, FAKE, 16, FAKE, FAKE, 513, FAKE, None, FAKE, ws, None) == -1
    assert f(FAKE, FAKE, 16, FAKE, FAKE, 512, FAKE, None, FAKE, ws - 1, None) == -3
    g = lib.ds4x_sparse_attn_decode_batched
    wa = lib.ds4x_sparse_attn_decode_workspace(512)
    assert g(FAKE, None, 16, FAKE, 512, FAKE, s, FAKE, None, FAKE, wa, None) == -1
    assert g(FAKE, FAKE, 0, FAKE, 512, FAKE, s, FAKE, None, FAKE, wa, None) == -1
    assert g(FAKE, FAKE, 16, FAKE, 512, FAKE, s, FAKE, None, FAKE, wa - 1, None) == -3
    h = lib.ds4x_sparse_attn_prefill
    assert h(FAKE, 100, FAKE, 0, 512, FAKE, s, FAKE, None, FAKE, wa, None) == -1
    assert h(FAKE, 100, FAKE, 65536, 512, FAKE, s, FAKE, None, FAKE, wa, None) == -1
    assert h(FAKE, 0, FAKE, 8, 512, FAKE, s, FAKE, None, FAKE, wa, None) == -1
    assert h(FAKE, 100, FAKE + 4, 8, 512, FAKE, s, FAKE, None, FAKE, wa, None) == -1
    assert h(FAKE, 100, FAKE, 8, 512, FAKE, s, FAKE, None, FAKE, wa - 1, None) == -3


def test_prefill_scorer_argument_checks(lib):
    f = lib.ds4x_quantize_query_e4m3
    assert f(None, 4, FAKE, FAKE, None) == -1
    assert f(FAKE, 0, FAKE, FAKE, None) == -1
    assert f(FAKE, 4, FAKE + 4, FAKE, None) == -1
    g = lib.ds4x_index_score_topk_prefill
    ws = lib.ds4x_index_score_topk_prefill_workspace(65536, 2048, 512)
    assert ws >= 2048 * 64 * 128 * 2
    assert g(None, 65536, FAKE, FAKE, FAKE, 2048, 63488, 512, FAKE, None, FAKE, ws, None) == -1
    assert g(FAKE, 0, FAKE, FAKE, FAKE, 2048, 63488, 512, FAKE, None, FAKE, ws, None) == -1
    assert g(FAKE, 65536, FAKE, FAKE, FAKE, 0, 63488, 512, FAKE, None, FAKE, ws, None) == -1
    assert g(FAKE, 65536, FAKE, FAKE, FAKE, 2048, 63488, 0, FAKE, None, FAKE, ws, None) == -1
    assert g(FAKE, 65536, FAKE, FAKE, FAKE, 2048, 63488, 512, FAKE, None, FAKE, ws - 1, None) == -3


def test_dense_attention_argument_checks(lib):
    s = ctypes.c_float(0.044)
    wsz = lib.ds4x_dense_attn_decode_workspace
    # header, item LSEs (64 floats an item, rounded up to 256 bytes), item outputs (64 x 512 floats an
    # item); items of 128 rows up to 32,768 rows, then 256, 384 and 512 rows
    for n, items in [(1, 1), (128, 1), (129, 2), (8192, 64), (32768, 256), (32769, 129), (65536, 256),
                     (65537, 171), (98305, 193), (100000, 196), (8192 * 512, 8192)]:
        assert wsz(n) == 256 + ((items * 64 * 4 + 255) // 256) * 256 + items * 64 * 512 * 4, n
    f = lib.ds4x_dense_attn_decode
    ws = wsz(8192)
    assert f(None, 8192, FAKE, s, FAKE, None, FAKE, ws, None) == -1
    assert f(FAKE, 8192, None, s, FAKE, None, FAKE, ws, None) == -1
    assert f(FAKE, 8192, FAKE, s, None, None, FAKE, ws, None) == -1
    assert f(FAKE, 8192, FAKE, s, FAKE, None, None, ws, None) == -1
    assert f(FAKE, 0, FAKE, s, FAKE, None, FAKE, ws, None) == -1
    assert f(FAKE, 8192 * 512 + 1, FAKE, s, FAKE, None, FAKE, 1 << 40, None) == -1  # beyond DS4X_DENSE_MAX_ROWS
    assert f(FAKE + 4, 8192, FAKE, s, FAKE, None, FAKE, ws, None) == -1
    assert f(FAKE, 8192, FAKE, s, FAKE, FAKE + 4, FAKE, ws, None) == -1
    assert f(FAKE, 8192, FAKE, s, FAKE, None, FAKE, ws - 1, None) == -3


def test_window_attention_argument_checks(lib):
    s = ctypes.c_float(0.044)
    ws = lib.ds4x_window_sparse_attn_decode_workspace()
    # header, two items' LSEs and fp32 outputs, two index lists, two row pointers and lengths
    assert ws == 256 + 2 * 64 * 4 + 2 * 64 * 512 * 4 + 2 * 512 * 4 + 16 + 16
    f = lib.ds4x_window_sparse_attn_decode
    ok = (FAKE, 1000, FAKE, 512, FAKE, 10, 20, FAKE, s, FAKE, None, FAKE, ws, None)

    def call(**kw):
        names = ["kv", "n", "idx", "k", "ring", "pos", "w", "q", "scale", "out", "lse", "ws", "wsb", "stream"]
        args = dict(zip(names, ok))
        args.update(kw)
        return f(*[args[n] for n in names])

    for key in ("kv", "idx", "ring", "q", "out", "ws"):
        assert call(**{key: None}) == -1, key
    assert call(ring=FAKE + 4) == -1
    assert call(lse=FAKE + 4) == -1
    assert call(n=0) == -1
    assert call(k=0) == -1 and call(k=513) == -1
    assert call(pos=-1) == -1 and call(pos=256) == -1
    assert call(w=-1) == -1 and call(w=257) == -1
    assert call(wsb=ws - 1) == -3


def test_ring_rows_match_the_pages_allocation():
    """DS4X_RING_ROWS: the raw ring the pages' allocation example counts,
    43 layers x 256 rows x 583 bytes = the printed raw-ring bytes."""
    g = golden("packed_cache_abi.txt")
    text = open(HEADER).read()
    ring = int(re.search(r"#define DS4X_RING_ROWS (\d+)", text).group(1))
    assert 43 * ring * int(g["kv_row_bytes"]) == int(g["alloc_raw_rings"])


def test_decode_step_argument_checks(lib):
    s = ctypes.c_float(0.044)
    f = lib.ds4x_csa_decode_step
    ws = lib.ds4x_csa_decode_step_workspace(100000, 512)
    assert ws >= lib.ds4x_index_score_topk_workspace(100000, 512)
    assert ws >= lib.ds4x_sparse_attn_decode_workspace(512)
    ok = (FAKE, FAKE, 100000, FAKE, FAKE, 512, FAKE, s, FAKE, None, FAKE, None, FAKE, ws, None)
    for i in (0, 1, 3, 4, 6, 8, 10, 12):  # every required pointer
        args = list(ok)
        args[i] = None
        assert f(*args) == -1, i
    args = list(ok); args[1] = FAKE + 8
    assert f(*args) == -1  # misaligned
    args = list(ok); args[2] = 0
    assert f(*args) == -1
    args = list(ok); args[5] = 513
    assert f(*args) == -1
    args = list(ok); args[13] = ws - 1
    assert f(*args) == -3
