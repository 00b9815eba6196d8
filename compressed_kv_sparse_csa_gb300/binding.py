"""ctypes binding of libds4x (include/ds4x.h): argument marshalling only.

Every function takes torch tensors on the current CUDA device, checks their
dtype / shape / contiguity, and passes raw device pointers and the current
stream to the C entry point of the same name.  All computation runs in the
library's CUDA kernels; there is no Python or CPU fallback.  A missing or
unloadable library raises at first use.
"""

from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH

_LIB = None

_c_i32 = ctypes.c_int32
_c_i64 = ctypes.c_int64
_c_size = ctypes.c_size_t
_c_p = ctypes.c_void_p
_c_f32 = ctypes.c_float

_SIGNATURES = {
    "ds4x_status_str": (ctypes.c_char_p, [ctypes.c_int]),
    "ds4x_abi_version": (ctypes.c_int, []),
    "ds4x_cache_bytes": (_c_i64, [_c_i64]),
    "ds4x_workspace_init": (ctypes.c_int, [_c_p, _c_size, _c_p]),
    "ds4x_copy_async": (ctypes.c_int, [_c_p, _c_p, _c_size, _c_p]),
    "ds4x_workspace_status": (ctypes.c_int, [_c_p, _c_p, ctypes.POINTER(_c_i32)]),
    "ds4x_cache_append": (ctypes.c_int, [_c_p, _c_p, _c_i64, _c_i64, _c_p, _c_p, _c_i64, _c_p]),
    "ds4x_index_score_topk_workspace": (_c_size, [_c_i64, _c_i32]),
    "ds4x_index_score_topk": (ctypes.c_int, [_c_p, _c_i64, _c_p, _c_p, _c_i32, _c_p, _c_p, _c_p, _c_size, _c_p]),
    "ds4x_sparse_attn_decode_workspace": (_c_size, [_c_i32]),
    "ds4x_sparse_attn_decode": (ctypes.c_int, [_c_p, _c_i64, _c_p, _c_i32, _c_p, _c_f32, _c_p, _c_p, _c_p, _c_size, _c_p]),
    "ds4x_sparse_attn_decode_noalloc": (ctypes.c_int, [_c_p, _c_i64, _c_p, _c_i32, _c_p, _c_f32, _c_p, _c_p, _c_p]),
    "ds4x_dense_attn_decode_workspace": (_c_size, [_c_i64]),
    "ds4x_dense_attn_decode": (ctypes.c_int, [_c_p, _c_i64, _c_p, _c_f32, _c_p, _c_p, _c_p, _c_size, _c_p]),
    "ds4x_window_sparse_attn_decode_workspace": (_c_size, []),
    "ds4x_checkpoint_bytes": (_c_i64, [_c_p, _c_i32]),
    "ds4x_checkpoint_save": (ctypes.c_int, [_c_p, _c_i32, _c_p, _c_i64]),
    "ds4x_checkpoint_inspect": (ctypes.c_int, [_c_p, _c_i64, _c_p, _c_p, _c_i32]),
    "ds4x_checkpoint_load": (ctypes.c_int, [_c_p, _c_i64, _c_p, _c_i32]),
    "ds4x_window_sparse_attn_decode": (ctypes.c_int, [_c_p, _c_i64, _c_p, _c_i32, _c_p, _c_i32, _c_i32, _c_p, _c_f32,
                                                      _c_p, _c_p, _c_p, _c_size, _c_p]),
    "ds4x_csa_decode_step_workspace": (_c_size, [_c_i64, _c_i32]),
    "ds4x_csa_decode_step": (ctypes.c_int, [_c_p, _c_p, _c_i64, _c_p, _c_p, _c_i32, _c_p, _c_f32, _c_p, _c_p, _c_p,
                                            _c_p, _c_p, _c_size, _c_p]),
    "ds4x_index_score_topk_batched_workspace": (_c_size, [_c_i32, _c_i32]),
    "ds4x_index_score_topk_batched": (ctypes.c_int, [_c_p, _c_p, _c_i32, _c_p, _c_p, _c_i32, _c_p, _c_p, _c_p, _c_size,
                                                      _c_p]),
    "ds4x_sparse_attn_decode_batched": (ctypes.c_int, [_c_p, _c_p, _c_i32, _c_p, _c_i32, _c_p, _c_f32, _c_p, _c_p, _c_p,
                                                        _c_size, _c_p]),
    "ds4x_sparse_attn_prefill": (ctypes.c_int, [_c_p, _c_i64, _c_p, _c_i32, _c_i32, _c_p, _c_f32, _c_p, _c_p, _c_p,
                                                 _c_size, _c_p]),
    "ds4x_quantize_query_e4m3": (ctypes.c_int, [_c_p, _c_i64, _c_p, _c_p, _c_p]),
    "ds4x_index_score_topk_prefill_workspace": (_c_size, [_c_i64, _c_i32, _c_i32]),
    "ds4x_index_score_topk_prefill": (ctypes.c_int, [_c_p, _c_i64, _c_p, _c_p, _c_p, _c_i32, _c_i64, _c_i32, _c_p, _c_p,
                                                      _c_p, _c_size, _c_p]),
}


class Ds4xError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {status} ({status_str(status)})")


def lib():
    """Load libds4x.so (built by __graft_entry__.build()); raise if absent."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run __graft_entry__.build() first")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _LIB = L
    return _LIB


def status_str(status: int) -> str:
    return lib().ds4x_status_str(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t, dtype, name, numel=None, allow_none=False):
    if t is None:
        if allow_none:
            return
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements, needs {numel}")


def _call(fn, *args):
    st = getattr(lib(), fn)(*args)
    if st != 0:
        raise Ds4xError(fn, st)


def ds4x_abi_version() -> int:
    return lib().ds4x_abi_version()


def ds4x_cache_bytes(context_tokens: int) -> int:
    return lib().ds4x_cache_bytes(int(context_tokens))


def ds4x_workspace_init(ws, stream=None):
    _check(ws, torch.uint8, "ws")
    _call("ds4x_workspace_init", _ptr(ws), ws.numel(), _stream(stream))


def ds4x_copy_async(dst, src, stream=None):
    """Kernel-side copy of src's bytes into dst (each a contiguous CUDA tensor
    or a pinned host tensor; same number of bytes)."""
    for name, t in (("dst", dst), ("src", src)):
        if not (t.is_cuda or t.is_pinned()):
            raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    nbytes = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != nbytes:
        raise ValueError("dst and src differ in size")
    _call("ds4x_copy_async", _ptr(dst), _ptr(src), nbytes, _stream(stream))


def ds4x_workspace_status(ws, stream=None) -> int:
    _check(ws, torch.uint8, "ws")
    out = _c_i32(0)
    _call("ds4x_workspace_status", _ptr(ws), _stream(stream), ctypes.byref(out))
    return out.value


def ds4x_cache_append(kv_rows, idx_rows, pos, kv_in, idx_in, stream=None):
    """Pack kv_in f32 [n, 512] / idx_in f32 [n, 128] into rows [pos, pos+n)
    of kv_rows u8 [cap, 583] / idx_rows u8 [cap, 68] (either may be None)."""
    _check(kv_rows, torch.uint8, "kv_rows", allow_none=True)
    _check(idx_rows, torch.uint8, "idx_rows", allow_none=True)
    _check(kv_in, torch.float32, "kv_in", allow_none=kv_rows is None)
    _check(idx_in, torch.float32, "idx_in", allow_none=idx_rows is None)
    src = kv_in if kv_in is not None else idx_in
    n = src.shape[0]
    cap = (kv_rows if kv_rows is not None else idx_rows).numel() // (583 if kv_rows is not None else 68)
    if kv_rows is not None and idx_rows is not None and idx_rows.numel() // 68 != cap:
        raise ValueError("kv_rows and idx_rows hold different row counts")
    _call("ds4x_cache_append", _ptr(kv_rows), _ptr(idx_rows), cap, int(pos), _ptr(kv_in), _ptr(idx_in), n,
          _stream(stream))


def ds4x_index_score_topk_workspace(n_rows: int, k: int) -> int:
    return lib().ds4x_index_score_topk_workspace(int(n_rows), int(k))


def ds4x_index_score_topk(idx_rows, n_rows, q_bf16, w, k, out_idx, out_score, ws, stream=None):
    """Score n_rows packed indexer rows and write the exact top-k indices
    (and scores, if out_score is given) in score-descending order."""
    _check(idx_rows, torch.uint8, "idx_rows", numel=int(n_rows) * 68)
    _check(q_bf16, torch.bfloat16, "q_bf16", numel=64 * 128)
    _check(w, torch.float32, "w", numel=64)
    _check(out_idx, torch.int32, "out_idx", numel=int(k))
    _check(out_score, torch.float32, "out_score", numel=int(k), allow_none=True)
    _check(ws, torch.uint8, "ws")
    _call("ds4x_index_score_topk", _ptr(idx_rows), int(n_rows), _ptr(q_bf16), _ptr(w), int(k), _ptr(out_idx),
          _ptr(out_score), _ptr(ws), ws.numel(), _stream(stream))


def ds4x_sparse_attn_decode_workspace(k: int) -> int:
    return lib().ds4x_sparse_attn_decode_workspace(int(k))


def ds4x_sparse_attn_decode(kv_rows, n_rows, idx, k, q_bf16, softmax_scale, out_bf16, lse, ws, stream=None):
    """Decode attention of q_bf16 [64, 512] over the k rows listed in idx."""
    _check(kv_rows, torch.uint8, "kv_rows", numel=int(n_rows) * 583)
    _check(idx, torch.int32, "idx", numel=int(k))
    _check(q_bf16, torch.bfloat16, "q_bf16", numel=64 * 512)
    _check(out_bf16, torch.bfloat16, "out_bf16", numel=64 * 512)
    _check(lse, torch.float32, "lse", numel=64, allow_none=True)
    _check(ws, torch.uint8, "ws")
    _call("ds4x_sparse_attn_decode", _ptr(kv_rows), int(n_rows), _ptr(idx), int(k), _ptr(q_bf16),
          float(softmax_scale), _ptr(out_bf16), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))


def ds4x_dense_attn_decode_workspace(n_rows: int) -> int:
    return lib().ds4x_dense_attn_decode_workspace(int(n_rows))


def ds4x_dense_attn_decode(kv_rows, n_rows, q_bf16, softmax_scale, out_bf16, lse, ws, stream=None):
    """Dense decode attention of q_bf16 [64, 512] over every row [0, n_rows)
    of kv_rows (the HCA layers' attention over all compressed rows)."""
    _check(kv_rows, torch.uint8, "kv_rows", numel=int(n_rows) * 583)
    _check(q_bf16, torch.bfloat16, "q_bf16", numel=64 * 512)
    _check(out_bf16, torch.bfloat16, "out_bf16", numel=64 * 512)
    _check(lse, torch.float32, "lse", numel=64, allow_none=True)
    _check(ws, torch.uint8, "ws")
    _call("ds4x_dense_attn_decode", _ptr(kv_rows), int(n_rows), _ptr(q_bf16), float(softmax_scale), _ptr(out_bf16),
          _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))


def ds4x_window_sparse_attn_decode_workspace() -> int:
    return lib().ds4x_window_sparse_attn_decode_workspace()


def ds4x_window_sparse_attn_decode(kv_rows, n_rows, idx, k, ring_rows, ring_pos, w, q_bf16, softmax_scale, out_bf16,
                                   lse, ws, stream=None):
    """Decode attention of q_bf16 [64, 512] over the k rows listed in idx and
    the raw window's w ring rows (slots ring_pos, ring_pos - 1, ... mod 256)."""
    _check(kv_rows, torch.uint8, "kv_rows", numel=int(n_rows) * 583)
    _check(idx, torch.int32, "idx", numel=int(k))
    _check(ring_rows, torch.uint8, "ring_rows", numel=256 * 583)
    _check(q_bf16, torch.bfloat16, "q_bf16", numel=64 * 512)
    _check(out_bf16, torch.bfloat16, "out_bf16", numel=64 * 512)
    _check(lse, torch.float32, "lse", numel=64, allow_none=True)
    _check(ws, torch.uint8, "ws")
    _call("ds4x_window_sparse_attn_decode", _ptr(kv_rows), int(n_rows), _ptr(idx), int(k), _ptr(ring_rows),
          int(ring_pos), int(w), _ptr(q_bf16), float(softmax_scale), _ptr(out_bf16), _ptr(lse), _ptr(ws), ws.numel(),
          _stream(stream))


# ---- packed-row checkpoints: host memory (numpy uint8 arrays and bytes) ----

class _LayerRows(ctypes.Structure):
    _fields_ = [("ratio", _c_i32), ("ring_live", _c_i32), ("ring_pos", _c_i32), ("reserved", _c_i32),
                ("ring_rows", _c_p), ("kv_rows", _c_p), ("idx_rows", _c_p), ("n_kv", _c_i64), ("n_idx", _c_i64)]


class _LayerCounts(ctypes.Structure):
    _fields_ = [("ratio", _c_i32), ("ring_live", _c_i32), ("n_kv", _c_i64), ("n_idx", _c_i64)]


class _LayerBuffers(ctypes.Structure):
    _fields_ = [("ring_rows", _c_p), ("kv_rows", _c_p), ("idx_rows", _c_p), ("kv_cap", _c_i64), ("idx_cap", _c_i64)]


def _np_ptr(a):
    import numpy as np

    if a is None:
        return None
    if not (isinstance(a, np.ndarray) and a.dtype == np.uint8 and a.flags["C_CONTIGUOUS"]):
        raise ValueError("checkpoint rows must be contiguous numpy uint8 arrays")
    return a.ctypes.data


def _layer_rows(layers):
    arr = (_LayerRows * max(1, len(layers)))()
    for i, L in enumerate(layers):
        kv, ix = L.get("kv_rows"), L.get("idx_rows")
        arr[i] = _LayerRows(int(L["ratio"]), int(L.get("ring_live", 0)), int(L.get("ring_pos", 0)), 0,
                            _np_ptr(L.get("ring_rows")), _np_ptr(kv), _np_ptr(ix),
                            0 if kv is None else kv.size // 583, 0 if ix is None else ix.size // 68)
    return arr


def ds4x_checkpoint_save(layers) -> bytes:
    """layers: dicts with ratio, ring_live, ring_pos, ring_rows (uint8 [256 * 583],
    physical order), kv_rows (uint8 [n * 583]) and idx_rows (uint8 [n * 68])."""
    arr = _layer_rows(layers)
    nbytes = lib().ds4x_checkpoint_bytes(ctypes.addressof(arr), len(layers))
    if nbytes < 0:
        raise Ds4xError("ds4x_checkpoint_bytes", int(nbytes))
    out = ctypes.create_string_buffer(int(nbytes))
    _call("ds4x_checkpoint_save", ctypes.addressof(arr), len(layers), ctypes.addressof(out), int(nbytes))
    return out.raw


def ds4x_checkpoint_inspect(data: bytes):
    """The layer counts of a checkpoint (raises Ds4xError for a bad one)."""
    n = _c_i32(0)
    buf = ctypes.create_string_buffer(bytes(data), len(data))
    _call("ds4x_checkpoint_inspect", ctypes.addressof(buf), len(data), ctypes.byref(n), None, 0)
    counts = (_LayerCounts * max(1, n.value))()
    _call("ds4x_checkpoint_inspect", ctypes.addressof(buf), len(data), ctypes.byref(n), ctypes.addressof(counts),
          n.value)
    return [{"ratio": c.ratio, "ring_live": c.ring_live, "n_kv": c.n_kv, "n_idx": c.n_idx} for c in counts[:n.value]]


def ds4x_checkpoint_load(data: bytes, bufs):
    """Loads into bufs: dicts with ring_rows (uint8 [256 * 583]), kv_rows and
    idx_rows (uint8, their capacity in rows from their size)."""
    arr = (_LayerBuffers * max(1, len(bufs)))()
    for i, b in enumerate(bufs):
        kv, ix = b.get("kv_rows"), b.get("idx_rows")
        arr[i] = _LayerBuffers(_np_ptr(b.get("ring_rows")), _np_ptr(kv), _np_ptr(ix),
                               0 if kv is None else kv.size // 583, 0 if ix is None else ix.size // 68)
    buf = ctypes.create_string_buffer(bytes(data), len(data))
    _call("ds4x_checkpoint_load", ctypes.addressof(buf), len(data), ctypes.addressof(arr), len(bufs))


def ds4x_sparse_attn_decode_noalloc(kv_rows, n_rows, idx, k, q_bf16, softmax_scale, out_bf16, lse, stream=None):
    """ds4x_sparse_attn_decode without a workspace, for callers that cannot
    allocate device memory at decode time; its scratch is a static array
    inside the library shared by all calls (serialise overlapping calls)."""
    _check(kv_rows, torch.uint8, "kv_rows", numel=int(n_rows) * 583)
    _check(idx, torch.int32, "idx", numel=int(k))
    _check(q_bf16, torch.bfloat16, "q_bf16", numel=64 * 512)
    _check(out_bf16, torch.bfloat16, "out_bf16", numel=64 * 512)
    _check(lse, torch.float32, "lse", numel=64, allow_none=True)
    _call("ds4x_sparse_attn_decode_noalloc", _ptr(kv_rows), int(n_rows), _ptr(idx), int(k), _ptr(q_bf16),
          float(softmax_scale), _ptr(out_bf16), _ptr(lse), _stream(stream))


def ds4x_csa_decode_step_workspace(n_rows: int, k: int) -> int:
    return lib().ds4x_csa_decode_step_workspace(int(n_rows), int(k))


def ds4x_csa_decode_step(idx_rows, kv_rows, n_rows, q_idx_bf16, w, k, q_attn_bf16, softmax_scale, out_idx, out_score,
                         out_bf16, lse, ws, stream=None):
    """One decode step: score + exact top-k over idx_rows, then attention of
    q_attn_bf16 [64, 512] over the selected kv_rows."""
    n = int(n_rows)
    _check(idx_rows, torch.uint8, "idx_rows", numel=n * 68)
    _check(kv_rows, torch.uint8, "kv_rows", numel=n * 583)
    _check(q_idx_bf16, torch.bfloat16, "q_idx_bf16", numel=64 * 128)
    _check(w, torch.float32, "w", numel=64)
    _check(q_attn_bf16, torch.bfloat16, "q_attn_bf16", numel=64 * 512)
    _check(out_idx, torch.int32, "out_idx", numel=int(k))
    _check(out_score, torch.float32, "out_score", numel=int(k), allow_none=True)
    _check(out_bf16, torch.bfloat16, "out_bf16", numel=64 * 512)
    _check(lse, torch.float32, "lse", numel=64, allow_none=True)
    _check(ws, torch.uint8, "ws")
    _call("ds4x_csa_decode_step", _ptr(idx_rows), _ptr(kv_rows), n, _ptr(q_idx_bf16), _ptr(w), int(k),
          _ptr(q_attn_bf16), float(softmax_scale), _ptr(out_idx), _ptr(out_score), _ptr(out_bf16), _ptr(lse), _ptr(ws),
          ws.numel(), _stream(stream))


def ds4x_index_score_topk_batched_workspace(n_sess: int, k: int) -> int:
    return lib().ds4x_index_score_topk_batched_workspace(int(n_sess), int(k))


def ds4x_index_score_topk_batched(idx_row_ptrs, n_rows, q_bf16, w, k, out_idx, out_score, ws, stream=None):
    """Score + exact top-k for a batch of sessions: idx_row_ptrs int64 [S]
    holds each session's device row pointer, n_rows int64 [S] its length;
    q_bf16 [S, 64, 128], w [S, 64], out_idx int32 [S, k]."""
    _check(idx_row_ptrs, torch.int64, "idx_row_ptrs")
    S = idx_row_ptrs.numel()
    _check(n_rows, torch.int64, "n_rows", numel=S)
    _check(q_bf16, torch.bfloat16, "q_bf16", numel=S * 64 * 128)
    _check(w, torch.float32, "w", numel=S * 64)
    _check(out_idx, torch.int32, "out_idx", numel=S * int(k))
    _check(out_score, torch.float32, "out_score", numel=S * int(k), allow_none=True)
    _check(ws, torch.uint8, "ws")
    _call("ds4x_index_score_topk_batched", _ptr(idx_row_ptrs), _ptr(n_rows), S, _ptr(q_bf16), _ptr(w), int(k),
          _ptr(out_idx), _ptr(out_score), _ptr(ws), ws.numel(), _stream(stream))


def ds4x_sparse_attn_decode_batched(kv_row_ptrs, n_rows, idx, k, q_bf16, softmax_scale, out_bf16, lse, ws,
                                    stream=None):
    """Decode attention for a batch of sessions: kv_row_ptrs int64 [S] device
    row pointers, n_rows int64 [S], idx int32 [S, k], q_bf16 [S, 64, 512]."""
    _check(kv_row_ptrs, torch.int64, "kv_row_ptrs")
    S = kv_row_ptrs.numel()
    _check(n_rows, torch.int64, "n_rows", numel=S)
    _check(idx, torch.int32, "idx", numel=S * int(k))
    _check(q_bf16, torch.bfloat16, "q_bf16", numel=S * 64 * 512)
    _check(out_bf16, torch.bfloat16, "out_bf16", numel=S * 64 * 512)
    _check(lse, torch.float32, "lse", numel=S * 64, allow_none=True)
    _check(ws, torch.uint8, "ws")
    _call("ds4x_sparse_attn_decode_batched", _ptr(kv_row_ptrs), _ptr(n_rows), S, _ptr(idx), int(k), _ptr(q_bf16),
          float(softmax_scale), _ptr(out_bf16), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))


def ds4x_sparse_attn_prefill(kv_rows, n_rows, idx, n_queries, k, q_bf16, softmax_scale, out_bf16, lse, ws,
                             stream=None):
    """Per-query sparse attention of q_bf16 [T, 64, 512] over each query's k
    rows idx [T, k] of one cache."""
    _check(kv_rows, torch.uint8, "kv_rows", numel=int(n_rows) * 583)
    _check(idx, torch.int32, "idx", numel=int(n_queries) * int(k))
    _check(q_bf16, torch.bfloat16, "q_bf16", numel=int(n_queries) * 64 * 512)
    _check(out_bf16, torch.bfloat16, "out_bf16", numel=int(n_queries) * 64 * 512)
    _check(lse, torch.float32, "lse", numel=int(n_queries) * 64, allow_none=True)
    _check(ws, torch.uint8, "ws")
    _call("ds4x_sparse_attn_prefill", _ptr(kv_rows), int(n_rows), _ptr(idx), int(n_queries), int(k), _ptr(q_bf16),
          float(softmax_scale), _ptr(out_bf16), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))


def ds4x_quantize_query_e4m3(q, codes, scales, stream=None):
    """q f32 [..., 128] -> codes u8 [..., 128], scales u8 [..., 4]."""
    _check(q, torch.float32, "q")
    n = q.numel() // 128
    _check(codes, torch.uint8, "codes", numel=n * 128)
    _check(scales, torch.uint8, "scales", numel=n * 4)
    _call("ds4x_quantize_query_e4m3", _ptr(q), n, _ptr(codes), _ptr(scales), _stream(stream))


def ds4x_index_score_topk_prefill_workspace(n_rows: int, n_queries: int, k: int) -> int:
    return lib().ds4x_index_score_topk_prefill_workspace(int(n_rows), int(n_queries), int(k))


def ds4x_index_score_topk_prefill(idx_rows, n_rows, q_codes, q_scales, w, n_queries, causal_base, k, out_idx,
                                  out_score, ws, stream=None):
    """Per-query exact top-k for a chunk of prefill tokens (query i sees rows
    t < causal_base + i); q_codes u8 [T, 64, 128], q_scales u8 [T, 64, 4],
    w f32 [T, 64], out_idx int32 [T, k]."""
    T = int(n_queries)
    _check(idx_rows, torch.uint8, "idx_rows", numel=int(n_rows) * 68)
    _check(q_codes, torch.uint8, "q_codes", numel=T * 64 * 128)
    _check(q_scales, torch.uint8, "q_scales", numel=T * 64 * 4)
    _check(w, torch.float32, "w", numel=T * 64)
    _check(out_idx, torch.int32, "out_idx", numel=T * int(k))
    _check(out_score, torch.float32, "out_score", numel=T * int(k), allow_none=True)
    _check(ws, torch.uint8, "ws")
    _call("ds4x_index_score_topk_prefill", _ptr(idx_rows), int(n_rows), _ptr(q_codes), _ptr(q_scales), _ptr(w), T,
          int(causal_base), int(k), _ptr(out_idx), _ptr(out_score), _ptr(ws), ws.numel(), _stream(stream))
