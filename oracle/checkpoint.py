"""Packed-row checkpoints: an independent plain-Python writer and reader of
the byte layout ds4x.h specifies.  Test infrastructure only (see
``oracle/__init__``).

Disk checkpoints keep the native packed rows, and payload version 3 rejects
other versions such as the F32-cache version 2 (DS4X README, "Optimization
details"); the raw window's live rows go in logical order, oldest first
(ds4 README, "Disk KV Cache").  Layout: a 64-byte header ("DS4X", version,
header bytes, layer count, ring rows, KV and indexer row bytes, entry bytes,
total bytes, zeros), one 32-byte entry per layer (ratio, live window rows,
KV rows, indexer rows, zero), then each layer's window, KV and indexer rows.
"""

from __future__ import annotations

import struct

import numpy as np

RING, KV, IDX = 256, 583, 68
VERSION = 3


def window_logical(ring_rows, ring_pos, live):
    """The live window rows oldest first from a physical ring [256 * 583]."""
    ring = np.asarray(ring_rows, dtype=np.uint8).reshape(RING, KV)
    slots = [(ring_pos - live + 1 + j) % RING for j in range(live)]
    return ring[slots]


def write(layers) -> bytes:
    entries, rows = [], []
    for L in layers:
        live = int(L.get("ring_live", 0))
        kv = np.asarray(L.get("kv_rows", np.zeros(0, np.uint8)), dtype=np.uint8).reshape(-1)
        ix = np.asarray(L.get("idx_rows", np.zeros(0, np.uint8)), dtype=np.uint8).reshape(-1)
        entries.append(struct.pack("<IIQQQ", int(L["ratio"]), live, kv.size // KV, ix.size // IDX, 0))
        if live:
            rows.append(window_logical(L["ring_rows"], int(L["ring_pos"]), live).tobytes())
        rows.append(kv.tobytes())
        rows.append(ix.tobytes())
    body = b"".join(entries) + b"".join(rows)
    total = 64 + len(body)
    header = b"DS4X" + struct.pack("<IIIIIIIQ", VERSION, 64, len(layers), RING, KV, IDX, 32, total) + bytes(24)
    return header + body


def read(data: bytes):
    """Layers as dicts (window rows oldest first); ValueError on a bad file."""
    if len(data) < 64 or data[:4] != b"DS4X":
        raise ValueError("format")
    ver, hb, nl, ring, kvb, idxb, eb, total = struct.unpack_from("<IIIIIIIQ", data, 4)
    if ver != VERSION:
        raise ValueError("version")
    if (hb, ring, kvb, idxb, eb) != (64, RING, KV, IDX, 32) or any(data[40:64]) or total != len(data[:total]):
        raise ValueError("format")
    off, rows_off, layers = 64, 64 + 32 * nl, []
    for _ in range(nl):
        ratio, live, n_kv, n_idx, zero = struct.unpack_from("<IIQQQ", data, off)
        off += 32
        ok = zero == 0 and live <= RING and (
            (ratio == 0 and n_kv == 0 and n_idx == 0) or (ratio == 128 and n_idx == 0) or (ratio == 4 and n_idx == n_kv))
        if not ok:
            raise ValueError("format")
        w = np.frombuffer(data, np.uint8, live * KV, rows_off).reshape(live, KV)
        rows_off += live * KV
        k = np.frombuffer(data, np.uint8, n_kv * KV, rows_off).reshape(n_kv, KV)
        rows_off += n_kv * KV
        x = np.frombuffer(data, np.uint8, n_idx * IDX, rows_off).reshape(n_idx, IDX)
        rows_off += n_idx * IDX
        layers.append({"ratio": ratio, "window": w, "kv_rows": k, "idx_rows": x})
    if rows_off != total or len(data) < total:
        raise ValueError("format")
    return layers
