"""Packed-row checkpoints (host code, no GPU): the layout at fixed offsets
for a hand-built one-layer file; the library against an independent Python
writer, byte for byte; round trips (window rows oldest first, wrapping past
ring slot 0); and the rejections: another magic, another payload version
(the F32-cache version 2), a truncated or corrupt file, inconsistent layers,
too little room."""

import struct

import numpy as np
import pytest

from oracle import checkpoint as K

EFORMAT, EVERSION, EINVAL, ERANGE = -8, -9, -1, -2


@pytest.fixture(scope="module")
def B():
    from compressed_kv_sparse_csa_gb300 import binding

    binding.lib()
    return binding


def _rows(rng, n, width):
    return rng.integers(0, 256, size=n * width, dtype=np.uint8)


def _layers(seed):
    rng = np.random.default_rng(seed)
    out = []
    for ratio in (0, 4, 128, 4, 128, 0):
        live = int(rng.choice([0, 1, 37, 256]))
        n = 0 if ratio == 0 else int(rng.integers(0, 40))
        out.append({"ratio": ratio, "ring_live": live, "ring_pos": int(rng.integers(0, 256)),
                    "ring_rows": _rows(rng, 256, 583), "kv_rows": _rows(rng, n, 583),
                    "idx_rows": _rows(rng, n if ratio == 4 else 0, 68)})
    return out


def test_layout_of_a_one_layer_file(B):
    rng = np.random.default_rng(1)
    ring, kv, ix = _rows(rng, 256, 583), _rows(rng, 1, 583), _rows(rng, 1, 68)
    data = B.ds4x_checkpoint_save([{"ratio": 4, "ring_live": 1, "ring_pos": 200, "ring_rows": ring,
                                    "kv_rows": kv, "idx_rows": ix}])
    total = 64 + 32 + 583 + 583 + 68
    assert len(data) == total
    assert data[0:4] == b"DS4X"
    assert struct.unpack_from("<IIIIIIIQ", data, 4) == (3, 64, 1, 256, 583, 68, 32, total)
    assert data[40:64] == bytes(24)
    assert struct.unpack_from("<IIQQQ", data, 64) == (4, 1, 1, 1, 0)
    assert data[96:96 + 583] == ring[200 * 583:201 * 583].tobytes()  # the one live row: slot ring_pos
    assert data[96 + 583:96 + 1166] == kv.tobytes()
    assert data[96 + 1166:] == ix.tobytes()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_library_matches_the_python_writer(B, seed):
    layers = _layers(seed)
    assert B.ds4x_checkpoint_save(layers) == K.write(layers)


def test_window_wraps_past_slot_zero(B):
    rng = np.random.default_rng(5)
    ring = _rows(rng, 256, 583)
    data = B.ds4x_checkpoint_save([{"ratio": 0, "ring_live": 10, "ring_pos": 3, "ring_rows": ring}])
    slots = [250, 251, 252, 253, 254, 255, 0, 1, 2, 3]  # oldest first
    want = ring.reshape(256, 583)[slots]
    got = np.frombuffer(data, np.uint8, 10 * 583, 96).reshape(10, 583)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("seed", [3, 4])
def test_round_trip(B, seed):
    layers = _layers(seed)
    data = B.ds4x_checkpoint_save(layers)
    counts = B.ds4x_checkpoint_inspect(data)
    assert [(c["ratio"], c["ring_live"], c["n_kv"], c["n_idx"]) for c in counts] == [
        (L["ratio"], L["ring_live"], L["kv_rows"].size // 583, L["idx_rows"].size // 68) for L in layers]
    bufs = [{"ring_rows": np.zeros(256 * 583, np.uint8), "kv_rows": np.zeros(64 * 583, np.uint8),
             "idx_rows": np.zeros(64 * 68, np.uint8)} for _ in layers]
    B.ds4x_checkpoint_load(data, bufs)
    for L, b in zip(layers, bufs):
        live = L["ring_live"]
        assert np.array_equal(b["ring_rows"].reshape(256, 583)[:live],
                              K.window_logical(L["ring_rows"], L["ring_pos"], live))
        assert np.array_equal(b["kv_rows"][:L["kv_rows"].size], L["kv_rows"])
        assert np.array_equal(b["idx_rows"][:L["idx_rows"].size], L["idx_rows"])
    # the Python reader sees the same rows
    for L, r in zip(layers, K.read(data)):
        assert np.array_equal(r["kv_rows"].reshape(-1), L["kv_rows"])


def _status(B, data):
    try:
        B.ds4x_checkpoint_inspect(data)
        return 0
    except B.Ds4xError as e:
        return e.status


def _corrupt(data, off, fmt, value):
    b = bytearray(data)
    struct.pack_into(fmt, b, off, value)
    return bytes(b)


def test_rejections(B):
    data = B.ds4x_checkpoint_save(_layers(7))
    assert _status(B, data) == 0
    cases = [
        (b"DS4V" + data[4:], EFORMAT),                    # another magic
        (_corrupt(data, 4, "<I", 2), EVERSION),           # the F32-cache payload version
        (_corrupt(data, 4, "<I", 4), EVERSION),
        (data[:-1], EFORMAT),                             # truncated
        (data[:63], EFORMAT),
        (_corrupt(data, 32, "<Q", len(data) + 1), EFORMAT),  # total bytes
        (_corrupt(data, 20, "<I", 584), EFORMAT),         # KV row bytes
        (_corrupt(data, 16, "<I", 128), EFORMAT),         # ring rows
        (_corrupt(data, 50, "<B", 1), EFORMAT),           # reserved header bytes
        (_corrupt(data, 64, "<I", 7), EFORMAT),           # ratio of layer 0
        (_corrupt(data, 64 + 4, "<I", 257), EFORMAT),     # live window rows
        (_corrupt(data, 64 + 24, "<Q", 1), EFORMAT),      # entry's zero field
    ]
    for bad, status in cases:
        assert _status(B, bad) == status
        with pytest.raises(ValueError):
            K.read(bad)


def test_bad_layers_and_room(B):
    rng = np.random.default_rng(9)
    kv, ix = _rows(rng, 3, 583), _rows(rng, 2, 68)
    with pytest.raises(B.Ds4xError) as e:  # CSA rows without as many indexer rows
        B.ds4x_checkpoint_save([{"ratio": 4, "kv_rows": kv, "idx_rows": ix}])
    assert e.value.status == EINVAL
    with pytest.raises(B.Ds4xError) as e:  # HCA layers carry no indexer rows
        B.ds4x_checkpoint_save([{"ratio": 128, "kv_rows": kv, "idx_rows": _rows(rng, 3, 68)}])
    assert e.value.status == EINVAL
    data = B.ds4x_checkpoint_save([{"ratio": 128, "kv_rows": kv}])
    with pytest.raises(B.Ds4xError) as e:  # room for 2 KV rows, 3 stored
        B.ds4x_checkpoint_load(data, [{"kv_rows": np.zeros(2 * 583, np.uint8)}])
    assert e.value.status == ERANGE
    with pytest.raises(B.Ds4xError) as e:  # the file holds one layer
        B.ds4x_checkpoint_load(data, [{"kv_rows": np.zeros(3 * 583, np.uint8)}] * 2)
    assert e.value.status == EINVAL
