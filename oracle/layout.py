"""Row sizes and the persistent packed-cache allocation -- oracle.

Test infrastructure only (see ``oracle/__init__``).

DS4X README, "Packed cache ABI": a KV row is 448 E4M3 bytes + 64 FP16 RoPE
values + 7 UE8M0 scales = 583 bytes; an indexer row is 128 E2M1 values at two
per byte + 4 UE8M0 scales = 68 bytes.  For DeepSeek-V4-Flash the layers are
2 without compressed history, 21 CSA layers at ratio 4 (KV + indexer rows)
and 20 HCA layers at ratio 128 (KV rows only); with the 32-token prefill
chunk every one of the 43 layers also holds a 256-row raw ring.  The
persistent allocation for a context of L tokens is therefore

    43 * 256 * 583 + 21 * (L // 4 + 2) * (583 + 68) + 20 * (L // 128 + 2) * 583
"""

from __future__ import annotations

from .codecs import IDX_ROW_BYTES, KV_ROW_BYTES

N_LAYERS_WITH_RING = 43
RAW_RING_ROWS = 256
N_CSA_LAYERS = 21
CSA_RATIO = 4
N_HCA_LAYERS = 20
HCA_RATIO = 128


def raw_ring_bytes() -> int:
    return N_LAYERS_WITH_RING * RAW_RING_ROWS * KV_ROW_BYTES


def compressed_bytes(L: int) -> int:
    csa = N_CSA_LAYERS * (L // CSA_RATIO + 2) * (KV_ROW_BYTES + IDX_ROW_BYTES)
    hca = N_HCA_LAYERS * (L // HCA_RATIO + 2) * KV_ROW_BYTES
    return csa + hca


def kv_cache_bytes(L: int) -> int:
    """Total persistent packed KV + indexer bytes for a context of L tokens."""
    return raw_ring_bytes() + compressed_bytes(L)


def csa_rows(L: int) -> int:
    """Compressed rows one CSA layer holds for a context of L tokens."""
    return L // CSA_RATIO + 2
