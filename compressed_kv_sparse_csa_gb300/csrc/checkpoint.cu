// Packed-row checkpoints of the path's per-layer state (host code only).
//
// Disk checkpoints store the native packed rows, and the payload ABI version
// (3) rejects payloads of any other version, such as the F32-cache version 2
// (DS4X README, "Optimization details"); the raw sliding-window rows are
// stored in logical position order rather than physical ring order (ds4
// README, "Disk KV Cache").  The byte layout is this library's own and is
// specified next to the entry points in ds4x.h.
#include <cstring>

#include "ds4x_internal.cuh"

namespace {

constexpr uint32_t kMagic = 0x58345344u;  // "DS4X", little-endian
constexpr uint32_t kVersion = 3;
constexpr uint32_t kHeaderBytes = 64;
constexpr uint32_t kEntryBytes = 32;

void put_u32(uint8_t *p, uint32_t v) {
  for (int i = 0; i < 4; ++i) p[i] = uint8_t(v >> (8 * i));
}
void put_u64(uint8_t *p, uint64_t v) {
  for (int i = 0; i < 8; ++i) p[i] = uint8_t(v >> (8 * i));
}
uint32_t get_u32(const uint8_t *p) {
  uint32_t v = 0;
  for (int i = 0; i < 4; ++i) v |= uint32_t(p[i]) << (8 * i);
  return v;
}
uint64_t get_u64(const uint8_t *p) {
  uint64_t v = 0;
  for (int i = 0; i < 8; ++i) v |= uint64_t(p[i]) << (8 * i);
  return v;
}

// Rows of a layer kind: ratio 0 keeps only the raw window, 128 (HCA) KV rows,
// 4 (CSA) KV rows and as many indexer rows.
bool counts_ok(int64_t ratio, int64_t live, int64_t n_kv, int64_t n_idx) {
  if (live < 0 || live > DS4X_RING_ROWS || n_kv < 0 || n_idx < 0) return false;
  if (ratio == 0) return n_kv == 0 && n_idx == 0;
  if (ratio == 128) return n_idx == 0;
  if (ratio == 4) return n_idx == n_kv;
  return false;
}

// Bytes of a layer's rows; -1 past the int64 range.
int64_t layer_bytes(int64_t live, int64_t n_kv, int64_t n_idx) {
  const int64_t lim = INT64_MAX / 2 / DS4X_KV_ROW_BYTES;
  if (n_kv > lim || n_idx > lim) return -1;
  return (live + n_kv) * DS4X_KV_ROW_BYTES + n_idx * DS4X_IDX_ROW_BYTES;
}

// The whole file's size from its layer table, or a negative status.
int64_t table_total(const uint8_t *table, int32_t n_layers) {
  int64_t total = int64_t(kHeaderBytes) + int64_t(kEntryBytes) * n_layers;
  for (int32_t l = 0; l < n_layers; ++l) {
    const uint8_t *e = table + size_t(l) * kEntryBytes;
    const int64_t ratio = get_u32(e), live = get_u32(e + 4);
    const uint64_t n_kv = get_u64(e + 8), n_idx = get_u64(e + 16), zero = get_u64(e + 24);
    if (zero != 0 || n_kv > uint64_t(INT64_MAX) || n_idx > uint64_t(INT64_MAX)) return DS4X_EFORMAT;
    if (!counts_ok(ratio, live, int64_t(n_kv), int64_t(n_idx))) return DS4X_EFORMAT;
    const int64_t b = layer_bytes(live, int64_t(n_kv), int64_t(n_idx));
    if (b < 0 || total > INT64_MAX - b) return DS4X_EFORMAT;
    total += b;
  }
  return total;
}

// Checks the header and the table of src; returns the layer count or a
// negative status.
int64_t check_file(const uint8_t *src, int64_t src_bytes) {
  if (src == nullptr || src_bytes < int64_t(kHeaderBytes)) return DS4X_EFORMAT;
  if (get_u32(src) != kMagic) return DS4X_EFORMAT;
  if (get_u32(src + 4) != kVersion) return DS4X_EVERSION;
  if (get_u32(src + 8) != kHeaderBytes || get_u32(src + 16) != DS4X_RING_ROWS ||
      get_u32(src + 20) != DS4X_KV_ROW_BYTES || get_u32(src + 24) != DS4X_IDX_ROW_BYTES ||
      get_u32(src + 28) != kEntryBytes)
    return DS4X_EFORMAT;
  for (int i = 40; i < int(kHeaderBytes); ++i)
    if (src[i] != 0) return DS4X_EFORMAT;
  const uint32_t n_layers = get_u32(src + 12);
  if (n_layers > uint32_t(DS4X_CHECKPOINT_MAX_LAYERS)) return DS4X_EFORMAT;
  if (src_bytes < int64_t(kHeaderBytes) + int64_t(kEntryBytes) * n_layers) return DS4X_EFORMAT;
  const int64_t total = table_total(src + kHeaderBytes, int32_t(n_layers));
  if (total < 0) return total;
  if (int64_t(get_u64(src + 32)) != total || src_bytes < total) return DS4X_EFORMAT;
  return n_layers;
}

}  // namespace

extern "C" {

int64_t ds4x_checkpoint_bytes(const ds4x_layer_rows *layers, int32_t n_layers) {
  if (n_layers < 0 || n_layers > DS4X_CHECKPOINT_MAX_LAYERS || (n_layers > 0 && layers == nullptr)) return DS4X_EINVAL;
  int64_t total = int64_t(kHeaderBytes) + int64_t(kEntryBytes) * n_layers;
  for (int32_t l = 0; l < n_layers; ++l) {
    const ds4x_layer_rows &x = layers[l];
    if (!counts_ok(x.ratio, x.ring_live, x.n_kv, x.n_idx)) return DS4X_EINVAL;
    if ((x.ring_live > 0 && (x.ring_rows == nullptr || x.ring_pos < 0 || x.ring_pos >= DS4X_RING_ROWS)) ||
        (x.n_kv > 0 && x.kv_rows == nullptr) || (x.n_idx > 0 && x.idx_rows == nullptr))
      return DS4X_EINVAL;
    const int64_t b = layer_bytes(x.ring_live, x.n_kv, x.n_idx);
    if (b < 0 || total > INT64_MAX - b) return DS4X_EINVAL;
    total += b;
  }
  return total;
}

int ds4x_checkpoint_save(const ds4x_layer_rows *layers, int32_t n_layers, uint8_t *dst, int64_t dst_bytes) {
  const int64_t total = ds4x_checkpoint_bytes(layers, n_layers);
  if (total < 0) return int(total);
  if (dst == nullptr) return DS4X_EINVAL;
  if (dst_bytes < total) return DS4X_ERANGE;
  std::memset(dst, 0, size_t(kHeaderBytes) + size_t(kEntryBytes) * size_t(n_layers));
  put_u32(dst, kMagic);
  put_u32(dst + 4, kVersion);
  put_u32(dst + 8, kHeaderBytes);
  put_u32(dst + 12, uint32_t(n_layers));
  put_u32(dst + 16, DS4X_RING_ROWS);
  put_u32(dst + 20, DS4X_KV_ROW_BYTES);
  put_u32(dst + 24, DS4X_IDX_ROW_BYTES);
  put_u32(dst + 28, kEntryBytes);
  put_u64(dst + 32, uint64_t(total));
  uint8_t *rows = dst + kHeaderBytes + size_t(kEntryBytes) * n_layers;
  for (int32_t l = 0; l < n_layers; ++l) {
    const ds4x_layer_rows &x = layers[l];
    uint8_t *e = dst + kHeaderBytes + size_t(l) * kEntryBytes;
    put_u32(e, uint32_t(x.ratio));
    put_u32(e + 4, uint32_t(x.ring_live));
    put_u64(e + 8, uint64_t(x.n_kv));
    put_u64(e + 16, uint64_t(x.n_idx));
    // the window oldest first: slots ring_pos - live + 1 .. ring_pos (mod the ring)
    for (int32_t j = 0; j < x.ring_live; ++j) {
      const int32_t slot = (x.ring_pos - x.ring_live + 1 + j + 2 * DS4X_RING_ROWS) % DS4X_RING_ROWS;
      std::memcpy(rows, x.ring_rows + size_t(slot) * DS4X_KV_ROW_BYTES, DS4X_KV_ROW_BYTES);
      rows += DS4X_KV_ROW_BYTES;
    }
    if (x.n_kv > 0) std::memcpy(rows, x.kv_rows, size_t(x.n_kv) * DS4X_KV_ROW_BYTES);
    rows += size_t(x.n_kv) * DS4X_KV_ROW_BYTES;
    if (x.n_idx > 0) std::memcpy(rows, x.idx_rows, size_t(x.n_idx) * DS4X_IDX_ROW_BYTES);
    rows += size_t(x.n_idx) * DS4X_IDX_ROW_BYTES;
  }
  return DS4X_OK;
}

int ds4x_checkpoint_inspect(const uint8_t *src, int64_t src_bytes, int32_t *n_layers, ds4x_layer_counts *counts,
                            int32_t counts_cap) {
  if (n_layers == nullptr) return DS4X_EINVAL;
  const int64_t nl = check_file(src, src_bytes);
  if (nl < 0) return int(nl);
  *n_layers = int32_t(nl);
  if (counts != nullptr) {
    if (counts_cap < nl) return DS4X_ERANGE;
    for (int64_t l = 0; l < nl; ++l) {
      const uint8_t *e = src + kHeaderBytes + size_t(l) * kEntryBytes;
      counts[l].ratio = int32_t(get_u32(e));
      counts[l].ring_live = int32_t(get_u32(e + 4));
      counts[l].n_kv = int64_t(get_u64(e + 8));
      counts[l].n_idx = int64_t(get_u64(e + 16));
    }
  }
  return DS4X_OK;
}

int ds4x_checkpoint_load(const uint8_t *src, int64_t src_bytes, const ds4x_layer_buffers *bufs, int32_t n_layers) {
  const int64_t nl = check_file(src, src_bytes);
  if (nl < 0) return int(nl);
  if (n_layers != nl || (nl > 0 && bufs == nullptr)) return DS4X_EINVAL;
  // check every destination before writing any
  for (int64_t l = 0; l < nl; ++l) {
    const uint8_t *e = src + kHeaderBytes + size_t(l) * kEntryBytes;
    const int64_t live = get_u32(e + 4), n_kv = int64_t(get_u64(e + 8)), n_idx = int64_t(get_u64(e + 16));
    const ds4x_layer_buffers &b = bufs[l];
    if ((live > 0 && b.ring_rows == nullptr) || (n_kv > 0 && b.kv_rows == nullptr) ||
        (n_idx > 0 && b.idx_rows == nullptr))
      return DS4X_EINVAL;
    if (n_kv > b.kv_cap || n_idx > b.idx_cap) return DS4X_ERANGE;
  }
  const uint8_t *rows = src + kHeaderBytes + size_t(kEntryBytes) * nl;
  for (int64_t l = 0; l < nl; ++l) {
    const uint8_t *e = src + kHeaderBytes + size_t(l) * kEntryBytes;
    const int64_t live = get_u32(e + 4), n_kv = int64_t(get_u64(e + 8)), n_idx = int64_t(get_u64(e + 16));
    const ds4x_layer_buffers &b = bufs[l];
    if (live > 0) std::memcpy(b.ring_rows, rows, size_t(live) * DS4X_KV_ROW_BYTES);  // slots 0 .. live - 1
    rows += size_t(live) * DS4X_KV_ROW_BYTES;
    if (n_kv > 0) std::memcpy(b.kv_rows, rows, size_t(n_kv) * DS4X_KV_ROW_BYTES);
    rows += size_t(n_kv) * DS4X_KV_ROW_BYTES;
    if (n_idx > 0) std::memcpy(b.idx_rows, rows, size_t(n_idx) * DS4X_IDX_ROW_BYTES);
    rows += size_t(n_idx) * DS4X_IDX_ROW_BYTES;
  }
  return DS4X_OK;
}

}  // extern "C"
