/*
 * ds4x.h -- C ABI of the GB300 (sm_103a) compressed-KV sparse-attention
 * (CSA) decode path.
 *
 * The path (DS4X README, "What DS4X changes" and "Optimization details"):
 *   1. a CSA indexer scores every compressed history row, reading packed
 *      68-byte MXFP4 rows directly;
 *   2. an exact top-k (k <= 512) picks rows under the float total order of
 *      the score with the lower row index winning ties;
 *   3. sparse attention runs over the selected 583-byte packed KV rows.
 * A cache writer quantises and packs new rows into both formats.
 *
 * Row formats (DS4X README, "Packed cache ABI"):
 *   KV row (583 B)      = 448 E4M3FN codes (element order)
 *                       + 64 FP16 RoPE values, little-endian (128 B)
 *                       + 7 UE8M0 scales, one per 64-value non-RoPE block
 *   indexer row (68 B)  = 128 E2M1 codes, two per byte, even element in the
 *                         low nibble (64 B)
 *                       + 4 UE8M0 scales, one per 32-value block
 *   A UE8M0 byte b stands for 2^(b - 127).  Row i of an array of n rows
 *   starts at byte i * 583 (KV) or i * 68 (indexer); arrays are contiguous.
 *
 * Conventions for every entry point below:
 *   - Every pointer is a DEVICE pointer unless stated otherwise, and must be
 *     16-byte aligned.  The caller owns all memory (rows, inputs, outputs and
 *     workspace); the library allocates nothing.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) and never synchronise it.
 *   - Calls return DS4X_OK (0) or a negative status.  Arguments are checked
 *     on the host before anything is launched; a failed check launches
 *     nothing and leaves every buffer untouched.  DS4X_ECUDA reports a
 *     launch failure (the CUDA error is left for cudaGetLastError to read).
 *     No call traps, asserts or throws across the ABI.
 *   - Inputs must be finite; NaN or infinite inputs give unspecified (but
 *     memory-safe) results.
 *   - bfloat16 data is passed as uint16_t bit patterns.
 *   - The library runs only on compute capability 10.3 (GB300);
 *     anything else returns DS4X_EARCH.
 */
#ifndef DS4X_H
#define DS4X_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Identical to cudaStream_t. */
typedef struct CUstream_st *ds4x_stream_t;

#define DS4X_ABI_VERSION 1

#define DS4X_KV_ROW_BYTES 583
#define DS4X_KV_DIM 512
#define DS4X_KV_NOPE 448
#define DS4X_KV_ROPE 64
#define DS4X_KV_BLOCK 64
#define DS4X_IDX_ROW_BYTES 68
#define DS4X_IDX_DIM 128
#define DS4X_IDX_BLOCK 32
#define DS4X_IDX_HEADS 64
#define DS4X_ATTN_HEADS 64
#define DS4X_TOPK_MAX 512
#define DS4X_MAX_SESSIONS 64
#define DS4X_PREFILL_MAX_QUERIES 65535
#define DS4X_DENSE_MAX_ROWS (8192LL * 512)
#define DS4X_RING_ROWS 256
#define DS4X_CHECKPOINT_MAX_LAYERS 4096

enum {
  DS4X_OK = 0,
  DS4X_EINVAL = -1,     /* null or misaligned pointer, bad size or k      */
  DS4X_ERANGE = -2,     /* pos / n outside the cache capacity              */
  DS4X_EWORKSPACE = -3, /* workspace smaller than the *_workspace() size   */
  DS4X_EARCH = -4,      /* current device is not compute capability 10.3   */
  DS4X_ECUDA = -5,      /* a CUDA runtime call or launch failed            */
  DS4X_ETIMEOUT = -6,   /* device status: a bounded wait gave up           */
  DS4X_EDEVICE = -7,    /* device status: kernel-detected bad input        */
  DS4X_EFORMAT = -8,    /* not a checkpoint of this layout, or corrupt     */
  DS4X_EVERSION = -9    /* a checkpoint of another payload version         */
};

/* Static text for a status code (host pointer, never NULL). */
const char *ds4x_status_str(int status);

/* DS4X_ABI_VERSION of the built library. */
int ds4x_abi_version(void);

/*
 * Persistent packed KV + indexer bytes a DeepSeek-V4-Flash context of
 * `context_tokens` tokens needs (DS4X README, "Packed cache ABI": 43 layers
 * with a 256-row raw ring, 21 CSA layers at ratio 4 holding KV and indexer
 * rows, 20 HCA layers at ratio 128 holding KV rows):
 *   43*256*583 + 21*(L/4 + 2)*(583 + 68) + 20*(L/128 + 2)*583.
 * Host-only arithmetic.  Returns -1 for a negative argument.
 */
int64_t ds4x_cache_bytes(int64_t context_tokens);

/*
 * Zero-fills a workspace before its first use (cudaMemsetAsync on
 * `stream`).  Every workspace passed to ds4x_index_score_topk or
 * ds4x_sparse_attn_decode must have been zero-filled once, by this call or
 * otherwise; each call leaves it ready for the next call on the same
 * stream.  One workspace must not be used by two calls that may overlap on
 * the GPU.
 *
 * Bytes 12..15 of a scorer workspace (ds4x_index_score_topk and its batched
 * and prefill forms) hold a u32: the arrivals its CTA exchange waits for
 * beyond the CTAs of the session.  It is 0 in normal use.  A nonzero value
 * makes the exchange's bounded wait run out (every CTA gives up after 0.5 s,
 * writes no output and sets DS4X_ETIMEOUT): it exists to test the time-out
 * path.  After a call that set DS4X_ETIMEOUT the workspace must be
 * zero-filled again before its next use.
 */
int ds4x_workspace_init(void *ws, size_t ws_bytes, ds4x_stream_t stream);

/*
 * Copies `bytes` bytes from src to dst with a kernel on `stream` (16-byte
 * words, the tail byte by byte).  Either pointer may be device memory or
 * page-locked host memory the GPU can address (cudaHostAlloc / pinned
 * memory under unified addressing): a decode loop that keeps a step's inputs
 * and results in pinned host memory moves them with this call inside its
 * CUDA graph, instead of copy-engine copies whose hand-over to and from the
 * kernels costs several microseconds each.  The pages have no counterpart
 * to it.  dst and src 16-byte aligned and not overlapping; bytes may be 0
 * (nothing is launched).  Asynchronous; the caller keeps both buffers alive
 * until the stream has passed the copy.  Errors: DS4X_EINVAL.
 */
int ds4x_copy_async(void *dst, const void *src, size_t bytes, ds4x_stream_t stream);

/*
 * Reads the device status word at the head of a workspace (a blocking copy
 * after synchronising `stream`) into *status_host and clears it.  It is
 * DS4X_OK, or DS4X_EDEVICE when an attention call met an index outside
 * [-1, n_rows) (that row was skipped), or DS4X_ETIMEOUT when a bounded wait
 * inside the scorer gave up.  Returns DS4X_OK or DS4X_ECUDA.
 */
int ds4x_workspace_status(void *ws, ds4x_stream_t stream, int32_t *status_host);

/*
 * Cache writer: quantise and pack n new rows into positions [pos, pos+n).
 * (DS4X README, "What DS4X changes": persistent history is kept as packed
 * 583-byte KV rows and 68-byte MXFP4 indexer rows.)
 *
 *   kv_rows   u8 [capacity][583]  written at rows pos..pos+n-1; may be NULL
 *   idx_rows  u8 [capacity][68]   written at rows pos..pos+n-1; may be NULL
 *             (not both NULL; a layer without an indexer passes NULL)
 *   kv_in     f32 [n][512]: 448 non-RoPE values then 64 RoPE values
 *             (required when kv_rows != NULL)
 *   idx_in    f32 [n][128] (required when idx_rows != NULL)
 *
 * Each 32-value indexer block and 64-value KV block gets the scale 2^e with
 * e the least integer such that amax <= emax * 2^e (emax = 6 for E2M1, 448
 * for E4M3; amax = 0 gives e = 0; e clamped to [-127, 127]); elements are
 * x / 2^e rounded to nearest, ties to even, sign kept; RoPE values are
 * rounded to FP16 (nearest even).  Output bytes are bit-exact with that
 * rule.  Errors: DS4X_EINVAL (pointers, n < 1), DS4X_ERANGE (pos < 0 or
 * pos + n > capacity).
 */
int ds4x_cache_append(uint8_t *kv_rows, uint8_t *idx_rows, int64_t capacity, int64_t pos,
                      const float *kv_in, const float *idx_in, int64_t n,
                      ds4x_stream_t stream);

/* Workspace bytes ds4x_index_score_topk needs for n_rows rows and k. */
size_t ds4x_index_score_topk_workspace(int64_t n_rows, int32_t k);

/*
 * CSA indexer score + exact top-k over n_rows packed indexer rows.
 * (DS4X README, "Optimization details": the B1 indexer reads the 68-byte
 * rows directly; "CSA score/top-512 fusion": each scorer CTA keeps an exact
 * local top-512 of sortable (score, index) keys and merges them, so the
 * full score array is never materialised; float total order, lower index
 * wins ties.)
 *
 *   s_t = sum_{h<64} w[h] * max(0, sum_{j<128} q[h][j] * k_t[j])
 *
 *   idx_rows   u8 [n_rows][68]
 *   q_bf16     bf16 [64][128] indexer query
 *   w          f32 [64] head weights
 *   k          1..512
 *   out_idx    i32 [k]: row indices, score descending then index
 *              ascending; entries past n_rows are -1
 *   out_score  f32 [k] or NULL: the scores (fp32 accumulation), NaN past
 *              n_rows
 *   ws         workspace of >= ds4x_index_score_topk_workspace(n_rows, k)
 *              bytes, zero-filled before first use (ds4x_workspace_init)
 *
 * Errors: DS4X_EINVAL (pointers, n_rows < 1, k outside 1..512),
 * DS4X_EWORKSPACE.
 */
int ds4x_index_score_topk(const uint8_t *idx_rows, int64_t n_rows, const uint16_t *q_bf16,
                          const float *w, int32_t k, int32_t *out_idx, float *out_score,
                          void *ws, size_t ws_bytes, ds4x_stream_t stream);

/* Workspace bytes ds4x_sparse_attn_decode needs for k selected rows. */
size_t ds4x_sparse_attn_decode_workspace(int32_t k);

/*
 * Sparse (indexed) decode attention over selected packed KV rows, split
 * over row ranges with a log-sum-exp combine (one kernel: the splits of a
 * head group form a thread-block cluster and combine in shared memory).  (DS4X README, "Packed cache
 * ABI" row layout; "Nsight Systems" lists the indexed attention kernel
 * group.)  Keys and values are the same dequantised 512-vector (448
 * E4M3 * 2^(scale-127) values then 64 FP16 values), shared by all 64 heads:
 *
 *   l_hj = softmax_scale * (q_h . v_j);  p = softmax_j(l);  o_h = sum_j p_hj v_j
 *
 *   kv_rows        u8 [n_rows][583]
 *   idx            i32 [k]: row indices; -1 entries are skipped; entries
 *                  >= n_rows or < -1 are skipped and flag DS4X_EDEVICE in
 *                  the workspace status word
 *   k              1..512
 *   q_bf16         bf16 [64][512]
 *   out_bf16       bf16 [64][512] (rounded to nearest even; all-skipped
 *                  heads give 0)
 *   lse            f32 [64] or NULL: max_j l_hj + log(sum_j exp(l_hj - max))
 *                  (-inf when every row was skipped)
 *   ws             >= ds4x_sparse_attn_decode_workspace(k) bytes, zero-filled
 *                  before first use
 *
 * Errors: DS4X_EINVAL (pointers, n_rows < 1, k outside 1..512),
 * DS4X_EWORKSPACE.
 */
int ds4x_sparse_attn_decode(const uint8_t *kv_rows, int64_t n_rows, const int32_t *idx,
                            int32_t k, const uint16_t *q_bf16, float softmax_scale,
                            uint16_t *out_bf16, float *lse, void *ws, size_t ws_bytes,
                            ds4x_stream_t stream);

/*
 * One decode step of a CSA layer in one call: ds4x_index_score_topk
 * followed by ds4x_sparse_attn_decode over the k rows it selected, on one
 * stream, with one workspace (the attention is launched as a programmatic
 * dependent of the scorer, as when the two are called in turn).  The results
 * are exactly those of the two calls (out_idx / out_score as the scorer's,
 * out_bf16 / lse as the attention's).
 *
 *   idx_rows, n_rows, q_idx_bf16, w, k, out_idx, out_score  as ds4x_index_score_topk
 *   kv_rows, q_attn_bf16, softmax_scale, out_bf16, lse      as ds4x_sparse_attn_decode
 *   ws         >= ds4x_csa_decode_step_workspace(n_rows, k) bytes, zero-filled
 *              before first use; its status word covers both kernels
 *
 * Errors: DS4X_EINVAL (pointers, n_rows < 1, k outside 1..512),
 * DS4X_EWORKSPACE, DS4X_EARCH, DS4X_ECUDA.
 */
size_t ds4x_csa_decode_step_workspace(int64_t n_rows, int32_t k);
int ds4x_csa_decode_step(const uint8_t *idx_rows, const uint8_t *kv_rows, int64_t n_rows, const uint16_t *q_idx_bf16,
                         const float *w, int32_t k, const uint16_t *q_attn_bf16, float softmax_scale,
                         int32_t *out_idx, float *out_score, uint16_t *out_bf16, float *lse, void *ws,
                         size_t ws_bytes, ds4x_stream_t stream);

/*
 * Micro-batched decode: the CSA indexer score + exact top-k of n_sess
 * independent sessions in one launch (the sessions' CTAs are split in
 * proportion to their history lengths; each session is merged by the last
 * of its CTAs).  Per session exactly ds4x_index_score_topk.
 *
 *   idx_rows   device array of n_sess device pointers, session s: u8 [n_rows[s]][68]
 *   n_rows     device array i64 [n_sess] (a session with n_rows <= 0 gets -1 indices)
 *   n_sess     1..DS4X_MAX_SESSIONS
 *   q_bf16     bf16 [n_sess][64][128]
 *   w          f32 [n_sess][64]
 *   k          1..512
 *   out_idx    i32 [n_sess][k], each row as ds4x_index_score_topk's out_idx
 *   out_score  f32 [n_sess][k] or NULL
 *   ws         >= ds4x_index_score_topk_batched_workspace(n_sess, k) bytes,
 *              zero-filled before first use
 *
 * Errors: DS4X_EINVAL (pointers, n_sess or k out of range), DS4X_EWORKSPACE.
 */
size_t ds4x_index_score_topk_batched_workspace(int32_t n_sess, int32_t k);
int ds4x_index_score_topk_batched(const uint8_t *const *idx_rows, const int64_t *n_rows, int32_t n_sess,
                                  const uint16_t *q_bf16, const float *w, int32_t k, int32_t *out_idx,
                                  float *out_score, void *ws, size_t ws_bytes, ds4x_stream_t stream);

/*
 * Micro-batched decode attention: ds4x_sparse_attn_decode for n_sess
 * independent sessions in one launch (grid dimension z = session).
 *
 *   kv_rows    device array of n_sess device pointers, session s: u8 [n_rows[s]][583]
 *   n_rows     device array i64 [n_sess]
 *   idx        i32 [n_sess][k]
 *   q_bf16     bf16 [n_sess][64][512]
 *   out_bf16   bf16 [n_sess][64][512]
 *   lse        f32 [n_sess][64] or NULL
 *   ws         >= ds4x_sparse_attn_decode_workspace(k) bytes, zero-filled
 *              before first use (its status word covers every session)
 *
 * Errors: DS4X_EINVAL (pointers, n_sess or k out of range), DS4X_EWORKSPACE.
 */
int ds4x_sparse_attn_decode_batched(const uint8_t *const *kv_rows, const int64_t *n_rows, int32_t n_sess,
                                    const int32_t *idx, int32_t k, const uint16_t *q_bf16, float softmax_scale,
                                    uint16_t *out_bf16, float *lse, void *ws, size_t ws_bytes,
                                    ds4x_stream_t stream);

/*
 * Query quantiser for the chunked-prefill scorer: each 128-value vector (one
 * token, one head) becomes 128 E4M3 codes with one UE8M0 scale per 32 values
 * (least e with amax <= 448 * 2^e, amax = 0 giving e = 0, e clamped to
 * [-127, 127]; x / 2^e rounded to nearest, ties to even, sign kept).
 *
 *   q          f32 [n_vec128][128]
 *   codes      u8 [n_vec128][128]
 *   scales     u8 [n_vec128][4]
 *
 * Output bytes are bit-exact with that rule.  Errors: DS4X_EINVAL.
 */
int ds4x_quantize_query_e4m3(const float *q, int64_t n_vec128, uint8_t *codes, uint8_t *scales,
                              ds4x_stream_t stream);

/*
 * Chunked-prefill CSA score + per-query exact top-k (DS4X README, "Packed
 * prefill implementation": batch score/top-k over the packed indexer rows).
 * Query token i (0..n_queries-1) sees rows t < causal_base + i:
 *
 *   s_it = sum_h w[i][h] * max(0, q^[i][h] . k_t),  q^ = E4M3 code * 2^(scale-127)
 *
 * and gets the exact top-k of its visible rows (score descending, lower
 * index first; -1 / NaN past its visible count).  Runs as launches of up to
 * 2 x (SM count) query tokens: a tensor-core contraction that streams the
 * key tiles once per pair of tokens (one block-scaled MMA over both tokens'
 * 64 heads) and writes their fp32 scores into the workspace, then one
 * exact top-k per token over those scores.
 *
 *   idx_rows   u8 [n_rows][68]
 *   q_codes    u8 [n_queries][64][128], q_scales u8 [n_queries][64][4]
 *              (ds4x_quantize_query_e4m3; any scale byte 0..254)
 *   w          f32 [n_queries][64]
 *   out_idx    i32 [n_queries][k]; out_score f32 [n_queries][k] or NULL
 *   ws         >= ds4x_index_score_topk_prefill_workspace(n_rows, n_queries, k)
 *              bytes (the 256-byte status header, then the fp32 scores of
 *              up to 512 tokens over n_rows rows), zero-filled before first use
 *
 * Errors: DS4X_EINVAL (pointers, sizes, k), DS4X_EWORKSPACE.
 */
size_t ds4x_index_score_topk_prefill_workspace(int64_t n_rows, int32_t n_queries, int32_t k);
int ds4x_index_score_topk_prefill(const uint8_t *idx_rows, int64_t n_rows, const uint8_t *q_codes,
                                  const uint8_t *q_scales, const float *w, int32_t n_queries, int64_t causal_base,
                                  int32_t k, int32_t *out_idx, float *out_score, void *ws, size_t ws_bytes,
                                  ds4x_stream_t stream);

/*
 * Prefill sparse attention: each of n_queries query tokens attends over its
 * own k selected rows of one packed KV cache (DS4X README, "Packed prefill
 * implementation": per-token sparse attention after the batched score/top-k).
 * Per query the attention of ds4x_sparse_attn_decode (the same skip and
 * DS4X_EDEVICE rules, zeros and -inf for a query with no valid row), computed
 * with tcgen05 fp16 products over 128-row tiles: each non-RoPE value enters as
 * fp16 relative to the largest scale of its block over the query's rows, so
 * it is exact while the query's rows' scales of a block lie within 2^15 of
 * each other (beyond, a value rounds at 2^-24 of that block's largest scale);
 * the query enters exactly, the softmax weights with 22 significant bits, sums
 * in fp32.  One persistent CTA per SM takes the queries in turn.
 *
 *   kv_rows    u8 [n_rows][583]
 *   idx        i32 [n_queries][k]
 *   n_queries  1..DS4X_PREFILL_MAX_QUERIES
 *   q_bf16     bf16 [n_queries][64][512]
 *   out_bf16   bf16 [n_queries][64][512]
 *   lse        f32 [n_queries][64] or NULL
 *   ws         >= ds4x_sparse_attn_decode_workspace(k) bytes, zero-filled
 *
 * Errors: DS4X_EINVAL (pointers, sizes, k out of range), DS4X_EWORKSPACE.
 */
int ds4x_sparse_attn_prefill(const uint8_t *kv_rows, int64_t n_rows, const int32_t *idx, int32_t n_queries,
                             int32_t k, const uint16_t *q_bf16, float softmax_scale, uint16_t *out_bf16,
                             float *lse, void *ws, size_t ws_bytes, ds4x_stream_t stream);

/*
 * Allocation-free form of ds4x_sparse_attn_decode, for callers that cannot
 * allocate device memory when they decode: an engine whose device memory is
 * partitioned once at start-up and may not grow, or a plugin hosted by a
 * runtime that exposes no allocator, where a cudaMalloc in the middle of a
 * step would also synchronise the device.  The pages have no counterpart to
 * this call; it exists for those integrations only.
 *
 * Arguments, results and errors are those of ds4x_sparse_attn_decode without
 * the workspace.  The workspace (its 256-byte status header; the split
 * partials stay in shared memory) is one static device array inside the
 * library (k outside 1..512 returns DS4X_EINVAL); every GPU that loads the
 * library holds that array until the process exits.  The call allocates
 * nothing and calls no allocating routine.  Its first call on a device looks
 * up the array's device address (cudaGetSymbolAddress, with that device
 * current); make that first call before any stream capture.  The address is
 * kept for the life of the process, so the call must not be used on a
 * device after cudaDeviceReset has destroyed the context that first looked
 * it up (the reloaded module may place the array elsewhere).  All calls share
 * the one array, so calls that may overlap on the GPU (different streams, or
 * several host threads) race and must be serialised by the caller.  Nothing
 * in the array needs to start at zero; out-of-range indices are skipped as
 * in ds4x_sparse_attn_decode, but with no workspace there is no status word
 * to report them.
 */
int ds4x_sparse_attn_decode_noalloc(const uint8_t *kv_rows, int64_t n_rows, const int32_t *idx,
                                    int32_t k, const uint16_t *q_bf16, float softmax_scale,
                                    uint16_t *out_bf16, float *lse, ds4x_stream_t stream);

/* Dense decode attention over EVERY row of a KV row array: the HCA layers'
 * exact attention over all their compressed rows (DS4X README, "Optimization
 * details", the HCA bullet: exact score-split attention with no row
 * ceiling).  For each head h < 64, over t in [0, n_rows):
 *
 *   l_ht = softmax_scale * (q_h . v_t),  o_h = sum_t softmax_t(l_ht) v_t,
 *   lse_h = log sum_t e^(l_ht)
 *
 * with v_t the dequantised row as in ds4x_sparse_attn_decode.  Computed as
 * items of R consecutive rows, R = 128 * min(4, max(1, ceil(n_rows /
 * 32768))) (128 rows up to 32,768 rows, so 64 items at 8192 rows), each
 * through the tensor-core kernel of ds4x_sparse_attn_prefill (with its
 * numerics, the block scales' range taken over the item's rows) writing its
 * normalised fp32 output and LSE into the workspace, then a log-sum-exp
 * combine over the items.  Workspace: 256 + items * (256 + 131072) bytes,
 * items = ceil(n_rows / R).
 *
 *   kv_rows   u8 [n_rows][583]
 *   n_rows    1 .. DS4X_DENSE_MAX_ROWS
 *   q_bf16    u16 [64][512]
 *   out_bf16  u16 [64][512] (bf16, round to nearest even)
 *   lse       f32 [64] or NULL
 *   ws        ds4x_dense_attn_decode_workspace(n_rows) bytes, owned by the
 *             caller; no initialisation needed; its first 256 bytes are
 *             the status header (ds4x_workspace_status)
 *
 * Errors: DS4X_EINVAL (null or misaligned pointer, n_rows out of range),
 * DS4X_EWORKSPACE (ws_bytes too small), DS4X_EARCH, DS4X_ECUDA.
 */
size_t ds4x_dense_attn_decode_workspace(int64_t n_rows);

/* Decode attention over k selected compressed rows AND the raw sliding
 * window: each layer keeps a raw KV ring of DS4X_RING_ROWS packed 583-byte
 * rows (DS4X README, "Packed cache ABI": the raw ring padded to 256 rows),
 * whose live rows are the most recent tokens.  One softmax over the union of
 * the two row sets (no deduplication), i.e. the log-sum-exp merge of the
 * sparse and the window attention:
 *
 *   rows = { kv_rows[idx[j]] : j < k, idx[j] >= 0 }
 *        + { ring_rows[(ring_pos - j) mod 256] : j < w }
 *
 *   kv_rows, n_rows, idx, k      as ds4x_sparse_attn_decode (1 <= k <= 512)
 *   ring_rows u8 [DS4X_RING_ROWS][583], physical ring order
 *   ring_pos  the newest window row's slot, 0 .. 255
 *   w         live window rows, 0 .. 256
 *   q_bf16, softmax_scale, out_bf16, lse   as ds4x_sparse_attn_decode
 *   ws        ds4x_window_sparse_attn_decode_workspace() bytes; its first
 *             256 bytes are the status header (an index outside
 *             [-1, n_rows) is skipped and flags DS4X_EDEVICE there)
 *
 * Errors: DS4X_EINVAL (null or misaligned pointer, k, ring_pos or w out of
 * range), DS4X_EWORKSPACE, DS4X_EARCH, DS4X_ECUDA.
 */
size_t ds4x_window_sparse_attn_decode_workspace(void);
int ds4x_window_sparse_attn_decode(const uint8_t *kv_rows, int64_t n_rows, const int32_t *idx, int32_t k,
                                   const uint8_t *ring_rows, int32_t ring_pos, int32_t w,
                                   const uint16_t *q_bf16, float softmax_scale, uint16_t *out_bf16,
                                   float *lse, void *ws, size_t ws_bytes, ds4x_stream_t stream);
int ds4x_dense_attn_decode(const uint8_t *kv_rows, int64_t n_rows, const uint16_t *q_bf16,
                           float softmax_scale, uint16_t *out_bf16, float *lse, void *ws,
                           size_t ws_bytes, ds4x_stream_t stream);

/* ---- Packed-row checkpoints (host memory, no CUDA call) -----------------
 *
 * A checkpoint holds, per layer, the native packed rows: the raw sliding
 * window's live rows, the compressed KV rows and (CSA layers) the indexer
 * rows.  Disk checkpoints store the packed rows and the payload version (3)
 * rejects payloads of any other version, such as F32-cache version 2 (DS4X
 * README, "Optimization details"); the window rows go in logical position
 * order, oldest first, not physical ring order (ds4 README, "Disk KV Cache").
 * Tokens, logits and the compressor's frontier tensors are model state and
 * are not part of it.
 *
 * Layout (little-endian; this library's own):
 *   header, 64 bytes: "DS4X", u32 payload version = 3, u32 header bytes =
 *     64, u32 layer count, u32 ring rows = 256, u32 KV row bytes = 583,
 *     u32 indexer row bytes = 68, u32 layer entry bytes = 32, u64 total
 *     bytes, 24 zero bytes
 *   one 32-byte entry per layer: u32 ratio (0: raw window only; 4: CSA, KV
 *     and as many indexer rows; 128: HCA, KV rows), u32 live window rows
 *     (0..256), u64 KV rows, u64 indexer rows, u64 zero
 *   then per layer, in order: the live window rows (583 B each, oldest
 *     first), the KV rows (583 B each), the indexer rows (68 B each)
 *
 * All pointers here are host pointers, any alignment.  A file is checked
 * whole (magic, version, sizes, every entry, the total) before any row is
 * read: DS4X_EFORMAT for anything that is not this layout or is truncated,
 * DS4X_EVERSION for another payload version.
 */
typedef struct ds4x_layer_rows {
  int32_t ratio;              /* 0, 4 or 128 */
  int32_t ring_live;          /* live window rows, 0..DS4X_RING_ROWS */
  int32_t ring_pos;           /* the newest window row's slot, 0..255 */
  int32_t reserved;
  const uint8_t *ring_rows;   /* [DS4X_RING_ROWS][583], physical ring order */
  const uint8_t *kv_rows;     /* [n_kv][583] */
  const uint8_t *idx_rows;    /* [n_idx][68], CSA layers only */
  int64_t n_kv, n_idx;        /* CSA: n_idx == n_kv; HCA: n_idx == 0; ratio 0: both 0 */
} ds4x_layer_rows;

typedef struct ds4x_layer_counts {
  int32_t ratio, ring_live;
  int64_t n_kv, n_idx;
} ds4x_layer_counts;

typedef struct ds4x_layer_buffers {
  uint8_t *ring_rows;         /* [DS4X_RING_ROWS][583]: the window lands in slots
                                 0..ring_live-1, oldest first (newest slot ring_live-1) */
  uint8_t *kv_rows;           /* room for kv_cap rows */
  uint8_t *idx_rows;          /* room for idx_cap rows */
  int64_t kv_cap, idx_cap;
} ds4x_layer_buffers;

/* Bytes of the checkpoint of n_layers layers (0..DS4X_CHECKPOINT_MAX_LAYERS),
 * or DS4X_EINVAL for an inconsistent layer (counts, ratio, null rows). */
int64_t ds4x_checkpoint_bytes(const ds4x_layer_rows *layers, int32_t n_layers);
/* Writes the checkpoint into dst (DS4X_ERANGE if dst_bytes is too small). */
int ds4x_checkpoint_save(const ds4x_layer_rows *layers, int32_t n_layers, uint8_t *dst, int64_t dst_bytes);
/* Checks src whole; gives its layer count and, if counts is not NULL (room
 * for counts_cap layers, else DS4X_ERANGE), each layer's counts. */
int ds4x_checkpoint_inspect(const uint8_t *src, int64_t src_bytes, int32_t *n_layers, ds4x_layer_counts *counts,
                            int32_t counts_cap);
/* Checks src whole and every destination (DS4X_EINVAL for n_layers other
 * than the file's or a missing buffer, DS4X_ERANGE for too little room)
 * before copying the rows. */
int ds4x_checkpoint_load(const uint8_t *src, int64_t src_bytes, const ds4x_layer_buffers *bufs, int32_t n_layers);

#ifdef __cplusplus
}
#endif

#endif /* DS4X_H */
