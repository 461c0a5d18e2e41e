/*
 * mixattn.h -- C ABI of the mixed-batch attention library for GB300 (sm_103a).
 *
 * One launch serves chunked-prefill rows (a causal query slice at a position
 * offset) and decode rows (one query each) of the same batch, reading a paged
 * KV cache stored as 32-element blocks (fp16, Q8_0 or Q4_0) and dequantising
 * inside the attention.  A second entry point quantises new K/V into the
 * cache.  Everything runs on the caller's CUDA stream; there is no CPU
 * fallback.
 *
 * Sources (reference page "自研RDNA高併發推論引擎 以AI Max+ 395為範例",
 * lcz.me topic 2938):
 *   - §1 "統一 mixed-batch 介面": chunk rows and decode rows share one
 *     ForwardBatch and one attention kernel            -> mixattn_run
 *   - §1 guarantees table: a prompt is fed one bounded chunk per round
 *                                                      -> chunk rows
 *   - §2 modes table: q8 = blocked 8-bit, one f16 scale per 32 elements
 *     (34 B); 4-bit K and/or V packed into 18 B blocks -> mixattn_kv_fmt
 *   - §2: "blocked mode is bit-exact at the codec level"
 *                                                      -> mixattn_kv_append_quant
 *   - §2 occupancy table: bytes per KV position        -> mixattn_kv_cache_bytes
 *
 * Conventions
 *   - All pointers named *_d or documented "device" are device pointers; the
 *     library never frees them.  Host arrays are read during the call only.
 *   - Every function returns a mixattn_status (0 = OK) unless stated.  Host
 *     validation happens before any launch; on an error nothing is launched.
 *   - Kernels check page ids and slots on the device.  A bad one sets a bit in
 *     a device error word and the offending page or token is skipped (no trap);
 *     read and clear it with mixattn_device_error().  A decode split or chunk
 *     piece whose every page was skipped has no keys: its outputs are NaN.
 *   - Device checks surface at the next call: once a kernel has set an error
 *     bit on a device (a bad page id or slot, or a bounded wait that gave up),
 *     every later call of mixattn_kv_append_quant, mixattn_kv_export_blocks,
 *     mixattn_run and mixattn_mixed_attention on that device returns
 *     MIXATTN_ERR_DEVICE_CHECK and launches nothing, until
 *     mixattn_device_error(1) clears the word.  The host learns of it through
 *     a pinned, host-mapped flag that the kernels set beside the word, so the
 *     check costs no synchronisation; it sees kernels that have finished, and
 *     the first mixattn_plan_create on a device arms it (before that, and on
 *     the no-allocation entry point, only mixattn_device_error reports).
 *   - No call allocates device memory.  mixattn_plan_create allocates one
 *     pinned host buffer, owned by the plan, and the first one on a device a
 *     64-byte pinned flag that lives until the process exits.
 *   - Outputs are rounded to the nearest fp16, saturating at +-65504: a Q8_0
 *     block whose largest element is 65504 dequantises it to 127 * 516 = 65532,
 *     and a mean dominated by such values stays finite.
 */
#ifndef MIXATTN_H
#define MIXATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* KV block formats (§2 modes table).  K and V are chosen independently, so
 * the page's mixed K8V4 / K4V8 modes are expressible. */
typedef enum {
  MIXATTN_KV_F16 = 0,  /* plain fp16, no scale plane                          */
  MIXATTN_KV_Q8_0 = 1, /* fp16 d = amax/127, int8 q = round(x/d)  (34 B/block) */
  MIXATTN_KV_Q4_0 = 2  /* fp16 d = m/-8, 4-bit q = min(15, trunc(x/d + 8.5)),
                          value (q-8)*d; byte k = q_k | q_{k+16} << 4 (18 B)  */
} mixattn_kv_fmt;

/* Row kinds of one ForwardBatch (§1). */
typedef enum {
  MIXATTN_ROW_DECODE = 0, /* one query at position seq_len-1; q_offset == seq_len-1 */
  MIXATTN_ROW_CHUNK = 1   /* seq_len-q_offset queries at positions q_offset..seq_len-1 */
} mixattn_row_kind;

typedef enum {
  MIXATTN_OK = 0,
  MIXATTN_ERR_INVALID_ARG = -1,  /* a pointer, size or row descriptor is invalid   */
  MIXATTN_ERR_UNSUPPORTED = -2,  /* valid but not built: head_dim, group size ...  */
  MIXATTN_ERR_WORKSPACE = -3,    /* workspace NULL, misaligned or too small         */
  MIXATTN_ERR_CUDA = -4,         /* a CUDA runtime call failed (launch, copy)       */
  MIXATTN_ERR_DEVICE_CHECK = -5  /* a device-side check failed (see device_error)   */
} mixattn_status;

/* Device error word bits (mixattn_device_error). */
#define MIXATTN_DEVERR_PAGE_ID 0x1u  /* page_table entry outside [0, num_pages)     */
#define MIXATTN_DEVERR_SLOT 0x2u     /* slot_mapping entry >= num_pages * page_size */
#define MIXATTN_DEVERR_TIMEOUT 0x4u  /* a bounded device wait gave up               */

/* A cudaStream_t passed as an opaque pointer (NULL = the legacy default stream). */
typedef void* mixattn_stream;

/*
 * The paged KV cache.  Plain data; the caller owns every plane.
 *
 * Physical slot s = page * page_size + offset holds one token.  Per page and
 * kv head, K and V each have a quant plane and (quantised formats) a scale
 * plane, so every page plane is one contiguous, 16-byte aligned run:
 *
 *   quant plane  [num_pages][num_kv_heads][page_size][row_bytes]
 *                row_bytes = 2*head_dim (F16), head_dim (Q8_0), head_dim/2 (Q4_0)
 *                Q8_0 row: block b = int8 q of elements 32b..32b+31, in order
 *                Q4_0 row: block b = 16 bytes, byte k = q_k | q_{k+16} << 4
 *   scale plane  [num_pages][num_kv_heads][page_size][head_dim/32] fp16 d
 *                (NULL for F16)
 *
 * A canonical GGUF-style block (34 / 18 bytes) is the scale followed by that
 * block's quant bytes; mixattn_kv_export_blocks gathers them.
 * Every plane pointer must be 256-byte aligned.
 */
typedef struct {
  int32_t num_pages;    /* physical pages in the pool, > 0                       */
  int32_t page_size;    /* tokens per page; must be 32                           */
  int32_t num_kv_heads; /* > 0                                                   */
  int32_t head_dim;     /* 64 or 128                                             */
  int32_t k_fmt;        /* mixattn_kv_fmt of K                                   */
  int32_t v_fmt;        /* mixattn_kv_fmt of V                                   */
  void* k_quant;        /* device */
  void* k_scale;        /* device, NULL iff k_fmt == F16 */
  void* v_quant;        /* device */
  void* v_scale;        /* device, NULL iff v_fmt == F16 */
} mixattn_kv_cache;

/*
 * Bytes of each plane of a cache with these dimensions (pointers ignored).
 * plane_bytes_out (may be NULL) receives {k_quant, k_scale, v_quant, v_scale}.
 * Returns the total, or 0 if the dimensions or formats are invalid.
 * Per token and kv head this is 2D (F16), D + D/16 (Q8_0) and D/2 + D/16
 * (Q4_0) bytes for each of K and V: the §2 occupancy table's 2 : 1.0625 :
 * 0.5625 ratio.
 */
size_t mixattn_kv_cache_bytes(const mixattn_kv_cache* cache, size_t plane_bytes_out[4]);

/*
 * Quantise-on-append (§2 blocked KV; the verify path of §1 writes its rows
 * the same way).  For each new token t with slot_mapping[t] >= 0, every
 * (kv head, 32-element block along head_dim) of k_new / v_new is encoded in
 * the cache format and written to slot slot_mapping[t].  Bit-exact with the
 * codec definition above: fp32 arithmetic, x * (1/d) with IEEE division,
 * round-half-away (Q8_0), truncation after a separately rounded +8.5 (Q4_0),
 * lowest index wins a Q4_0 magnitude tie, fp16 scale rounded to nearest even.
 *
 *   k_new, v_new   device fp16 [n_new][num_kv_heads][head_dim], 16-byte aligned
 *   slot_mapping   device int32 [n_new]; negative = skip (padding token);
 *                  >= num_pages*page_size sets MIXATTN_DEVERR_SLOT, skipped
 *   n_new          >= 0 (0 launches nothing)
 * Two new tokens mapping to one slot race (last writer unspecified).
 */
int mixattn_kv_append_quant(const mixattn_kv_cache* cache, const void* k_new, const void* v_new,
                            const int32_t* slot_mapping, int32_t n_new, mixattn_stream stream);

/*
 * Gather canonical blocks from the cache (for checks and persistence).
 *   which   0 = K, 1 = V
 *   slots   device int32 [n] physical slots (each < num_pages*page_size)
 *   out     device uint8 [n][num_kv_heads][head_dim/32][block_bytes],
 *           block_bytes = 64 (F16), 34 (Q8_0), 18 (Q4_0); no alignment needed
 */
int mixattn_kv_export_blocks(const mixattn_kv_cache* cache, int32_t which, const int32_t* slots,
                             int32_t n, void* out, mixattn_stream stream);

/*
 * Plan: the host-side tiling of one ForwardBatch, reused for every layer.
 *
 * Rows are packed in order: the queries of row r start at
 * sum_{r'<r} (seq_len[r'] - q_offset[r']).  For every row
 *   decode: q_offset == seq_len - 1, seq_len >= 1
 *   chunk:  0 <= q_offset < seq_len
 * and ceil(seq_len / page_size) <= max_pages.  seq_len counts the new tokens,
 * whose K/V must already be in the cache (append first, then attend).
 *
 * Tiles: chunk rows are cut into (kv head, 128/G query tokens x G heads)
 * tensor-core tiles, heaviest first; when a chunk row has too few tiles to keep
 * every SM of the current device busy to the end, the key range of each of its
 * tiles is cut into 2-4 pieces whose partial results merge by log-sum-exp
 * (a choice made from the row itself and the device's SM count).  Decode rows
 * are cut into (kv head, page range) split-K tiles whose size depends only on
 * the row's own length; a chunk row of at most 24 (query, head) rows (a
 * speculative-verify pass: up to 6 draft tokens at G = 4) runs on such tiles too,
 * each holding up to 8 (query, head) rows.  So a row's output bits do not depend
 * on the rest of the batch.
 *
 *   num_q_heads      multiple of cache->num_kv_heads; G = num_q_heads /
 *                    num_kv_heads must be 1, 2, 4 or 8
 *   row_kinds, seq_lens, q_offsets   host int32 [n_rows], n_rows >= 1
 *   max_pages        row stride of the page table passed to mixattn_run
 *   workspace_bytes  out: device workspace mixattn_run needs
 */
typedef struct mixattn_plan mixattn_plan;

int mixattn_plan_create(mixattn_plan** plan_out, const mixattn_kv_cache* cache, int32_t num_q_heads,
                        int32_t n_rows, const int32_t* row_kinds, const int32_t* seq_lens,
                        const int32_t* q_offsets, int32_t max_pages, size_t* workspace_bytes);

/*
 * The same with a sliding window (reference page, §2 per-model table: the
 * Gemma 4 row's SWA layers read the same Q8 cache): every query at position p
 * sees keys max(0, p - window + 1) .. p only; window 0 is full causal attention
 * (mixattn_plan_create).  The tiling skips the pages and KV tiles before each
 * row's window, so a decode row reads ~window keys whatever its length.  A
 * model with both layer kinds keeps one plan per kind over the same batch.
 * window < 0 -> MIXATTN_ERR_INVALID_ARG.  mixattn_plan_update keeps the window.
 */
int mixattn_plan_create_window(mixattn_plan** plan_out, const mixattn_kv_cache* cache, int32_t num_q_heads,
                               int32_t window, int32_t n_rows, const int32_t* row_kinds, const int32_t* seq_lens,
                               const int32_t* q_offsets, int32_t max_pages, size_t* workspace_bytes);

/* Re-tile an existing plan for a new batch (same cache and heads), reusing its
 * pinned buffer when it is large enough.  Waits for the plan's previous
 * mixattn_run to have copied the old tile list before overwriting it. */
int mixattn_plan_update(mixattn_plan* plan, int32_t n_rows, const int32_t* row_kinds,
                        const int32_t* seq_lens, const int32_t* q_offsets, int32_t max_pages,
                        size_t* workspace_bytes);

/* Total query tokens (rows of q and o) and tile counts of a plan (every piece
 * of a cut chunk tile counts as one chunk tile). */
int mixattn_plan_info(const mixattn_plan* plan, int32_t* total_q, int32_t* n_chunk_tiles,
                      int32_t* n_decode_tiles);

/*
 * The mixed-batch attention step: one fused kernel over all tiles of the plan.
 * For every query at position p of row r and q head h (kv head h / G):
 *   o = sum_j softmax_j( q . k^_j / sqrt(head_dim) ) v^_j,  j = 0 .. p,
 * with k^, v^ the dequantised cache values.  fp16 in/out, fp32 softmax and
 * accumulation; decode rows are split over pages and merged by log-sum-exp.
 *
 *   q           device fp16 [total_q][num_q_heads][head_dim], 16-byte aligned
 *   page_table  device int32 [n_rows][max_pages]; entry i of row r is the
 *               physical page of the row's tokens 32i..32i+31
 *   o           device fp16 [total_q][num_q_heads][head_dim], 16-byte aligned
 *   workspace   device, >= workspace_bytes of the plan, 256-byte aligned; its
 *               contents need not be initialised and are overwritten
 * The call is asynchronous on `stream`: it enqueues two kernels, one that reads
 * the tile list from the plan's mapped pinned buffer into the workspace (no
 * copy-engine transfer, so it never waits behind the caller's own host-to-device
 * copies on other streams) and the attention kernel.  Runs of the
 * same plan on different streams must not overlap (they share the buffer only
 * for reading; the workspace is the caller's).
 */
int mixattn_run(const mixattn_plan* plan, const void* q, const int32_t* page_table, void* o,
                void* workspace, size_t workspace_bytes, mixattn_stream stream);

void mixattn_plan_destroy(mixattn_plan* plan);

/*
 * One call: mixed_attention(q, page_table, seq_lens, q_offsets, row_kinds) -> o.
 * A convenience path that synchronises: it plans (allocating the plan's pinned
 * buffer), runs, and frees the plan, and freeing pinned memory waits for the
 * device, so the call returns only after the stream's work up to the attention
 * launch has finished.  A serving loop should keep a plan and call
 * mixattn_plan_update + mixattn_run instead, which never wait.  workspace as
 * for mixattn_run; query its size with mixattn_workspace_bytes.
 */
int mixattn_mixed_attention(const mixattn_kv_cache* cache, int32_t num_q_heads, const void* q,
                            const int32_t* page_table, int32_t max_pages, int32_t n_rows,
                            const int32_t* seq_lens, const int32_t* q_offsets,
                            const int32_t* row_kinds, void* o, void* workspace,
                            size_t workspace_bytes, mixattn_stream stream);

/* Workspace bytes mixattn_mixed_attention needs for this batch (host arrays). */
int mixattn_workspace_bytes(const mixattn_kv_cache* cache, int32_t num_q_heads, int32_t n_rows,
                            const int32_t* row_kinds, const int32_t* seq_lens,
                            const int32_t* q_offsets, int32_t max_pages, size_t* workspace_bytes);

/*
 * The same attention step with no allocation of any kind.  The reference pages
 * have no counterpart of this entry point; it exists for callers that cannot
 * give the library a device workspace: a host runtime that reserves all GPU
 * memory up front and forbids further cudaMalloc calls, a latency-critical
 * serving loop where a device allocation would synchronise the device, or a
 * plain C host with no allocator for device buffers.
 *
 * Arguments are those of mixattn_mixed_attention minus the workspace: the
 * workspace lives in a library-owned file-scope device array of 16 MiB, which
 * every GPU that loads the library holds until the process exits, and the tile
 * list is staged in a library-owned host array.  No cudaMalloc, cudaFree,
 * cudaHostAlloc or other allocating routine is called.
 *   - Chunk tiles are never cut into key-range pieces here (that would need
 *     room for their partial results).  A batch whose remaining workspace
 *     exceeds 16 MiB -- at head_dim 128 and 4 q heads per kv head, about 8000
 *     decode split tiles -- returns MIXATTN_ERR_WORKSPACE and launches nothing.
 *   - The first call on a device looks up the array's device address (once per
 *     device, with that device current); make that first call before any stream
 *     capture.
 *   - All calls share the one array, which keeps the previous call's contents;
 *     each call re-zeroes what must start at zero (the split counters).  Calls
 *     whose GPU work overlaps -- on two streams, or from host threads without
 *     ordering -- race on the array.
 *   - The tile list is copied from pageable host memory, so the call waits for
 *     the stream's earlier work before it returns.
 */
int mixattn_mixed_attention_noalloc(const mixattn_kv_cache* cache, int32_t num_q_heads, const void* q,
                                    const int32_t* page_table, int32_t max_pages, int32_t n_rows,
                                    const int32_t* seq_lens, const int32_t* q_offsets,
                                    const int32_t* row_kinds, void* o, mixattn_stream stream);

/* Synchronously read (and, if clear != 0, reset) the device error word of the
 * current device: an OR of MIXATTN_DEVERR_* bits set by kernels since the
 * last clear.  Returns the word, or a negative status. */
int64_t mixattn_device_error(int32_t clear);

const char* mixattn_status_string(int32_t status);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t mixattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MIXATTN_H */
