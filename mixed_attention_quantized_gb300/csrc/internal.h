// internal.h -- structures shared by the host planner and the kernels.
//
// The planner (abi.cu) cuts a ForwardBatch into tiles; the fused attention
// kernel reads them from the workspace.  Everything here is plain data so the
// same definitions compile on the host and the device.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "../../include/mixattn.h"

#ifdef __CUDACC__
#define MIXATTN_HD __host__ __device__ __forceinline__
#else
#define MIXATTN_HD inline
#endif

namespace mixattn {

constexpr int kPage = 32;          // tokens per page (the cache's page_size)
constexpr int kBlock = 32;         // elements per quantisation block
constexpr int kThreads = 256;      // threads of a decode CTA (8 warps)
constexpr int kWarps = kThreads / 32;
constexpr int kFusedThreads = 512; // threads of a fused-launch CTA: three working warp groups and
                                   // an MMA/producer group on a chunk tile; a decode tile uses
                                   // the first kThreads
constexpr int kChunkM = 128;       // rows (query tokens x group heads) of a chunk tile
constexpr int kChunkN = 128;       // keys per KV tile of the chunk path (4 pages)
constexpr int kPagesPerKvTile = kChunkN / kPage;
constexpr int kMaxGroup = 8;       // q heads per kv head held in one mma N=8 tile
constexpr int kMaxDevices = 64;    // per-device caches of the host side (device ordinals below this)
constexpr int kVerifyMaxRows = 24; // a chunk row with q_len * G <= this (speculative verify) runs on
                                   // decode-style split-K tiles of up to 8 (query, head) rows: each
                                   // such group costs about a third of a 128-row tensor-core tile
                                   // per key, so up to three groups are cheaper than one tile

// Per-row data the kernel needs (copied with the tile list).
struct RowInfo {
  int32_t q_start;   // packed index of the row's first query token
  int32_t seq_len;   // keys of the row (its history plus the new tokens)
  int32_t q_offset;  // position of the row's first query
  int32_t n_splits;  // decode rows: split tiles per kv head; chunk rows: 0
};

// One tile of work for one CTA.
//   chunk:  queries begin .. begin+count-1 of `row` (count <= 128 / G), kv head kvh,
//           against 128-key KV tiles kv0 .. kv1-1; a tile whose key range is cut
//           into nsplit pieces (part = 0 .. nsplit-1, consecutive in the tile
//           list) leaves partial results that the last piece to finish merges
//   decode: pages begin .. begin+count-1 of `row`, kv head kvh, split `part` of the
//           row's n_splits, for queries kv1 .. kv1+nsplit-1 of the row (one query for a
//           decode row; up to 8 / G for a short chunk row); kv0 = partial slot of the
//           group's first split (its splits take slots kv0 .. kv0+n_splits-1, wherever
//           the tiles sit in the list), which also indexes the group's split ticket
struct TileDesc {
  int32_t row;
  int32_t kvh;
  int32_t begin;
  int32_t count;
  int32_t kv0;
  int32_t kv1;
  int32_t part;
  int32_t nsplit;
};

// Pages each warp of a decode CTA walks, a function of the row's own length
// only (so a row's result does not depend on the other rows of the batch):
// about 4 splits per (row, kv head) up to 1024 pages, then splits of 256 pages.
// Fewer, longer splits measured faster wherever a batch fills the GPU: each
// split pays a fixed set-up (page ids, first copies, Q, the warp merge) and its
// partial is merged serially by the last CTA of the (row, kv head).  Against ~8
// splits: 64 rows x 8192 tokens Q4_0 0.40 -> 0.47 of HBM, Q8_0 0.66 -> 0.75; the
// serving mix 209 -> 200 us; one 8192-token row alone 0.090 -> 0.076 (it fills
// only 32 CTAs).
MIXATTN_HD int decode_pages_per_warp(int n_pages) {
  int p = (n_pages + 31) / 32;
  return p < 1 ? 1 : (p > 32 ? 32 : p);
}

MIXATTN_HD int decode_pages_per_split(int n_pages) { return kWarps * decode_pages_per_warp(n_pages); }

MIXATTN_HD int quant_row_bytes(int fmt, int head_dim) {
  return fmt == MIXATTN_KV_F16 ? 2 * head_dim : (fmt == MIXATTN_KV_Q8_0 ? head_dim : head_dim / 2);
}

MIXATTN_HD int scale_row_bytes(int fmt, int head_dim) {
  return fmt == MIXATTN_KV_F16 ? 0 : 2 * (head_dim / kBlock);
}

// Workspace layout of one plan (byte offsets from the workspace base).
struct WorkspaceLayout {
  size_t rows;            // RowInfo[n_rows]
  size_t tiles;           // TileDesc[n_tiles]      (chunk tiles first)
  size_t counters;        // uint32[n_decode_tiles + n_chunk_tiles]  (zeroed by every run's copy):
                          // decode split tickets (indexed by a group's first partial slot), then
                          // chunk-piece tickets
  size_t upload_end;      // end of the block copied from the plan's host buffer
  size_t partials;        // float[n_decode_tiles][slot_rows][head_dim + 2]
  size_t chunk_partials;  // float[n_chunk_tiles][128][head_dim + 2] when any chunk tile is split
  size_t total;
};

MIXATTN_HD size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// slot_rows: rows of one decode partial slot, G (every decode-kind tile holds one
// query) or 8 when the plan has verify groups
MIXATTN_HD WorkspaceLayout workspace_layout(int n_rows, int n_tiles, int n_decode_tiles, int slot_rows,
                                            int head_dim, bool chunk_split) {
  const size_t n_chunk = (size_t)(n_tiles - n_decode_tiles);
  WorkspaceLayout L;
  L.rows = 256;
  L.tiles = align_up(L.rows + sizeof(RowInfo) * (size_t)n_rows, 16);
  L.counters = align_up(L.tiles + sizeof(TileDesc) * (size_t)n_tiles, 16);
  L.upload_end = align_up(L.counters + sizeof(uint32_t) * ((size_t)n_decode_tiles + n_chunk), 16);
  L.partials = align_up(L.upload_end, 256);
  L.chunk_partials =
      align_up(L.partials + sizeof(float) * (size_t)n_decode_tiles * slot_rows * (head_dim + 2), 256);
  L.total = align_up(L.chunk_partials + (chunk_split ? sizeof(float) * n_chunk * kChunkM * (head_dim + 2) : 0), 256);
  return L;
}

// Kernel arguments (passed by value).
struct AttnParams {
  const void* q;              // fp16 [total_q][hq][D]
  void* o;                    // fp16 [total_q][hq][D]
  const uint8_t* k_quant;
  const uint16_t* k_scale;
  const uint8_t* v_quant;
  const uint16_t* v_scale;
  const int32_t* page_table;  // [n_rows][max_pages]
  const RowInfo* rows;
  const TileDesc* tiles;
  uint32_t* counters;         // [n_decode_tiles] split tickets, then one per chunk tile (piece tickets)
  float* partials;            // [n_decode_tiles][slot_rows][D + 2]
  float* chunk_partials;      // O [n_chunk_tiles][128][D], then (m, l) [n_chunk_tiles][128] of the
                              // pieces of cut chunk tiles
  uint32_t* chunk_counters;   // [n_chunk_tiles]: piece tickets, indexed by a tile's first piece
  int32_t max_pages;
  int32_t num_pages;
  int32_t n_chunk_tiles;
  int32_t n_chunk_ctas;       // CTAs walking the chunk tiles (set by the launcher)
  int32_t chunk_kv_tiles;     // KV tiles over all chunk tiles
  int32_t n_decode_tiles;
  int32_t hq;
  int32_t hkv;
  int32_t group;              // hq / hkv, 1..8
  int32_t log2_group;
  float scale_log2;           // log2(e) / sqrt(D)
  int32_t window = 0;         // > 0: sliding window, the query at position p sees keys p-window+1 .. p
  int32_t slot_rows = 0;      // rows of a decode partial slot (0: group)
};

// First key a query at position `pos` sees (0 without a window).
MIXATTN_HD int window_first_key(int pos, int window) {
  return (window > 0 && pos + 1 > window) ? pos + 1 - window : 0;
}

}  // namespace mixattn

#ifdef __CUDACC__
#include <cuda_runtime.h>
namespace mixattn {
// Launchers, one translation unit per (K format, V format) pair.
#define MIXATTN_DECLARE_LAUNCH(NAME) \
  cudaError_t NAME(int head_dim, const AttnParams& p, unsigned int* err, cudaStream_t s);
MIXATTN_DECLARE_LAUNCH(launch_attention_f16_f16)
MIXATTN_DECLARE_LAUNCH(launch_attention_q8_q8)
MIXATTN_DECLARE_LAUNCH(launch_attention_q4_q4)
MIXATTN_DECLARE_LAUNCH(launch_attention_q8_q4)
MIXATTN_DECLARE_LAUNCH(launch_attention_q4_q8)
#undef MIXATTN_DECLARE_LAUNCH
cudaError_t launch_kv_append(const mixattn_kv_cache& c, const void* k_new, const void* v_new,
                             const int32_t* slots, int32_t n_new, unsigned int* err, cudaStream_t s);
cudaError_t launch_kv_export(const mixattn_kv_cache& c, int which, const int32_t* slots, int32_t n,
                             void* out, unsigned int* err, cudaStream_t s);

}  // namespace mixattn
#endif  // __CUDACC__
