// noalloc.cu -- the mixed-batch attention step without any allocation.
//
// Some callers cannot hand this library a device workspace: a host runtime that
// reserves all GPU memory up front and forbids further cudaMalloc calls, a
// latency-critical serving loop in which a device allocation would synchronise
// the whole device, or a plain C host with no allocator for device buffers at
// all.  For them, mixattn_mixed_attention_noalloc runs the same kernels with
// the workspace in a file-scope device array owned by the library, and stages
// the tile list in a file-scope host array; it calls no cudaMalloc, cudaFree,
// cudaHostAlloc or any other allocating routine.
//
// Costs of that choice, stated in include/mixattn.h as well:
//   * every GPU that loads the library holds kStaticScratchBytes (16 MiB) of
//     device memory until the process exits;
//   * batches whose workspace exceeds it are rejected with MIXATTN_ERR_WORKSPACE;
//   * all calls share the one array (and the host staging array), so calls whose
//     GPU work overlaps -- on two streams, or from two host threads without
//     ordering -- race on it; the split counters are re-zeroed by every call;
//   * the tile list is copied from pageable host memory, which waits for the
//     stream's earlier work before the call returns.
#include <cuda_runtime.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "internal.h"

namespace mixattn {

unsigned int* device_error_address();  // abi.cu

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // device workspace, per GPU
constexpr size_t kStaticUploadBytes = size_t(1) << 20;    // host staging of rows + tiles + counters

}  // namespace

static __device__ __align__(256) uint8_t g_noalloc_scratch[kStaticScratchBytes];

namespace {

alignas(256) uint8_t g_upload[kStaticUploadBytes];  // host side, guarded by g_upload_mu
std::mutex g_upload_mu;

// Device address of g_noalloc_scratch on the current device.  In host code the
// array's name is only a stand-in, so the address is looked up once per device
// (with that device current) and cached.
uint8_t* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  static std::mutex mu;
  static uint8_t* ptrs[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<uint8_t*>(p);
  }
  return ptrs[dev];
}

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_cache_noalloc(const mixattn_kv_cache* c) {
  if (!c) return MIXATTN_ERR_INVALID_ARG;
  if (c->num_pages <= 0 || c->num_kv_heads <= 0 || c->head_dim <= 0) return MIXATTN_ERR_INVALID_ARG;
  if (c->page_size != kPage) return MIXATTN_ERR_UNSUPPORTED;
  if (c->head_dim % kBlock != 0) return MIXATTN_ERR_INVALID_ARG;
  if (c->head_dim != 64 && c->head_dim != 128) return MIXATTN_ERR_UNSUPPORTED;
  auto ok_fmt = [](int f) { return f == MIXATTN_KV_F16 || f == MIXATTN_KV_Q8_0 || f == MIXATTN_KV_Q4_0; };
  if (!ok_fmt(c->k_fmt) || !ok_fmt(c->v_fmt)) return MIXATTN_ERR_INVALID_ARG;
  if ((c->k_fmt == MIXATTN_KV_F16) != (c->v_fmt == MIXATTN_KV_F16)) return MIXATTN_ERR_UNSUPPORTED;
  if ((int64_t)c->num_pages * kPage > INT32_MAX) return MIXATTN_ERR_INVALID_ARG;
  if (!c->k_quant || !c->v_quant || !aligned_to(c->k_quant, 256) || !aligned_to(c->v_quant, 256))
    return MIXATTN_ERR_INVALID_ARG;
  if (c->k_fmt != MIXATTN_KV_F16 && (!c->k_scale || !aligned_to(c->k_scale, 256))) return MIXATTN_ERR_INVALID_ARG;
  if (c->v_fmt != MIXATTN_KV_F16 && (!c->v_scale || !aligned_to(c->v_scale, 256))) return MIXATTN_ERR_INVALID_ARG;
  return MIXATTN_OK;
}

// Tiles the batch straight into g_upload (no heap): row table, chunk tiles
// (heaviest first), decode tiles (splits of one (row, kv head) consecutive),
// zeroed split counters.  Returns a status; fills the layout and counts.
int tile_into_upload(const mixattn_kv_cache& c, int hq, int n_rows, const int32_t* kinds, const int32_t* seq,
                     const int32_t* off, int max_pages, WorkspaceLayout* L_out, int* n_chunk_out,
                     int* n_decode_out, int32_t* kv_tiles_out) {
  if (n_rows <= 0 || !kinds || !seq || !off || max_pages <= 0) return MIXATTN_ERR_INVALID_ARG;
  if (hq <= 0 || hq % c.num_kv_heads != 0) return MIXATTN_ERR_INVALID_ARG;
  const int G = hq / c.num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return MIXATTN_ERR_UNSUPPORTED;
  const int hkv = c.num_kv_heads;
  const int T = kChunkM / G;
  // first pass: validate and count
  int64_t n_chunk = 0, n_decode = 0, total_q = 0;
  for (int r = 0; r < n_rows; ++r) {
    const int64_t s = seq[r], o = off[r];
    if (kinds[r] == MIXATTN_ROW_DECODE) {
      if (s < 1 || o != s - 1) return MIXATTN_ERR_INVALID_ARG;
    } else if (kinds[r] == MIXATTN_ROW_CHUNK) {
      if (o < 0 || o >= s) return MIXATTN_ERR_INVALID_ARG;
    } else {
      return MIXATTN_ERR_INVALID_ARG;
    }
    const int64_t n_pages = (s + kPage - 1) / kPage;
    if (n_pages > max_pages || n_pages > c.num_pages) return MIXATTN_ERR_INVALID_ARG;
    if (kinds[r] == MIXATTN_ROW_CHUNK) {
      n_chunk += (int64_t)hkv * ((s - o + T - 1) / T);
    } else {
      const int pps = decode_pages_per_split((int)n_pages);
      n_decode += (int64_t)hkv * ((n_pages + pps - 1) / pps);
    }
    total_q += s - o;
    if (total_q > INT32_MAX / std::max(hq, 1)) return MIXATTN_ERR_INVALID_ARG;
  }
  const int64_t n_tiles = n_chunk + n_decode;
  if (n_tiles > INT32_MAX / 2) return MIXATTN_ERR_INVALID_ARG;
  // this path never cuts chunk tiles (its scratch holds no chunk partials)
  const WorkspaceLayout L = workspace_layout(n_rows, (int)n_tiles, (int)n_decode, G, c.head_dim, false);
  if (L.total > kStaticScratchBytes || L.upload_end - L.rows > kStaticUploadBytes) return MIXATTN_ERR_WORKSPACE;

  // second pass: write the image
  memset(g_upload, 0, L.upload_end - L.rows);
  RowInfo* rows = reinterpret_cast<RowInfo*>(g_upload);
  TileDesc* tiles = reinterpret_cast<TileDesc*>(g_upload + (L.tiles - L.rows));
  int64_t ic = 0, id = n_chunk, q0 = 0, kv_tiles = 0;
  for (int r = 0; r < n_rows; ++r) {
    const int64_t s = seq[r], o = off[r], nq = s - o;
    const int64_t n_pages = (s + kPage - 1) / kPage;
    rows[r].q_start = (int32_t)q0;
    rows[r].seq_len = (int32_t)s;
    rows[r].q_offset = (int32_t)o;
    rows[r].n_splits = 0;
    if (kinds[r] == MIXATTN_ROW_CHUNK) {
      for (int g = 0; g < hkv; ++g)
        for (int64_t b = 0; b < nq; b += T) {
          const int32_t cnt = (int32_t)std::min<int64_t>(T, nq - b);
          const int64_t key_end = std::min<int64_t>(s, o + b + cnt);
          const int32_t n_kv = (int32_t)((key_end + kChunkN - 1) / kChunkN);
          tiles[ic++] = TileDesc{r, g, (int32_t)b, cnt, 0, n_kv, 0, 1};
          kv_tiles += n_kv;
        }
    } else {
      const int pps = decode_pages_per_split((int)n_pages);
      const int ns = (int)((n_pages + pps - 1) / pps);
      rows[r].n_splits = ns;
      for (int g = 0; g < hkv; ++g) {
        const int32_t first = (int32_t)(id - n_chunk);  // partial slot of split 0
        for (int sp = 0; sp < ns; ++sp)
          tiles[id++] =
              TileDesc{r, g, sp * pps, (int32_t)std::min<int64_t>(pps, n_pages - (int64_t)sp * pps), first, 0, sp, 1};
        // (kv1 = 0, nsplit = 1: the group is the decode row's one query)
      }
    }
    q0 += nq;
  }
  // heaviest chunk tiles first; ties in a fixed order (in place, no allocation)
  auto cost = [&](const TileDesc& t) {
    const RowInfo& ri = rows[t.row];
    const int64_t key_end = std::min<int64_t>(ri.seq_len, (int64_t)ri.q_offset + t.begin + t.count);
    return (key_end + kChunkN - 1) / kChunkN;
  };
  std::sort(tiles, tiles + n_chunk, [&](const TileDesc& a, const TileDesc& b) {
    const int64_t ca = cost(a), cb = cost(b);
    if (ca != cb) return ca > cb;
    if (a.row != b.row) return a.row < b.row;
    if (a.kvh != b.kvh) return a.kvh < b.kvh;
    return a.begin < b.begin;
  });
  // longest decode tiles first; ties in row order (each keeps its partial slot)
  std::sort(tiles + n_chunk, tiles + n_tiles, [](const TileDesc& a, const TileDesc& b) {
    if (a.count != b.count) return a.count > b.count;
    if (a.row != b.row) return a.row < b.row;
    if (a.kvh != b.kvh) return a.kvh < b.kvh;
    return a.begin < b.begin;
  });
  *L_out = L;
  *kv_tiles_out = (int32_t)std::min<int64_t>(kv_tiles, INT32_MAX);
  *n_chunk_out = (int)n_chunk;
  *n_decode_out = (int)n_decode;
  return MIXATTN_OK;
}

}  // namespace
}  // namespace mixattn

using namespace mixattn;

extern "C" int mixattn_mixed_attention_noalloc(const mixattn_kv_cache* cache, int32_t num_q_heads, const void* q,
                                               const int32_t* page_table, int32_t max_pages, int32_t n_rows,
                                               const int32_t* seq_lens, const int32_t* q_offsets,
                                               const int32_t* row_kinds, void* o, mixattn_stream stream) {
  int st = check_cache_noalloc(cache);
  if (st != MIXATTN_OK) return st;
  if (!q || !o || !page_table || !aligned_to(q, 16) || !aligned_to(o, 16) || !aligned_to(page_table, 4))
    return MIXATTN_ERR_INVALID_ARG;
  uint8_t* ws = scratch_address();
  unsigned int* err = device_error_address();
  if (!ws || !err) return MIXATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  std::lock_guard<std::mutex> lock(g_upload_mu);
  WorkspaceLayout L;
  int n_chunk = 0, n_decode = 0;
  int32_t chunk_kv_tiles = 0;
  st = tile_into_upload(*cache, num_q_heads, n_rows, row_kinds, seq_lens, q_offsets, max_pages, &L, &n_chunk,
                        &n_decode, &chunk_kv_tiles);
  if (st != MIXATTN_OK) return st;
  // pageable source: the call returns once g_upload has been consumed
  if (cudaMemcpyAsync(ws + L.rows, g_upload, L.upload_end - L.rows, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return MIXATTN_ERR_CUDA;

  const int G = num_q_heads / cache->num_kv_heads;
  int lg = 0;
  while ((1 << lg) < G) ++lg;
  AttnParams p;
  p.q = q;
  p.o = o;
  p.k_quant = static_cast<const uint8_t*>(cache->k_quant);
  p.k_scale = static_cast<const uint16_t*>(cache->k_scale);
  p.v_quant = static_cast<const uint8_t*>(cache->v_quant);
  p.v_scale = static_cast<const uint16_t*>(cache->v_scale);
  p.page_table = page_table;
  p.rows = reinterpret_cast<const RowInfo*>(ws + L.rows);
  p.tiles = reinterpret_cast<const TileDesc*>(ws + L.tiles);
  p.counters = reinterpret_cast<uint32_t*>(ws + L.counters);
  p.partials = reinterpret_cast<float*>(ws + L.partials);
  p.chunk_partials = reinterpret_cast<float*>(ws + L.chunk_partials);
  p.chunk_counters = p.counters + n_decode;
  p.max_pages = max_pages;
  p.num_pages = cache->num_pages;
  p.n_chunk_tiles = n_chunk;
  p.chunk_kv_tiles = chunk_kv_tiles;
  p.n_decode_tiles = n_decode;
  p.hq = num_q_heads;
  p.hkv = cache->num_kv_heads;
  p.group = G;
  p.log2_group = lg;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)cache->head_dim));
  const int kf = cache->k_fmt, vf = cache->v_fmt, d = cache->head_dim;
  cudaError_t e;
  if (kf == MIXATTN_KV_F16) e = launch_attention_f16_f16(d, p, err, s);
  else if (kf == MIXATTN_KV_Q8_0 && vf == MIXATTN_KV_Q8_0) e = launch_attention_q8_q8(d, p, err, s);
  else if (kf == MIXATTN_KV_Q4_0 && vf == MIXATTN_KV_Q4_0) e = launch_attention_q4_q4(d, p, err, s);
  else if (kf == MIXATTN_KV_Q8_0) e = launch_attention_q8_q4(d, p, err, s);
  else e = launch_attention_q4_q8(d, p, err, s);
  return e == cudaSuccess ? MIXATTN_OK : MIXATTN_ERR_CUDA;
}
