// abi.cu -- host side of the C ABI: validation, the ForwardBatch planner and
// the launches.  See include/mixattn.h for the contract of every entry point.
//
// Page "自研RDNA高併發推論引擎 以AI Max+ 395為範例": §1 (chunk rows and decode
// rows share one ForwardBatch and one attention kernel; a prompt is fed one
// bounded chunk per round) and §2 (blocked Q8 / 4-bit KV modes).
#include <cuda_runtime.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <functional>
#include <mutex>
#include <queue>
#include <vector>

#include "../../include/mixattn_sched.h"
#include "internal.h"

namespace mixattn {

// Per device: word 0 = OR of MIXATTN_DEVERR_* bits set by kernels; words 2-3 =
// device address of the host-mapped flag that kernels also set (0 until armed).
__device__ __align__(16) unsigned int g_device_error[4] = {0u, 0u, 0u, 0u};

namespace {

std::mutex g_err_mu;
unsigned int* g_err_word[kMaxDevices] = {};          // device address of g_device_error
volatile unsigned int* g_err_flag[kMaxDevices] = {};  // host view of the armed flag

// Address of this device's error block (kernels receive it as an argument).
unsigned int* error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_err_mu);
  if (!g_err_word[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    g_err_word[dev] = static_cast<unsigned int*>(p);
  }
  return g_err_word[dev];
}

// Arms the host-mapped flag of the current device (once): a pinned, mapped
// word whose device address is stored in the error block, so kernels that set
// an error bit also set the flag and the next call sees it without touching
// the device.  The copy runs on a private non-blocking stream in relaxed
// capture mode, so it neither waits for nor disturbs the caller's streams.
// Failure leaves the device unarmed (calls then cannot report earlier checks,
// mixattn_device_error still can).
void arm_device_check() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return;
  if (!error_word()) return;
  std::lock_guard<std::mutex> lock(g_err_mu);
  if (g_err_flag[dev]) return;
  cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
  if (cudaThreadExchangeStreamCaptureMode(&mode) != cudaSuccess) return;
  unsigned int* host = nullptr;
  void* dptr = nullptr;
  cudaStream_t st = nullptr;
  bool ok = cudaHostAlloc(reinterpret_cast<void**>(&host), 64, cudaHostAllocMapped | cudaHostAllocPortable) ==
            cudaSuccess;
  if (ok) {
    host[0] = 0u;
    reinterpret_cast<void**>(host)[1] = nullptr;
    ok = cudaHostGetDevicePointer(&dptr, host, 0) == cudaSuccess && dptr;
  }
  if (ok) {
    reinterpret_cast<void**>(host)[1] = dptr;  // the value copied into words 2-3
    ok = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) == cudaSuccess;
  }
  if (ok) {
    ok = cudaMemcpyToSymbolAsync(g_device_error, reinterpret_cast<void**>(host) + 1, sizeof(void*),
                                 2 * sizeof(unsigned int), cudaMemcpyHostToDevice, st) == cudaSuccess &&
         cudaStreamSynchronize(st) == cudaSuccess;
  }
  if (st) cudaStreamDestroy(st);
  if (ok) {
    g_err_flag[dev] = host;
  } else {
    if (host) cudaFreeHost(host);
    cudaGetLastError();  // nothing of this is the caller's error
  }
  cudaThreadExchangeStreamCaptureMode(&mode);
}

// MIXATTN_ERR_DEVICE_CHECK when a kernel on the current device has set an error
// bit since the last clear (seen through the armed flag), else MIXATTN_OK.
int pending_device_check() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MIXATTN_OK;
  volatile unsigned int* f = g_err_flag[dev];
  return (f && *f) ? MIXATTN_ERR_DEVICE_CHECK : MIXATTN_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool valid_fmt(int f) { return f == MIXATTN_KV_F16 || f == MIXATTN_KV_Q8_0 || f == MIXATTN_KV_Q4_0; }

// Dimensions and formats only (no pointers).
int check_cache_dims(const mixattn_kv_cache* c) {
  if (!c) return MIXATTN_ERR_INVALID_ARG;
  if (c->num_pages <= 0 || c->num_kv_heads <= 0 || c->head_dim <= 0) return MIXATTN_ERR_INVALID_ARG;
  if (c->page_size != kPage) return MIXATTN_ERR_UNSUPPORTED;
  if (c->head_dim % kBlock != 0) return MIXATTN_ERR_INVALID_ARG;
  if (c->head_dim != 64 && c->head_dim != 128) return MIXATTN_ERR_UNSUPPORTED;
  if (!valid_fmt(c->k_fmt) || !valid_fmt(c->v_fmt)) return MIXATTN_ERR_INVALID_ARG;
  const bool kf = c->k_fmt == MIXATTN_KV_F16, vf = c->v_fmt == MIXATTN_KV_F16;
  if (kf != vf) return MIXATTN_ERR_UNSUPPORTED;  // fp16 pairs only with fp16
  if ((int64_t)c->num_pages * kPage > INT32_MAX) return MIXATTN_ERR_INVALID_ARG;
  return MIXATTN_OK;
}

int check_cache(const mixattn_kv_cache* c) {
  int st = check_cache_dims(c);
  if (st != MIXATTN_OK) return st;
  if (!c->k_quant || !c->v_quant) return MIXATTN_ERR_INVALID_ARG;
  if (!aligned(c->k_quant, 256) || !aligned(c->v_quant, 256)) return MIXATTN_ERR_INVALID_ARG;
  if (c->k_fmt != MIXATTN_KV_F16 && (!c->k_scale || !aligned(c->k_scale, 256))) return MIXATTN_ERR_INVALID_ARG;
  if (c->v_fmt != MIXATTN_KV_F16 && (!c->v_scale || !aligned(c->v_scale, 256))) return MIXATTN_ERR_INVALID_ARG;
  return MIXATTN_OK;
}

cudaError_t dispatch_attention(int k_fmt, int v_fmt, int head_dim, const AttnParams& p, unsigned int* err,
                               cudaStream_t s) {
  if (k_fmt == MIXATTN_KV_F16) return launch_attention_f16_f16(head_dim, p, err, s);
  if (k_fmt == MIXATTN_KV_Q8_0 && v_fmt == MIXATTN_KV_Q8_0) return launch_attention_q8_q8(head_dim, p, err, s);
  if (k_fmt == MIXATTN_KV_Q4_0 && v_fmt == MIXATTN_KV_Q4_0) return launch_attention_q4_q4(head_dim, p, err, s);
  if (k_fmt == MIXATTN_KV_Q8_0) return launch_attention_q8_q4(head_dim, p, err, s);
  return launch_attention_q4_q8(head_dim, p, err, s);
}

// The tiling of one batch: the image uploaded to the workspace plus counts.
struct Tiling {
  std::vector<uint8_t> image;  // [rows | tiles | counters], from WorkspaceLayout::rows
  int32_t total_q = 0, n_chunk = 0, n_decode = 0;
  int32_t slot_rows = 0;       // rows of a decode partial slot
  int32_t chunk_kv_tiles = 0;  // KV tiles over all chunk tiles (their mean decides persistence)
  WorkspaceLayout L{};
};

// SMs of the current device (0 when it cannot be read: no chunk splitting).
int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// Pieces per chunk tile of one chunk row: the key range of each of the row's
// tiles is cut into s pieces (s = 1..4) when that shortens the row's share of
// the launch, judged by placing the pieces heaviest first on the least-loaded
// of n_sm SMs (one chunk CTA per SM).  A piece costs its KV tiles plus one for
// its prologue and the merge; rows with a tile shorter than 8 KV tiles are
// never cut.
int chunk_split_factor(const std::vector<int64_t>& costs, int n_sm) {
  if (n_sm <= 0 || costs.empty()) return 1;
  int64_t min_cost = costs[0];
  for (int64_t c : costs) min_cost = std::min(min_cost, c);
  if (min_cost < 8) return 1;
  auto makespan = [&](int s) {
    std::vector<int64_t> pieces;
    pieces.reserve(costs.size() * s);
    for (int64_t c : costs)
      for (int q = 0; q < s; ++q) pieces.push_back((c * (q + 1)) / s - (c * q) / s + (s > 1 ? 1 : 0));
    std::sort(pieces.begin(), pieces.end(), std::greater<int64_t>());
    std::priority_queue<int64_t, std::vector<int64_t>, std::greater<int64_t>> load;
    for (int i = 0; i < n_sm; ++i) load.push(0);
    int64_t span = 0;
    for (int64_t pc : pieces) {
      const int64_t l = load.top() + pc;
      load.pop();
      load.push(l);
      span = std::max(span, l);
    }
    return span;
  };
  int best = 1;
  int64_t best_span = makespan(1);
  for (int s = 2; s <= 4; ++s) {
    const int64_t sp = makespan(s);
    if (sp * 20 < best_span * 19) {  // at least 5% shorter
      best = s;
      best_span = sp;
    }
  }
  return best;
}

int build_tiling(const mixattn_kv_cache& c, int hq, int n_rows, const int32_t* kinds, const int32_t* seq,
                 const int32_t* off, int max_pages, int n_sm, int window, Tiling* out) {
  if (n_rows <= 0 || !kinds || !seq || !off || max_pages <= 0 || window < 0) return MIXATTN_ERR_INVALID_ARG;
  if (hq <= 0 || hq % c.num_kv_heads != 0) return MIXATTN_ERR_INVALID_ARG;
  const int G = hq / c.num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return MIXATTN_ERR_UNSUPPORTED;
  const int hkv = c.num_kv_heads;
  const int T = kChunkM / G;  // query tokens per chunk tile
  const int QPG = kMaxGroup / G;  // queries per decode-style tile of a verify row
  bool any_verify = false;

  std::vector<RowInfo> rows(n_rows);
  struct Chunk {
    TileDesc t;
    int64_t kv_first;  // first KV tile the tile's queries can see
    int64_t cost;      // KV tiles from there to the last query's key
    int split;
  };
  std::vector<Chunk> chunks;
  std::vector<TileDesc> decodes;
  int64_t total_q = 0;
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
    if (n_pages > max_pages) return MIXATTN_ERR_INVALID_ARG;
    if (n_pages > c.num_pages) return MIXATTN_ERR_INVALID_ARG;
    rows[r].q_start = (int32_t)total_q;
    rows[r].seq_len = (int32_t)s;
    rows[r].q_offset = (int32_t)o;
    rows[r].n_splits = 0;
    const int64_t nq = s - o;
    // a short chunk row (speculative verify: q_len * G <= kVerifyMaxRows) runs like decode
    // rows, on split-K tiles of up to 8 (query, head) rows
    const bool verify = kinds[r] == MIXATTN_ROW_CHUNK && nq * G <= kVerifyMaxRows;
    any_verify = any_verify || verify;
    if (kinds[r] == MIXATTN_ROW_CHUNK && !verify) {
      const size_t first_chunk = chunks.size();
      for (int g = 0; g < hkv; ++g) {
        for (int64_t b = 0; b < nq; b += T) {
          Chunk ch;
          ch.t.row = r;
          ch.t.kvh = g;
          ch.t.begin = (int32_t)b;
          ch.t.count = (int32_t)std::min<int64_t>(T, nq - b);
          ch.t.kv0 = ch.t.kv1 = ch.t.part = 0;
          ch.t.nsplit = 1;
          const int64_t key_end = std::min<int64_t>(s, o + b + ch.t.count);
          // a sliding window skips the KV tiles before the first query's first key
          ch.kv_first = window_first_key((int)(o + b), window) / kChunkN;
          ch.cost = (key_end + kChunkN - 1) / kChunkN - ch.kv_first;
          ch.split = 1;
          chunks.push_back(ch);
        }
      }
      // how far to cut this row's tiles depends on the row alone (and the GPU), so
      // a row's result does not depend on the rest of the batch
      std::vector<int64_t> costs;
      for (size_t i = first_chunk; i < chunks.size(); ++i) costs.push_back(chunks[i].cost);
      const int split = chunk_split_factor(costs, n_sm);
      for (size_t i = first_chunk; i < chunks.size(); ++i) chunks[i].split = split;
    } else {
      // pages from the one holding the first query's window start (page 0 without a
      // window) to the last; the split size depends on the row alone
      const int64_t first_page = window_first_key((int)o, window) / kPage;
      const int64_t n_win = n_pages - first_page;
      const int pps = decode_pages_per_split((int)n_win);
      const int ns = (int)((n_win + pps - 1) / pps);
      rows[r].n_splits = ns;
      // query groups innermost: the groups reading the same pages sit side by side in
      // the tile list (and so run at about the same time), and the pages they share
      // come from L2 after the first read; slots are numbered group-major
      const int64_t n_groups = (nq + QPG - 1) / QPG;
      for (int g = 0; g < hkv; ++g) {
        const int32_t base = (int32_t)decodes.size();
        for (int sp = 0; sp < ns; ++sp) {
          for (int64_t gi = 0; gi < n_groups; ++gi) {
            TileDesc t;
            t.row = r;
            t.kvh = g;
            t.begin = (int32_t)(first_page + (int64_t)sp * pps);
            t.count = (int32_t)std::min<int64_t>(pps, n_win - (int64_t)sp * pps);
            t.kv0 = base + (int32_t)(gi * ns);                            // partial slot of split 0
            t.kv1 = (int32_t)(gi * QPG);                                  // the group's first query
            t.part = sp;
            t.nsplit = (int32_t)std::min<int64_t>(QPG, nq - gi * QPG);  // the group's queries
            decodes.push_back(t);
          }
        }
      }
    }
    total_q += nq;
    if (total_q > INT32_MAX / std::max(hq, 1)) return MIXATTN_ERR_INVALID_ARG;
  }
  // heaviest chunk tiles first (they set the length of the launch), each cut
  // into `split` consecutive pieces of its key range; longest decode tiles first
  // too, so the last wave holds the short ones (each keeps its partial slot)
  std::stable_sort(chunks.begin(), chunks.end(), [](const Chunk& a, const Chunk& b) { return a.cost > b.cost; });
  std::stable_sort(decodes.begin(), decodes.end(),
                   [](const TileDesc& a, const TileDesc& b) { return a.count > b.count; });
  int64_t n_pieces = 0;
  bool any_split = false;
  for (const Chunk& ch : chunks) {
    n_pieces += ch.split;
    any_split = any_split || ch.split > 1;
  }
  const int64_t n_tiles = n_pieces + (int64_t)decodes.size();
  if (n_tiles > INT32_MAX / 2) return MIXATTN_ERR_INVALID_ARG;

  Tiling& T2 = *out;
  T2.total_q = (int32_t)total_q;
  T2.n_chunk = (int32_t)n_pieces;
  T2.n_decode = (int32_t)decodes.size();
  T2.slot_rows = any_verify ? kMaxGroup : G;
  T2.L = workspace_layout(n_rows, (int)n_tiles, T2.n_decode, T2.slot_rows, c.head_dim, any_split);
  T2.image.assign(T2.L.upload_end - T2.L.rows, 0);
  memcpy(T2.image.data(), rows.data(), sizeof(RowInfo) * rows.size());
  TileDesc* td = reinterpret_cast<TileDesc*>(T2.image.data() + (T2.L.tiles - T2.L.rows));
  int64_t at = 0, kv_tiles = 0;
  for (size_t i = 0; i < chunks.size(); ++i) {
    const int64_t n_kv = chunks[i].cost, kv_first = chunks[i].kv_first;
    kv_tiles += n_kv;
    const int split = chunks[i].split;
    for (int q = 0; q < split; ++q) {
      TileDesc t = chunks[i].t;
      t.kv0 = (int32_t)(kv_first + (n_kv * q) / split);
      t.kv1 = (int32_t)(kv_first + (n_kv * (q + 1)) / split);
      t.part = q;
      t.nsplit = split;
      td[at++] = t;
    }
  }
  for (size_t i = 0; i < decodes.size(); ++i) td[n_pieces + i] = decodes[i];
  T2.chunk_kv_tiles = (int32_t)std::min<int64_t>(kv_tiles, INT32_MAX);
  // counters stay zero: every run starts its split tickets from 0
  return MIXATTN_OK;
}

}  // namespace

// Address of this device's error word, for launchers in other translation units.
unsigned int* device_error_address() { return error_word(); }

}  // namespace mixattn

using namespace mixattn;

struct mixattn_plan {
  mixattn_kv_cache cache;
  int32_t hq = 0, group = 0, log2_group = 0, n_rows = 0, max_pages = 0;
  int32_t window = 0;  // sliding window of every run of the plan (0: full causal attention)
  Tiling tiling;
  uint8_t* host_buf = nullptr;  // pinned, mapped copy of tiling.image
  const uint8_t* host_dev = nullptr;  // the same buffer as the device sees it
  size_t host_cap = 0;
  cudaEvent_t copied = nullptr;
  bool copy_recorded = false;
};

namespace {

int plan_fill(mixattn_plan* p, int32_t n_rows, const int32_t* kinds, const int32_t* seq, const int32_t* off,
              int32_t max_pages, size_t* ws_bytes) {
  Tiling t;
  int st = build_tiling(p->cache, p->hq, n_rows, kinds, seq, off, max_pages, device_sm_count(), p->window, &t);
  if (st != MIXATTN_OK) return st;
  // the previous run may still be copying from the pinned buffer
  if (p->copy_recorded) {
    if (cudaEventSynchronize(p->copied) != cudaSuccess) return MIXATTN_ERR_CUDA;
    p->copy_recorded = false;
  }
  if (t.image.size() > p->host_cap) {
    if (p->host_buf) cudaFreeHost(p->host_buf);
    p->host_buf = nullptr;
    p->host_dev = nullptr;
    p->host_cap = 0;
    size_t cap = std::max<size_t>(t.image.size(), 4096);
    if (cudaHostAlloc(reinterpret_cast<void**>(&p->host_buf), cap, cudaHostAllocMapped | cudaHostAllocPortable) !=
        cudaSuccess) {
      p->host_buf = nullptr;
      return MIXATTN_ERR_CUDA;
    }
    void* dv = nullptr;
    if (cudaHostGetDevicePointer(&dv, p->host_buf, 0) != cudaSuccess || !dv) {
      cudaFreeHost(p->host_buf);
      p->host_buf = nullptr;
      return MIXATTN_ERR_CUDA;
    }
    p->host_dev = static_cast<const uint8_t*>(dv);
    p->host_cap = cap;
  }
  memcpy(p->host_buf, t.image.data(), t.image.size());
  p->n_rows = n_rows;
  p->max_pages = max_pages;
  p->tiling = std::move(t);
  if (ws_bytes) *ws_bytes = p->tiling.L.total;
  return MIXATTN_OK;
}

}  // namespace

extern "C" {

size_t mixattn_kv_cache_bytes(const mixattn_kv_cache* c, size_t plane_bytes_out[4]) {
  if (check_cache_dims(c) != MIXATTN_OK) return 0;
  const size_t rows = (size_t)c->num_pages * c->num_kv_heads * kPage;
  const size_t kq = rows * quant_row_bytes(c->k_fmt, c->head_dim);
  const size_t ks = rows * scale_row_bytes(c->k_fmt, c->head_dim);
  const size_t vq = rows * quant_row_bytes(c->v_fmt, c->head_dim);
  const size_t vs = rows * scale_row_bytes(c->v_fmt, c->head_dim);
  if (plane_bytes_out) {
    plane_bytes_out[0] = kq;
    plane_bytes_out[1] = ks;
    plane_bytes_out[2] = vq;
    plane_bytes_out[3] = vs;
  }
  return kq + ks + vq + vs;
}

int mixattn_kv_append_quant(const mixattn_kv_cache* cache, const void* k_new, const void* v_new,
                            const int32_t* slot_mapping, int32_t n_new, mixattn_stream stream) {
  int st = check_cache(cache);
  if (st != MIXATTN_OK) return st;
  if (n_new < 0) return MIXATTN_ERR_INVALID_ARG;
  if (n_new == 0) return MIXATTN_OK;
  if (!k_new || !v_new || !slot_mapping) return MIXATTN_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(slot_mapping, 4)) return MIXATTN_ERR_INVALID_ARG;
  if ((st = pending_device_check()) != MIXATTN_OK) return st;
  unsigned int* err = error_word();
  if (!err) return MIXATTN_ERR_CUDA;
  cudaError_t e = launch_kv_append(*cache, k_new, v_new, slot_mapping, n_new, err,
                                   static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MIXATTN_OK : MIXATTN_ERR_CUDA;
}

int mixattn_kv_export_blocks(const mixattn_kv_cache* cache, int32_t which, const int32_t* slots, int32_t n,
                             void* out, mixattn_stream stream) {
  int st = check_cache(cache);
  if (st != MIXATTN_OK) return st;
  if ((which != 0 && which != 1) || n < 0) return MIXATTN_ERR_INVALID_ARG;
  if (n == 0) return MIXATTN_OK;
  if (!slots || !out || !aligned(slots, 4)) return MIXATTN_ERR_INVALID_ARG;
  if ((st = pending_device_check()) != MIXATTN_OK) return st;
  unsigned int* err = error_word();
  if (!err) return MIXATTN_ERR_CUDA;
  cudaError_t e = launch_kv_export(*cache, which, slots, n, out, err, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MIXATTN_OK : MIXATTN_ERR_CUDA;
}

int mixattn_plan_create(mixattn_plan** plan_out, const mixattn_kv_cache* cache, int32_t num_q_heads,
                        int32_t n_rows, const int32_t* row_kinds, const int32_t* seq_lens,
                        const int32_t* q_offsets, int32_t max_pages, size_t* workspace_bytes) {
  return mixattn_plan_create_window(plan_out, cache, num_q_heads, 0, n_rows, row_kinds, seq_lens, q_offsets,
                                    max_pages, workspace_bytes);
}

int mixattn_plan_create_window(mixattn_plan** plan_out, const mixattn_kv_cache* cache, int32_t num_q_heads,
                               int32_t window, int32_t n_rows, const int32_t* row_kinds, const int32_t* seq_lens,
                               const int32_t* q_offsets, int32_t max_pages, size_t* workspace_bytes) {
  if (!plan_out) return MIXATTN_ERR_INVALID_ARG;
  *plan_out = nullptr;
  int st = check_cache(cache);
  if (st != MIXATTN_OK) return st;
  if (num_q_heads <= 0 || num_q_heads % cache->num_kv_heads) return MIXATTN_ERR_INVALID_ARG;
  if (window < 0) return MIXATTN_ERR_INVALID_ARG;
  arm_device_check();
  mixattn_plan* p = new mixattn_plan();
  p->cache = *cache;
  p->window = window;
  p->hq = num_q_heads;
  p->group = num_q_heads / cache->num_kv_heads;
  p->log2_group = 0;
  while ((1 << p->log2_group) < p->group) ++p->log2_group;
  st = plan_fill(p, n_rows, row_kinds, seq_lens, q_offsets, max_pages, workspace_bytes);
  if (st == MIXATTN_OK && cudaEventCreateWithFlags(&p->copied, cudaEventDisableTiming) != cudaSuccess)
    st = MIXATTN_ERR_CUDA;
  if (st != MIXATTN_OK) {
    mixattn_plan_destroy(p);
    return st;
  }
  *plan_out = p;
  return MIXATTN_OK;
}

int mixattn_plan_update(mixattn_plan* plan, int32_t n_rows, const int32_t* row_kinds, const int32_t* seq_lens,
                        const int32_t* q_offsets, int32_t max_pages, size_t* workspace_bytes) {
  if (!plan) return MIXATTN_ERR_INVALID_ARG;
  return plan_fill(plan, n_rows, row_kinds, seq_lens, q_offsets, max_pages, workspace_bytes);
}

int mixattn_plan_info(const mixattn_plan* plan, int32_t* total_q, int32_t* n_chunk_tiles,
                      int32_t* n_decode_tiles) {
  if (!plan) return MIXATTN_ERR_INVALID_ARG;
  if (total_q) *total_q = plan->tiling.total_q;
  if (n_chunk_tiles) *n_chunk_tiles = plan->tiling.n_chunk;
  if (n_decode_tiles) *n_decode_tiles = plan->tiling.n_decode;
  return MIXATTN_OK;
}

// Copies n16 16-byte words of a plan's tile list from its mapped pinned buffer
// into the workspace.
static __global__ void upload_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n16) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

int mixattn_run(const mixattn_plan* plan_c, const void* q, const int32_t* page_table, void* o, void* workspace,
                size_t workspace_bytes, mixattn_stream stream) {
  mixattn_plan* plan = const_cast<mixattn_plan*>(plan_c);
  if (!plan) return MIXATTN_ERR_INVALID_ARG;
  if (!q || !o || !page_table) return MIXATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(o, 16) || !aligned(page_table, 4)) return MIXATTN_ERR_INVALID_ARG;
  const WorkspaceLayout& L = plan->tiling.L;
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.total) return MIXATTN_ERR_WORKSPACE;
  if (int st = pending_device_check()) return st;
  unsigned int* err = error_word();
  if (!err) return MIXATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // the tile list comes in through a small kernel reading the mapped pinned buffer
  // rather than a copy-engine transfer, which would queue behind any large
  // host-to-device copy the caller has in flight on another stream
  {
    const size_t n16 = (L.upload_end - L.rows) / 16;
    const int blocks = (int)std::min<size_t>((n16 + 255) / 256, 128);
    upload_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<const uint4*>(plan->host_dev),
                                         reinterpret_cast<uint4*>(ws + L.rows), n16);
    if (cudaGetLastError() != cudaSuccess) return MIXATTN_ERR_CUDA;
  }
  if (cudaEventRecord(plan->copied, s) != cudaSuccess) return MIXATTN_ERR_CUDA;
  plan->copy_recorded = true;

  AttnParams p;
  const mixattn_kv_cache& c = plan->cache;
  p.q = q;
  p.o = o;
  p.k_quant = static_cast<const uint8_t*>(c.k_quant);
  p.k_scale = static_cast<const uint16_t*>(c.k_scale);
  p.v_quant = static_cast<const uint8_t*>(c.v_quant);
  p.v_scale = static_cast<const uint16_t*>(c.v_scale);
  p.page_table = page_table;
  p.rows = reinterpret_cast<const RowInfo*>(ws + L.rows);
  p.tiles = reinterpret_cast<const TileDesc*>(ws + L.tiles);
  p.counters = reinterpret_cast<uint32_t*>(ws + L.counters);
  p.partials = reinterpret_cast<float*>(ws + L.partials);
  p.chunk_partials = reinterpret_cast<float*>(ws + L.chunk_partials);
  p.chunk_counters = p.counters + plan->tiling.n_decode;
  p.max_pages = plan->max_pages;
  p.num_pages = c.num_pages;
  p.n_chunk_tiles = plan->tiling.n_chunk;
  p.chunk_kv_tiles = plan->tiling.chunk_kv_tiles;
  p.n_decode_tiles = plan->tiling.n_decode;
  p.hq = plan->hq;
  p.hkv = c.num_kv_heads;
  p.group = plan->group;
  p.log2_group = plan->log2_group;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)c.head_dim));
  p.window = plan->window;
  p.slot_rows = plan->tiling.slot_rows;
  cudaError_t e = dispatch_attention(c.k_fmt, c.v_fmt, c.head_dim, p, err, s);
  return e == cudaSuccess ? MIXATTN_OK : MIXATTN_ERR_CUDA;
}

void mixattn_plan_destroy(mixattn_plan* plan) {
  if (!plan) return;
  if (plan->copy_recorded && plan->copied) cudaEventSynchronize(plan->copied);
  if (plan->copied) cudaEventDestroy(plan->copied);
  if (plan->host_buf) cudaFreeHost(plan->host_buf);
  delete plan;
}

int mixattn_workspace_bytes(const mixattn_kv_cache* cache, int32_t num_q_heads, int32_t n_rows,
                            const int32_t* row_kinds, const int32_t* seq_lens, const int32_t* q_offsets,
                            int32_t max_pages, size_t* workspace_bytes) {
  int st = check_cache_dims(cache);
  if (st != MIXATTN_OK) return st;
  if (!workspace_bytes) return MIXATTN_ERR_INVALID_ARG;
  Tiling t;
  st = build_tiling(*cache, num_q_heads, n_rows, row_kinds, seq_lens, q_offsets, max_pages, device_sm_count(), 0,
                    &t);
  if (st != MIXATTN_OK) return st;
  *workspace_bytes = t.L.total;
  return MIXATTN_OK;
}

int mixattn_mixed_attention(const mixattn_kv_cache* cache, int32_t num_q_heads, const void* q,
                            const int32_t* page_table, int32_t max_pages, int32_t n_rows, const int32_t* seq_lens,
                            const int32_t* q_offsets, const int32_t* row_kinds, void* o, void* workspace,
                            size_t workspace_bytes, mixattn_stream stream) {
  mixattn_plan* plan = nullptr;
  int st = mixattn_plan_create(&plan, cache, num_q_heads, n_rows, row_kinds, seq_lens, q_offsets, max_pages,
                               nullptr);
  if (st != MIXATTN_OK) return st;
  st = mixattn_run(plan, q, page_table, o, workspace, workspace_bytes, stream);
  mixattn_plan_destroy(plan);  // waits for the tile-list copy only
  return st;
}

int64_t mixattn_device_error(int32_t clear) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return MIXATTN_ERR_CUDA;
  if (clear) {
    const unsigned int z = 0;
    if (cudaMemcpyToSymbol(g_device_error, &z, sizeof(z)) != cudaSuccess) return MIXATTN_ERR_CUDA;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices && g_err_flag[dev])
      *g_err_flag[dev] = 0u;
  }
  return (int64_t)v;
}

const char* mixattn_status_string(int32_t status) {
  switch (status) {
    case MIXATTN_OK: return "ok";
    case MIXATTN_ERR_INVALID_ARG: return "invalid argument";
    case MIXATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case MIXATTN_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MIXATTN_ERR_CUDA: return "CUDA runtime error";
    case MIXATTN_ERR_DEVICE_CHECK: return "device-side check failed";
    case MIXATTN_ERR_CLIENT_QUOTA: return "client quota: too many requests waiting for this client";
    default: return "unknown status";
  }
}

int32_t mixattn_version(void) { return 100; }

}  // extern "C"
