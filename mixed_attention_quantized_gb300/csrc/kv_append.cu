// kv_append.cu -- quantise-on-append and canonical-block export.
//
// Page "自研RDNA高併發推論引擎 以AI Max+ 395為範例", §2 modes table: the cache
// holds 32-element blocks, q8 = one fp16 scale + 32 int8 (34 B), 4-bit =
// one fp16 scale + 16 bytes of nibbles (18 B); §2 states the blocked codec is
// bit-exact.  The block formulas are the GGUF Q8_0 / Q4_0 ones that page's
// engine reads:
//   Q8_0  d = amax / 127,     q = round(x / d)                  (half away)
//   Q4_0  d = m / -8,         q = min(15, trunc(x / d + 8.5))   m = signed max
// computed as x * (1/d) in fp32 with IEEE division, each product and sum
// rounded separately (no contraction), the stored scale rounded to fp16.
//
// Work split: one warp encodes four consecutive 32-element blocks; lane l owns
// elements 4(l%8) .. 4(l%8)+3 of block l/8, so every global load and every
// quant store of a warp is one contiguous, coalesced run.
#include <cuda_runtime.h>

#include "device_utils.cuh"
#include "internal.h"

namespace mixattn {

namespace {

struct AppendArgs {
  const uint16_t* x;     // fp16 [n_new][hkv][D]
  const int32_t* slots;  // [n_new]
  uint8_t* quant;        // [num_pages][hkv][32][row_bytes]
  uint16_t* scale;       // [num_pages][hkv][32][D/32]
  int64_t n_blocks;      // n_new * hkv * D/32
  int32_t hkv;
  int32_t nb;            // D / 32
  int32_t num_slots;     // num_pages * 32
  unsigned int* err;
};

__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }

template <int FMT>
__device__ __forceinline__ void encode_group(const AppendArgs& a, int64_t group, int lane) {
  const int64_t blk = group * 4 + (lane >> 3);
  const int sub = lane & 7;  // which 4 elements of the block
  const bool in_range = blk < a.n_blocks;
  int64_t b = 0, g = 0, t = 0;
  int32_t slot = -1;
  uint2 raw = make_uint2(0u, 0u);
  if (in_range) {
    b = blk % a.nb;
    const int64_t tg = blk / a.nb;
    g = tg % a.hkv;
    t = tg / a.hkv;
    slot = a.slots[t];
    raw = *reinterpret_cast<const uint2*>(a.x + blk * kBlock + 4 * sub);
  }
  if (slot >= a.num_slots) {
    if (sub == 0) set_device_error(a.err, MIXATTN_DEVERR_SLOT);
    slot = -1;
  }
  const float v[4] = {h2f(raw.x & 0xFFFFu), h2f(raw.x >> 16), h2f(raw.y & 0xFFFFu), h2f(raw.y >> 16)};
  // row of the slot in the [page][head][token] plane order
  const int64_t page = slot >= 0 ? slot / kPage : 0;
  const int64_t off = slot >= 0 ? slot % kPage : 0;
  const int64_t row = (page * a.hkv + g) * kPage + off;

  if constexpr (FMT == MIXATTN_KV_F16) {
    if (slot >= 0) {
      *reinterpret_cast<uint2*>(a.quant + row * (int64_t)(a.nb * 64) + b * 64 + 8 * sub) = raw;
    }
    return;
  } else if constexpr (FMT == MIXATTN_KV_Q8_0) {
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const float d = __fdiv_rn(amax, 127.0f);
    const float id = (d != 0.0f) ? __fdiv_rn(1.0f, d) : 0.0f;
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int q = (int)roundf(__fmul_rn(v[i], id));
      packed |= (uint32_t)(uint8_t)(int8_t)q << (8 * i);
    }
    if (slot >= 0) {
      *reinterpret_cast<uint32_t*>(a.quant + row * (int64_t)(a.nb * 32) + b * 32 + 4 * sub) = packed;
      if (sub == 0) a.scale[row * a.nb + b] = __half_as_ushort(__float2half_rn(d));
    }
  } else {  // Q4_0
    // element of largest magnitude, lowest index on ties
    float best_abs = -1.0f, best_val = 0.0f;
    int best_idx = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float m = fabsf(v[i]);
      if (m > best_abs) {
        best_abs = m;
        best_val = v[i];
        best_idx = 4 * sub + i;
      }
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      const float oa = __shfl_xor_sync(0xFFFFFFFFu, best_abs, o);
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, best_val, o);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, best_idx, o);
      if (oa > best_abs || (oa == best_abs && oi < best_idx)) {
        best_abs = oa;
        best_val = ov;
        best_idx = oi;
      }
    }
    const float m = best_abs > 0.0f ? best_val : 0.0f;  // an all-zero block keeps m = +0
    const float d = __fdiv_rn(m, -8.0f);
    const float id = (d != 0.0f) ? __fdiv_rn(1.0f, d) : 0.0f;
    uint32_t q4 = 0;  // four nibbles, one per byte
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float s = __fadd_rn(__fmul_rn(v[i], id), 8.5f);
      int q = (int)truncf(s);
      q = q > 15 ? 15 : q;
      q4 |= (uint32_t)q << (8 * i);
    }
    // element k (lanes 0-3 of the 8) pairs with element k+16 (lanes 4-7)
    const uint32_t hi = __shfl_down_sync(0xFFFFFFFFu, q4, 4);
    if (slot >= 0 && sub < 4) {
      *reinterpret_cast<uint32_t*>(a.quant + row * (int64_t)(a.nb * 16) + b * 16 + 4 * sub) = q4 | (hi << 4);
    }
    if (slot >= 0 && sub == 0) a.scale[row * a.nb + b] = __half_as_ushort(__float2half_rn(d));
  }
}

template <int FK, int FV>
__global__ void __launch_bounds__(256) kv_append_kernel(AppendArgs k, AppendArgs v, int64_t n_groups) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t gidx = warp; gidx < n_groups; gidx += n_warps) {
    if (blockIdx.y == 0) encode_group<FK>(k, gidx, lane);
    else encode_group<FV>(v, gidx, lane);
  }
}

struct ExportArgs {
  const uint8_t* quant;
  const uint16_t* scale;
  const int32_t* slots;
  uint8_t* out;
  int64_t n_items;  // n * hkv * nb
  int32_t hkv, nb, num_slots, fmt;
  unsigned int* err;
};

__global__ void __launch_bounds__(256) kv_export_kernel(ExportArgs a) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.n_items) return;
  const int64_t b = i % a.nb;
  const int64_t g = (i / a.nb) % a.hkv;
  const int64_t s = i / ((int64_t)a.nb * a.hkv);
  const int32_t slot = a.slots[s];
  const int bb = a.fmt == MIXATTN_KV_F16 ? 64 : (a.fmt == MIXATTN_KV_Q8_0 ? 34 : 18);
  uint8_t* dst = a.out + i * bb;
  if (slot < 0 || slot >= a.num_slots) {
    set_device_error(a.err, MIXATTN_DEVERR_SLOT);
    for (int j = 0; j < bb; ++j) dst[j] = 0;
    return;
  }
  const int64_t row = ((int64_t)(slot / kPage) * a.hkv + g) * kPage + slot % kPage;
  if (a.fmt == MIXATTN_KV_F16) {
    const uint8_t* src = a.quant + row * (int64_t)(a.nb * 64) + b * 64;
    for (int j = 0; j < 64; ++j) dst[j] = src[j];
    return;
  }
  const uint16_t d = a.scale[row * a.nb + b];
  dst[0] = (uint8_t)(d & 0xFFu);
  dst[1] = (uint8_t)(d >> 8);
  const int qb = a.fmt == MIXATTN_KV_Q8_0 ? 32 : 16;
  const uint8_t* src = a.quant + row * (int64_t)(a.nb * qb) + b * qb;
  for (int j = 0; j < qb; ++j) dst[2 + j] = src[j];
}

template <int FK>
cudaError_t launch_append_fk(int fv, dim3 grid, cudaStream_t s, const AppendArgs& k, const AppendArgs& v,
                             int64_t n_groups) {
  switch (fv) {
    case MIXATTN_KV_F16: kv_append_kernel<FK, MIXATTN_KV_F16><<<grid, 256, 0, s>>>(k, v, n_groups); break;
    case MIXATTN_KV_Q8_0: kv_append_kernel<FK, MIXATTN_KV_Q8_0><<<grid, 256, 0, s>>>(k, v, n_groups); break;
    default: kv_append_kernel<FK, MIXATTN_KV_Q4_0><<<grid, 256, 0, s>>>(k, v, n_groups); break;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_kv_append(const mixattn_kv_cache& c, const void* k_new, const void* v_new,
                             const int32_t* slots, int32_t n_new, unsigned int* err, cudaStream_t s) {
  AppendArgs k, v;
  const int nb = c.head_dim / kBlock;
  const int64_t n_blocks = (int64_t)n_new * c.num_kv_heads * nb;
  k.x = static_cast<const uint16_t*>(k_new);
  v.x = static_cast<const uint16_t*>(v_new);
  k.slots = v.slots = slots;
  k.quant = static_cast<uint8_t*>(c.k_quant);
  k.scale = static_cast<uint16_t*>(c.k_scale);
  v.quant = static_cast<uint8_t*>(c.v_quant);
  v.scale = static_cast<uint16_t*>(c.v_scale);
  k.n_blocks = v.n_blocks = n_blocks;
  k.hkv = v.hkv = c.num_kv_heads;
  k.nb = v.nb = nb;
  k.num_slots = v.num_slots = c.num_pages * kPage;
  k.err = v.err = err;
  const int64_t n_groups = (n_blocks + 3) / 4;
  int64_t blocks = (n_groups + 7) / 8;  // 8 warps per CTA
  if (blocks > 152 * 16) blocks = 152 * 16;
  dim3 grid((unsigned)blocks, 2);
  switch (c.k_fmt) {
    case MIXATTN_KV_F16: return launch_append_fk<MIXATTN_KV_F16>(c.v_fmt, grid, s, k, v, n_groups);
    case MIXATTN_KV_Q8_0: return launch_append_fk<MIXATTN_KV_Q8_0>(c.v_fmt, grid, s, k, v, n_groups);
    default: return launch_append_fk<MIXATTN_KV_Q4_0>(c.v_fmt, grid, s, k, v, n_groups);
  }
}

cudaError_t launch_kv_export(const mixattn_kv_cache& c, int which, const int32_t* slots, int32_t n, void* out,
                             unsigned int* err, cudaStream_t s) {
  ExportArgs a;
  a.fmt = which == 0 ? c.k_fmt : c.v_fmt;
  a.quant = static_cast<const uint8_t*>(which == 0 ? c.k_quant : c.v_quant);
  a.scale = static_cast<const uint16_t*>(which == 0 ? c.k_scale : c.v_scale);
  a.slots = slots;
  a.out = static_cast<uint8_t*>(out);
  a.hkv = c.num_kv_heads;
  a.nb = c.head_dim / kBlock;
  a.n_items = (int64_t)n * a.hkv * a.nb;
  a.num_slots = c.num_pages * kPage;
  a.err = err;
  const int64_t blocks = (a.n_items + 255) / 256;
  kv_export_kernel<<<(unsigned)blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace mixattn
