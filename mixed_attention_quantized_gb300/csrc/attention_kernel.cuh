// attention_kernel.cuh -- the mixed-batch attention step (one launch, two tile kinds).
//
// Page "自研RDNA高併發推論引擎 以AI Max+ 395為範例", §1 "統一 mixed-batch 介面":
// chunk rows and decode rows of one ForwardBatch go through one attention
// kernel, so the prefill tick also emits every due decode token.  For every
// query at position p of a row, q head h, kv head g = h / G:
//     o = sum_{j<=p} softmax_j(q . k^_j / sqrt(D)) v^_j
// over the dequantised cache values k^, v^ (§2 blocked formats).
//
// Decode tiles (HBM-bound, ~7.5 FLOP per byte): a CTA of 8 warps walks a page
// range of one (row, kv head).  Each warp keeps several 16-key M-tiles in
// flight through a cp.async ring in shared memory (16-byte chunks, 128-byte
// XOR swizzle so the fragment reads are conflict free) and runs QK^T and PV on
// mma.sync m16n8k16 with the G query heads in the N=8 dimension.  Quantised codes are
// turned into exact fp16 integers by a byte permute (no rounding); the Q8_0 /
// Q4_0 scales are applied in fp32: per key and 32-d block on the scores, and
// folded into P per key and block on the values.  Warp partials are merged in
// shared memory, split partials by the last CTA of the (row, kv head) to
// finish (atomic ticket, no spin).
//
// Chunk tiles (tensor-bound): a CTA of 16 warps owns 128 rows = 128/G query
// tokens x G heads of one kv head.  Two dequant warp groups load the raw K and V
// bytes straight from the cache and write 128-byte-swizzled fp16 operand tiles
// -- an exact hi/lo pair for quantised formats, since d*q needs up to 18
// significant bits; one thread issues every tcgen05.mma (S = Q K^T and O += P V,
// one MMA per half, Q, S, P and O in TMEM); a softmax warp group, one TMEM lane
// (query row) per thread, turns S into P.  K and S are double-buffered and P has
// its own columns, so QK of the next tile and the dequantisation overlap this
// tile's softmax and PV.
#pragma once

#include <algorithm>

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "device_utils.cuh"
#include "internal.h"

namespace mixattn {

// ===========================================================================
// Shared-memory plan of a chunk tile
// ===========================================================================
template <int FK, int FV, int D>
struct ChunkSmem {
  // quantised formats carry an exact low half: d*q = hi + lo, both fp16
  static constexpr bool kKLo = FK != MIXATTN_KV_F16;
  static constexpr bool kVLo = FV != MIXATTN_KV_F16;
  static constexpr int kTile = kChunkN * D * 2;             // one fp16 operand tile [D/64][128 keys][128 B]
  static constexpr int kKBuf = kTile * (kKLo ? 2 : 1);      // one K buffer: hi (+ lo)
  static constexpr int kK0 = 0;                             // K(j) lives in buffer j % 2
  static constexpr int kK1 = kKBuf;
  static constexpr int kVh = 2 * kKBuf;
  static constexpr int kVl = kVh + kTile;
  static constexpr int kBar = kVl + (kVLo ? kTile : 0);
  static constexpr int kBarBytes = 128;                     // mbarriers, TMEM address, abort flag
  static constexpr int kTotal = kBar + kBarBytes + 1024;   // + slack for 1024-B alignment
  static_assert(kTotal <= 227 * 1024, "chunk tile does not fit in shared memory");
};

// Staging ring of a decode warp: one stage = one M-tile (16 keys) of one page:
// the 16 contiguous K and V rows of the page plane, copied cooperatively in
// 16-byte chunks and placed with a 128-byte XOR swizzle (16-byte chunk index ^=
// 128-byte line index mod 8), so the fragment reads of every format are
// bank-conflict free; then the 16 keys' K and V scale rows.
template <int FK, int FV, int D>
struct DecodeSmem {
  static constexpr int kNb = D / kBlock;
  static constexpr int kRbK = FK == MIXATTN_KV_F16 ? 2 * D : (FK == MIXATTN_KV_Q8_0 ? D : D / 2);
  static constexpr int kRbV = FV == MIXATTN_KV_F16 ? 2 * D : (FV == MIXATTN_KV_Q8_0 ? D : D / 2);
  static constexpr int kSc = 16 * kNb * 2;  // 16 keys x D/32 fp16 scales
  static constexpr int kK = 0;
  static constexpr int kV = kK + 16 * kRbK;
  static constexpr int kKs = kV + 16 * kRbV;
  static constexpr int kVs = kKs + (FK == MIXATTN_KV_F16 ? 0 : kSc);
  static constexpr int kStage = (kVs + (FV == MIXATTN_KV_F16 ? 0 : kSc) + 127) / 128 * 128;
  static constexpr int stages_for(int budget) {
    return budget / (kWarps * kStage) > 8 ? 8 : (budget / (kWarps * kStage) < 2 ? 2 : budget / (kWarps * kStage));
  }
  // after the page loop the same memory holds the warp partials: m[8], l[8], O[8][D]
  static constexpr int kPerWarp = 16 + kMaxGroup * D;
  static constexpr int kMerge = kWarps * kPerWarp * 4;
  static constexpr int total(int ns) { return (kWarps * ns * kStage > kMerge ? kWarps * ns * kStage : kMerge) + 16; }
  // decode-only launches: two CTAs per SM when two stages per warp fit in ~106 KB,
  // else one CTA per SM with a deeper ring
  static constexpr int kPairBudget = 106 * 1024;
  static constexpr bool kTwoPerSm = kWarps * 2 * kStage <= kPairBudget;
  static constexpr int kSoloStages = stages_for(kTwoPerSm ? kPairBudget : 212 * 1024);
  static constexpr int kSoloMinBlocks = kTwoPerSm ? 2 : 1;
  static constexpr int kTotal = total(kSoloStages);
  static_assert(kTotal <= 227 * 1024, "decode staging does not fit in shared memory");
};

// 128-byte XOR swizzle of a byte offset inside a staged region.
__device__ __forceinline__ int swz(int o) { return o ^ (((o >> 7) & 7) << 4); }

// ===========================================================================
// Decode tiles
// ===========================================================================

template <int F, int D>
__device__ __forceinline__ constexpr int row_bytes() {
  return F == MIXATTN_KV_F16 ? 2 * D : (F == MIXATTN_KV_Q8_0 ? D : D / 2);
}

// Physical head dimension d held by lane row `rr` (0..15) of PV M-tile t,
// for the V format's fragment layout.
template <int FV>
__device__ __forceinline__ int pv_row_to_d(int t, int rr) {
  const int b = t >> 1, u = t & 1, r = rr & 7, hi = rr >> 3;
  if (FV == MIXATTN_KV_Q4_0) return 32 * b + 16 * u + 2 * r + hi;
  return 32 * b + 4 * r + 2 * u + hi;
}

__device__ __forceinline__ void unpack_scales(uint2 a, float* out) {
  out[0] = __half2float(__ushort_as_half(a.x & 0xFFFF));
  out[1] = __half2float(__ushort_as_half(a.x >> 16));
  out[2] = __half2float(__ushort_as_half(a.y & 0xFFFF));
  out[3] = __half2float(__ushort_as_half(a.y >> 16));
}

template <int NB>
__device__ __forceinline__ void load_scales(const uint8_t* p, float (&out)[NB]) {
  if (NB == 4) {
    float t[4];
    unpack_scales(lds64(p), t);
#pragma unroll
    for (int i = 0; i < NB; ++i) out[i] = t[i];
  } else {
    const uint32_t a = lds32(p);
    out[0] = __half2float(__ushort_as_half(a & 0xFFFF));
    out[NB - 1] = __half2float(__ushort_as_half(a >> 16));
  }
}

// Barrier over the 8 warps of a decode tile (a fused-launch CTA runs one tile
// on each half of its 16 warps, each half on its own named barrier).
__device__ __forceinline__ void decode_sync(int half) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + half), "n"(kThreads) : "memory");
}

template <int FK, int FV, int D, int NS>
__device__ __forceinline__ void decode_tile(const AttnParams& p, const TileDesc& t, int dec_idx, uint8_t* smem,
                                            unsigned int* err, int half) {
  using S = DecodeSmem<FK, FV, D>;
  constexpr int NB = D / kBlock;   // scale blocks per row
  constexpr int KS = D / 16;       // k-steps of QK / M-tiles of PV
  constexpr int RBK = row_bytes<FK, D>();
  constexpr int RBV = row_bytes<FV, D>();

  // `half`: which 8 warps of the CTA run this tile (a fused-launch CTA runs two)
  const int tid = threadIdx.x - half * kThreads, warp = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, c = lane & 3;
  const int G = p.group;
  const int g = t.kvh;
  const RowInfo ri = p.rows[t.row];
  const int n_pages_row = (ri.seq_len + kPage - 1) / kPage;
  const int ppw = decode_pages_per_warp(n_pages_row);
  const int pps = kWarps * ppw;
  const int split = t.begin / pps;
  const int wp0 = t.begin + warp * ppw;
  const int wp1 = min(t.begin + t.count, wp0 + ppw);
  const int n_mt = wp1 > wp0 ? 2 * (wp1 - wp0) : 0;  // the warp's M-tiles (16 keys each)

  // ---- Q as the A operand of S = Q K^T: head r in M row r (rows 8..15 zero) ----
  // k-slots 2c,2c+1 | 2c+8,2c+9 of k-step 2b+hs hold head dims
  //   Q8_0 / fp16: 32b+8c+4hs + {0,1 | 2,3};   Q4_0: 32b+16hs+4c + {0,1 | 2,3}
  uint32_t qa[KS][2];
  {
    const bool real = r < G;
    const uint16_t* qrow =
        static_cast<const uint16_t*>(p.q) + ((int64_t)ri.q_start * p.hq + (int64_t)g * G + (real ? r : 0)) * D;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      if (FK == MIXATTN_KV_Q4_0) {
        uint2 lo = real ? ldg_u64(qrow + 32 * b + 4 * c) : make_uint2(0u, 0u);
        uint2 hi = real ? ldg_u64(qrow + 32 * b + 16 + 4 * c) : make_uint2(0u, 0u);
        qa[2 * b][0] = lo.x;
        qa[2 * b][1] = lo.y;
        qa[2 * b + 1][0] = hi.x;
        qa[2 * b + 1][1] = hi.y;
      } else {
        uint4 v = real ? ldg_u128(qrow + 32 * b + 8 * c) : make_uint4(0u, 0u, 0u, 0u);
        qa[2 * b][0] = v.x;
        qa[2 * b][1] = v.y;
        qa[2 * b + 1][0] = v.z;
        qa[2 * b + 1][1] = v.w;
      }
    }
  }

  float o_acc[KS][4];
#pragma unroll
  for (int i = 0; i < KS; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
  float m_run = -CUDART_INF_F, l_run = 0.f;  // head r
  const float sl2 = p.scale_log2;

  const uint8_t* kq_base = p.k_quant + (int64_t)g * kPage * RBK;
  const uint8_t* vq_base = p.v_quant + (int64_t)g * kPage * RBV;
  const uint8_t* ks_base = reinterpret_cast<const uint8_t*>(p.k_scale) + (int64_t)g * kPage * NB * 2;
  const uint8_t* vs_base = reinterpret_cast<const uint8_t*>(p.v_scale) + (int64_t)g * kPage * NB * 2;
  const int64_t kq_page_stride = (int64_t)p.hkv * kPage * RBK;
  const int64_t vq_page_stride = (int64_t)p.hkv * kPage * RBV;
  const int64_t sc_page_stride = (int64_t)p.hkv * kPage * NB * 2;
  const int32_t* pt_row = p.page_table + (int64_t)t.row * p.max_pages;
  uint8_t* ring = smem + warp * NS * S::kStage;

  // Issue the copies of the warp's M-tile i into its stage, then close the group
  // (an empty group for i past the end keeps the group count uniform).
  auto issue = [&](int i) {
    if (i < n_mt) {
      const int pg = wp0 + (i >> 1), mt = i & 1;
      const int pid = pt_row[pg];
      if (pid >= 0 && pid < p.num_pages) {
        uint8_t* st = ring + (i % NS) * S::kStage;
        const uint8_t* kq = kq_base + (int64_t)pid * kq_page_stride + 16 * mt * RBK;
        const uint8_t* vq = vq_base + (int64_t)pid * vq_page_stride + 16 * mt * RBV;
#pragma unroll
        for (int j = lane; j < RBK; j += 32) cp_async16(st + S::kK + swz(16 * j), kq + 16 * j);
#pragma unroll
        for (int j = lane; j < RBV; j += 32) cp_async16(st + S::kV + swz(16 * j), vq + 16 * j);
        constexpr int SC = S::kSc / 16;  // 16-byte chunks of one scale slice
        if (FK != MIXATTN_KV_F16 && lane < SC)
          cp_async16(st + S::kKs + 16 * lane, ks_base + (int64_t)pid * sc_page_stride + 16 * mt * NB * 2 + 16 * lane);
        if (FV != MIXATTN_KV_F16 && lane >= 16 && lane < 16 + SC)
          cp_async16(st + S::kVs + 16 * (lane - 16),
                     vs_base + (int64_t)pid * sc_page_stride + 16 * mt * NB * 2 + 16 * (lane - 16));
      } else if (lane == 0 && (i & 1) == 0) {
        set_device_error(err, MIXATTN_DEVERR_PAGE_ID);
      }
    }
    cp_async_commit();
  };

#pragma unroll
  for (int i = 0; i < NS - 1; ++i) issue(i);

  const int kv0 = 2 * c;  // the lane's keys in an M-tile: kv0, kv0+1 (n-tile 0), kv0+8, kv0+9 (n-tile 1)
  for (int i = 0; i < n_mt; ++i) {
    issue(i + NS - 1);        // refills the stage consumed in the previous step
    cp_async_wait<NS - 1>();  // this lane's copies of M-tile i have landed
    __syncwarp();             // ... and every other lane's
    const int pg = wp0 + (i >> 1), mt = i & 1;
    const int pid = pt_row[pg];
    if (pid >= 0 && pid < p.num_pages) {
      const uint8_t* st = ring + (i % NS) * S::kStage;
      const int key0 = pg * kPage + 16 * mt;  // first key of the M-tile
      const bool partial = key0 + 16 > ri.seq_len;

      // ---------------- S = Q K^T: head r x keys kv0, kv0+1, kv0+8, kv0+9 ----------------
      float s[4] = {0.f, 0.f, 0.f, 0.f};
      float dk0[NB], dk1[NB], dk8[NB], dk9[NB];
      if (FK != MIXATTN_KV_F16) {
        load_scales<NB>(st + S::kKs + kv0 * NB * 2, dk0);
        load_scales<NB>(st + S::kKs + (kv0 + 1) * NB * 2, dk1);
        load_scales<NB>(st + S::kKs + (kv0 + 8) * NB * 2, dk8);
        load_scales<NB>(st + S::kKs + (kv0 + 9) * NB * 2, dk9);
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const uint8_t* kd = st + S::kK;
        uint32_t b0[2][2], b1[2][2];  // B fragments [n-tile][reg] of k-steps 2b and 2b+1 (keys r, r+8)
        if (FK == MIXATTN_KV_Q8_0) {
          const uint2 wl = lds64(kd + swz(r * RBK + 32 * b + 8 * c));
          const uint2 wh = lds64(kd + swz((r + 8) * RBK + 32 * b + 8 * c));
          s8x4_to_f16x2x2(wl.x, b0[0][0], b0[0][1]);
          s8x4_to_f16x2x2(wh.x, b0[1][0], b0[1][1]);
          s8x4_to_f16x2x2(wl.y, b1[0][0], b1[0][1]);
          s8x4_to_f16x2x2(wh.y, b1[1][0], b1[1][1]);
        } else if (FK == MIXATTN_KV_Q4_0) {
          const uint32_t yl = lds32(kd + swz(r * RBK + 16 * b + 4 * c));
          const uint32_t yh = lds32(kd + swz((r + 8) * RBK + 16 * b + 4 * c));
          u4x4_to_f16x2x2(yl & 0x0F0F0F0Fu, b0[0][0], b0[0][1]);
          u4x4_to_f16x2x2(yh & 0x0F0F0F0Fu, b0[1][0], b0[1][1]);
          u4x4_to_f16x2x2((yl >> 4) & 0x0F0F0F0Fu, b1[0][0], b1[0][1]);
          u4x4_to_f16x2x2((yh >> 4) & 0x0F0F0F0Fu, b1[1][0], b1[1][1]);
        } else {
          const uint4 wl = lds128(kd + swz(r * RBK + 2 * (32 * b + 8 * c)));
          const uint4 wh = lds128(kd + swz((r + 8) * RBK + 2 * (32 * b + 8 * c)));
          b0[0][0] = wl.x; b0[0][1] = wl.y; b0[1][0] = wh.x; b0[1][1] = wh.y;
          b1[0][0] = wl.z; b1[0][1] = wl.w; b1[1][0] = wh.z; b1[1][1] = wh.w;
        }
        const uint32_t a0[4] = {qa[2 * b][0], 0u, qa[2 * b][1], 0u};
        const uint32_t a1[4] = {qa[2 * b + 1][0], 0u, qa[2 * b + 1][1], 0u};
        if (FK == MIXATTN_KV_F16) {
          float u0[4], u1[4];
          mma_16816_c(u0, a0, b0[0], s[0], s[1], 0.f, 0.f);
          mma_16816(u0, a1, b1[0]);
          mma_16816_c(u1, a0, b0[1], s[2], s[3], 0.f, 0.f);
          mma_16816(u1, a1, b1[1]);
          s[0] = u0[0]; s[1] = u0[1]; s[2] = u1[0]; s[3] = u1[1];
        } else {
          float u0[4], u1[4];  // per-block dot products of exact integer codes
          mma_16816_c(u0, a0, b0[0], 0.f, 0.f, 0.f, 0.f);
          mma_16816(u0, a1, b1[0]);
          mma_16816_c(u1, a0, b0[1], 0.f, 0.f, 0.f, 0.f);
          mma_16816(u1, a1, b1[1]);
          s[0] = fmaf(dk0[b], u0[0], s[0]);
          s[1] = fmaf(dk1[b], u0[1], s[1]);
          s[2] = fmaf(dk8[b], u1[0], s[2]);
          s[3] = fmaf(dk9[b], u1[1], s[3]);
        }
      }

      // ---------------- online softmax over the 16 keys (head r) ----------------
      s[0] = key0 + kv0 < ri.seq_len ? s[0] * sl2 : -CUDART_INF_F;
      s[1] = key0 + kv0 + 1 < ri.seq_len ? s[1] * sl2 : -CUDART_INF_F;
      s[2] = key0 + kv0 + 8 < ri.seq_len ? s[2] * sl2 : -CUDART_INF_F;
      s[3] = key0 + kv0 + 9 < ri.seq_len ? s[3] * sl2 : -CUDART_INF_F;
      float pm = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
      pm = fmaxf(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, 1));
      pm = fmaxf(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, 2));
      // exact running max: the largest weight is exactly 1, so its fp16 P' is exact
      float alpha = 1.f;
      if (pm > m_run) {  // also the first M-tile with a valid key (m_run = -inf)
        alpha = ex2(m_run - pm);
        m_run = pm;
      }
      const float mref = m_run == -CUDART_INF_F ? 0.f : m_run;
      const float p0 = ex2(s[0] - mref), p1 = ex2(s[1] - mref);
      const float p8 = ex2(s[2] - mref), p9 = ex2(s[3] - mref);
      l_run = l_run * alpha + ((p0 + p1) + (p8 + p9));
      if (__any_sync(0xFFFFFFFFu, alpha != 1.f)) {
        // O columns are heads 2c, 2c+1: their factors live in lanes 8c and 8c+4
        const float a_even = __shfl_sync(0xFFFFFFFFu, alpha, 8 * c);
        const float a_odd = __shfl_sync(0xFFFFFFFFu, alpha, 8 * c + 4);
#pragma unroll
        for (int i2 = 0; i2 < KS; ++i2) {
          o_acc[i2][0] *= a_even;
          o_acc[i2][1] *= a_odd;
          o_acc[i2][2] *= a_even;
          o_acc[i2][3] *= a_odd;
        }
      }

      // ---------------- O^T += V^T P for the 16 keys ----------------
      // P is already in the B-operand layout: this lane holds P[key kv0.., kv0+9][head r].
      uint32_t bfr[NB][2];
      if (FV == MIXATTN_KV_F16) {
        bfr[0][0] = pack_f16x2(p0, p1);
        bfr[0][1] = pack_f16x2(p8, p9);
      } else {
        float dv0[NB], dv1[NB], dv8[NB], dv9[NB];
        load_scales<NB>(st + S::kVs + kv0 * NB * 2, dv0);
        load_scales<NB>(st + S::kVs + (kv0 + 1) * NB * 2, dv1);
        load_scales<NB>(st + S::kVs + (kv0 + 8) * NB * 2, dv8);
        load_scales<NB>(st + S::kVs + (kv0 + 9) * NB * 2, dv9);
        if (partial) {
          // p == 0 (a key past the row) stays 0 whatever its scale slot holds
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            bfr[b][0] = pack_f16x2(p0 != 0.f ? p0 * dv0[b] : 0.f, p1 != 0.f ? p1 * dv1[b] : 0.f);
            bfr[b][1] = pack_f16x2(p8 != 0.f ? p8 * dv8[b] : 0.f, p9 != 0.f ? p9 * dv9[b] : 0.f);
          }
        } else {
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            bfr[b][0] = pack_f16x2(p0 * dv0[b], p1 * dv1[b]);
            bfr[b][1] = pack_f16x2(p8 * dv8[b], p9 * dv9[b]);
          }
        }
      }

#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const uint8_t* vd = st + S::kV;
        uint32_t a_u0[4], a_u1[4];  // A fragments of PV M-tiles 2b (u=0) and 2b+1 (u=1)
        const uint32_t* bb = (FV == MIXATTN_KV_F16) ? bfr[0] : bfr[b];
        if (FV == MIXATTN_KV_Q8_0) {
          uint4 w;
          w.x = lds32(vd + swz(kv0 * RBV + 32 * b + 4 * r));
          w.y = lds32(vd + swz((kv0 + 1) * RBV + 32 * b + 4 * r));
          w.z = lds32(vd + swz((kv0 + 8) * RBV + 32 * b + 4 * r));
          w.w = lds32(vd + swz((kv0 + 9) * RBV + 32 * b + 4 * r));
          s8x4_to_f16x2x2(prmt(w.x, w.y, 0x5140u), a_u0[0], a_u0[1]);
          s8x4_to_f16x2x2(prmt(w.z, w.w, 0x5140u), a_u0[2], a_u0[3]);
          s8x4_to_f16x2x2(prmt(w.x, w.y, 0x7362u), a_u1[0], a_u1[1]);
          s8x4_to_f16x2x2(prmt(w.z, w.w, 0x7362u), a_u1[2], a_u1[3]);
        } else if (FV == MIXATTN_KV_Q4_0) {
          // the 4 bytes holding the lane's 2 bytes (block bytes 2r, 2r+1) at half (r & 1)
          uint4 w;
          w.x = lds32(vd + swz(kv0 * RBV + 16 * b + 4 * (r >> 1)));
          w.y = lds32(vd + swz((kv0 + 1) * RBV + 16 * b + 4 * (r >> 1)));
          w.z = lds32(vd + swz((kv0 + 8) * RBV + 16 * b + 4 * (r >> 1)));
          w.w = lds32(vd + swz((kv0 + 9) * RBV + 16 * b + 4 * (r >> 1)));
          const uint32_t sel = (r & 1) ? 0x7362u : 0x5140u;
          const uint32_t x01 = prmt(w.x, w.y, sel), x89 = prmt(w.z, w.w, sel);
          u4x4_to_f16x2x2(x01 & 0x0F0F0F0Fu, a_u0[0], a_u0[1]);
          u4x4_to_f16x2x2(x89 & 0x0F0F0F0Fu, a_u0[2], a_u0[3]);
          u4x4_to_f16x2x2((x01 >> 4) & 0x0F0F0F0Fu, a_u1[0], a_u1[1]);
          u4x4_to_f16x2x2((x89 >> 4) & 0x0F0F0F0Fu, a_u1[2], a_u1[3]);
        } else {
          // fp16 values: zero the words of keys past the row so stale data never reaches the MMA
          const bool ok0 = key0 + kv0 < ri.seq_len, ok1 = key0 + kv0 + 1 < ri.seq_len;
          const bool ok8 = key0 + kv0 + 8 < ri.seq_len, ok9 = key0 + kv0 + 9 < ri.seq_len;
          const int vo = 2 * (32 * b + 4 * r);
          const uint2 e0 = ok0 ? lds64(vd + swz(kv0 * RBV + vo)) : make_uint2(0u, 0u);
          const uint2 e1 = ok1 ? lds64(vd + swz((kv0 + 1) * RBV + vo)) : make_uint2(0u, 0u);
          const uint2 e8 = ok8 ? lds64(vd + swz((kv0 + 8) * RBV + vo)) : make_uint2(0u, 0u);
          const uint2 e9 = ok9 ? lds64(vd + swz((kv0 + 9) * RBV + vo)) : make_uint2(0u, 0u);
          a_u0[0] = prmt(e0.x, e1.x, 0x5410u);
          a_u0[1] = prmt(e0.x, e1.x, 0x7632u);
          a_u0[2] = prmt(e8.x, e9.x, 0x5410u);
          a_u0[3] = prmt(e8.x, e9.x, 0x7632u);
          a_u1[0] = prmt(e0.y, e1.y, 0x5410u);
          a_u1[1] = prmt(e0.y, e1.y, 0x7632u);
          a_u1[2] = prmt(e8.y, e9.y, 0x5410u);
          a_u1[3] = prmt(e8.y, e9.y, 0x7632u);
        }
        const uint32_t bop[2] = {bb[0], bb[1]};
        mma_16816(o_acc[2 * b], a_u0, bop);
        mma_16816(o_acc[2 * b + 1], a_u1, bop);
      }
    }
    __syncwarp();  // every lane is done with this stage before it is refilled
  }
  cp_async_wait<0>();

  // ---------------- warp partial -> shared memory ----------------
  l_run += __shfl_xor_sync(0xFFFFFFFFu, l_run, 1);
  l_run += __shfl_xor_sync(0xFFFFFFFFu, l_run, 2);
  decode_sync(half);  // the staging rings are no longer needed: reuse them as merge scratch
  float* ws = reinterpret_cast<float*>(smem);
  float* wm = ws + warp * S::kPerWarp;  // m[8], l[8], O[8][D]
  const int h0 = 2 * c, h1 = 2 * c + 1;
  if (c == 0 && r < G) {
    wm[r] = m_run;
    wm[8 + r] = l_run;
  }
#pragma unroll
  for (int tt = 0; tt < KS; ++tt) {
    const int d_lo = pv_row_to_d<FV>(tt, r), d_hi = pv_row_to_d<FV>(tt, r + 8);
    if (h0 < G) {
      wm[16 + h0 * D + d_lo] = o_acc[tt][0];
      wm[16 + h0 * D + d_hi] = o_acc[tt][2];
    }
    if (h1 < G) {
      wm[16 + h1 * D + d_lo] = o_acc[tt][1];
      wm[16 + h1 * D + d_hi] = o_acc[tt][3];
    }
  }
  decode_sync(half);

  // ---------------- merge the 8 warps ----------------
  const int n_out = G * D;
  const int n_warps_used = min(kWarps, (t.count + ppw - 1) / ppw);
  const bool single = ri.n_splits == 1;
  float* part = p.partials + (int64_t)dec_idx * G * (D + 2);
  for (int idx = tid; idx < n_out; idx += kThreads) {
    const int h = idx / D, d = idx - h * D;
    float mmax = -CUDART_INF_F;
    for (int w = 0; w < n_warps_used; ++w) mmax = fmaxf(mmax, ws[w * S::kPerWarp + h]);
    float lsum = 0.f, osum = 0.f;
    for (int w = 0; w < n_warps_used; ++w) {
      const float* x = ws + w * S::kPerWarp;
      const float sc = x[h] == -CUDART_INF_F ? 0.f : ex2(x[h] - mmax);
      lsum += sc * x[8 + h];
      osum += sc * x[16 + h * D + d];
    }
    if (single) {
      uint16_t* dst = static_cast<uint16_t*>(p.o) + ((int64_t)ri.q_start * p.hq + (int64_t)g * G + h) * D + d;
      *dst = __half_as_ushort(__float2half_rn(osum / lsum));
    } else {
      part[h * D + d] = osum;
      if (d == 0) {
        part[G * D + 2 * h] = mmax;
        part[G * D + 2 * h + 1] = lsum;
      }
    }
  }
  if (single) return;

  // ---------------- last CTA of (row, kv head) merges the splits ----------------
  __threadfence();
  decode_sync(half);
  __shared__ int s_last_of[2];
  int& s_last = s_last_of[half];
  if (tid == 0) {
    const unsigned prev = atomicAdd(&p.counters[(int64_t)t.row * p.hkv + g], 1u);
    s_last = (prev == (unsigned)(ri.n_splits - 1));
  }
  decode_sync(half);
  if (!s_last) return;
  __threadfence();
  const int first = dec_idx - split;
  const int ns = ri.n_splits;
  for (int idx = tid; idx < n_out; idx += kThreads) {
    const int h = idx / D, d = idx - h * D;
    float mmax = -CUDART_INF_F;
    for (int s2 = 0; s2 < ns; ++s2) {
      const float* x = p.partials + (int64_t)(first + s2) * G * (D + 2);
      mmax = fmaxf(mmax, __ldcg(x + G * D + 2 * h));
    }
    float lsum = 0.f, osum = 0.f;
    for (int s2 = 0; s2 < ns; ++s2) {
      const float* x = p.partials + (int64_t)(first + s2) * G * (D + 2);
      const float mx = __ldcg(x + G * D + 2 * h);
      const float sc = mx == -CUDART_INF_F ? 0.f : ex2(mx - mmax);
      lsum += sc * __ldcg(x + G * D + 2 * h + 1);
      osum += sc * __ldcg(x + h * D + d);
    }
    uint16_t* dst = static_cast<uint16_t*>(p.o) + ((int64_t)ri.q_start * p.hq + (int64_t)g * G + h) * D + d;
    *dst = __half_as_ushort(__float2half_rn(osum / lsum));
  }
}

// ===========================================================================
// Chunk tiles
// ===========================================================================

// Byte offset of 16-byte chunk `cc` (0..7) of row `row` in a 128-byte-swizzled
// tile of 128-byte rows (1024-byte atoms of 8 rows).
__device__ __forceinline__ uint32_t sw128_off(int row, int cc) {
  return (uint32_t)(row * 128 + ((cc ^ (row & 7)) << 4));
}

// v holds exact small integers (f16x2), s the fp16 scale in both halves.
// hi = fp16(v*s); lo = v*s - hi, which is exact in fp16: v*s has at most
// 18 significant bits, hi keeps the top 11, and the residual is a multiple of
// the scale's ulp (>= 2^-24) below 2^8 of them.  So hi + lo == v*s exactly.
__device__ __forceinline__ void split_hilo(uint32_t v, uint32_t s, uint32_t& hi, uint32_t& lo) {
  hi = hmul2_u32(v, s);
  lo = hfma2_u32(v, s, hneg2_u32(hi));  // the negation folds into the fma
}

// Dequantisation of the chunk path.  Thread t0 (0..127) of a dequant group owns
// one 16-byte output column chunk, dc = t0 % (D/8), of the keys
// key0 + i * KPI, key0 = t0 / (D/8): KPI is a multiple of 8, so the swizzle term
// (key & 7) is fixed per thread.  A key half (64 keys, pages 2h and 2h+1 of the
// tile) gives each thread NH keys: the first NH/2 in page 2h, the rest in page
// 2h+1.  Its raw bytes are loaded from the cache planes into registers one half
// ahead of their conversion.
template <int F, int D>
struct DequantGeom {
  static constexpr int NB = D / kBlock;
  static constexpr int CPR = D / 8;                 // 16-byte fp16 chunks per key row
  static constexpr int KPI = 128 / CPR;             // keys between a thread's keys (8 or 16)
  static constexpr int NH = kChunkN / 2 / KPI;      // keys per thread per half (8 or 4)
  static constexpr int RB = F == MIXATTN_KV_F16 ? 2 * D : (F == MIXATTN_KV_Q8_0 ? D : D / 2);  // row bytes
  static_assert(KPI % 8 == 0 && NH % 2 == 0 && (NH / 2) * KPI == kPage, "key half layout");
};

constexpr int kNoPage = -2147483647 - 1;  // page id of a page past a row's key range

// Raw bytes of one key half for one thread.
template <int F, int D>
struct HalfRaw {
  static constexpr int NH = DequantGeom<F, D>::NH;
  uint4 q[NH];     // fp16: the 8 values; Q8_0: 8 bytes in .x/.y; Q4_0: 8 bytes holding 16 nibbles
  uint32_t s[NH];  // quantised formats: the block's fp16 scale (low 16 bits)
};

// Load the raw bytes of key half h of a tile for thread t0.  `pa`, `pb` are the
// ids of the half's two pages (kNoPage: past the key range), `valid` the number of its keys that
// exist (keys past it, and keys of a missing page, read as zeros).
template <int F, int D>
__device__ __forceinline__ void load_half(HalfRaw<F, D>& r, const uint8_t* __restrict__ q_plane,
                                          const uint16_t* __restrict__ s_plane, int pa, int pb, int num_pages,
                                          int hkv, int g, int valid, int t0, unsigned int* err) {
  using Gm = DequantGeom<F, D>;
  const int dc = t0 % Gm::CPR, key0 = t0 / Gm::CPR;
  const int b = dc >> 2;
  int src_col;
  if (F == MIXATTN_KV_F16) src_col = 16 * dc;
  else if (F == MIXATTN_KV_Q8_0) src_col = 8 * dc;
  else src_col = 16 * b + 8 * (dc & 1);
  const bool bad_a = pa != kNoPage && (pa < 0 || pa >= num_pages);
  const bool bad_b = pb != kNoPage && (pb < 0 || pb >= num_pages);
  if (bad_a || bad_b) {  // a page of the key range with an id outside the cache
    set_device_error(err, MIXATTN_DEVERR_PAGE_ID);
    if (bad_a) pa = kNoPage;
    if (bad_b) pb = kNoPage;
  }
  // first plane row of this thread's keys in each page; key i then sits a
  // compile-time number of rows further
  const int64_t row_a = ((int64_t)(pa >= 0 ? pa : 0) * hkv + g) * kPage + key0;
  const int64_t row_b = ((int64_t)(pb >= 0 ? pb : 0) * hkv + g) * kPage + key0 - kPage;
  const uint8_t* qa = q_plane + row_a * Gm::RB + src_col;
  const uint8_t* qb = q_plane + row_b * Gm::RB + src_col;
  const uint16_t* sa = s_plane + row_a * Gm::NB + b;
  const uint16_t* sb = s_plane + row_b * Gm::NB + b;
#pragma unroll
  for (int i = 0; i < Gm::NH; ++i) {
    const bool first = i < Gm::NH / 2;
    const bool ok = (first ? pa : pb) >= 0 && key0 + i * Gm::KPI < valid;
    // predicated loads: nothing here waits for the data (it is used a half later)
    if (F == MIXATTN_KV_F16) {
      r.q[i] = ldg_u128_pred((first ? qa : qb) + i * Gm::KPI * Gm::RB, ok);
    } else {
      const uint2 x = ldg_u64_pred((first ? qa : qb) + i * Gm::KPI * Gm::RB, ok);
      r.q[i].x = x.x;
      r.q[i].y = x.y;
      r.s[i] = ldg_u16_pred((first ? sa : sb) + i * Gm::KPI * Gm::NB, ok);
    }
  }
}

// Convert the raw bytes of key half h (loaded by load_half) into the swizzled
// fp16 operand tile: hi, and the exact lo for quantised formats.
template <int F, int D, bool LO>
__device__ __forceinline__ void convert_half(const HalfRaw<F, D>& r, uint8_t* __restrict__ dst_hi,
                                             uint8_t* __restrict__ dst_lo, int h, int t0) {
  using Gm = DequantGeom<F, D>;
  const int dc = t0 % Gm::CPR, key0 = t0 / Gm::CPR;
  const int half = dc >> 3, cc = dc & 7;
  const int shift = F == MIXATTN_KV_Q4_0 ? ((dc >> 1) & 1) * 4 : 0;  // low nibbles, then high nibbles
  const int kh = key0 + kChunkN / 2 * h;
  const uint32_t doff = (uint32_t)(half * (kChunkN * 128) + kh * 128 + ((cc ^ (key0 & 7)) << 4));
#pragma unroll
  for (int i = 0; i < Gm::NH; ++i) {
    uint4 hi, lo = make_uint4(0u, 0u, 0u, 0u);
    if (F == MIXATTN_KV_F16) {
      hi = r.q[i];
    } else {
      const uint32_t sc = prmt(r.s[i], 0u, 0x1010u);  // the scale in both halves
      uint32_t h0, h1, h2, h3;
      if (F == MIXATTN_KV_Q8_0) {
        s8x4_to_f16x2x2(r.q[i].x, h0, h1);
        s8x4_to_f16x2x2(r.q[i].y, h2, h3);
      } else {
        u4x4_to_f16x2x2((r.q[i].x >> shift) & 0x0F0F0F0Fu, h0, h1);
        u4x4_to_f16x2x2((r.q[i].y >> shift) & 0x0F0F0F0Fu, h2, h3);
      }
      split_hilo(h0, sc, hi.x, lo.x);
      split_hilo(h1, sc, hi.y, lo.y);
      split_hilo(h2, sc, hi.z, lo.z);
      split_hilo(h3, sc, hi.w, lo.w);
    }
    *reinterpret_cast<uint4*>(dst_hi + doff + i * Gm::KPI * 128) = hi;
    if (LO) *reinterpret_cast<uint4*>(dst_lo + doff + i * Gm::KPI * 128) = lo;
  }
}

// The loop of one dequant group over the KV tiles of one chunk tile (one
// out-of-line copy per format serves the K and the V group, which then share
// instruction-cache lines).  Buffers and barrier phases follow the CTA's running
// KV-tile count jg = jg0 + j, which continues across the CTA's chunk tiles.
//   K group: K(jg) goes to buffer jg % 2 (hi at dst_hi[jg%2], lo at
//     dst_lo[jg%2]) once QK(jg-2) has released it (qk_done[jg%2]); after both
//     halves it arrives on ready[jg%2].
//   V group: V(jg) goes to the single buffer, half h once the PV MMAs of tile
//     jg-1 that read that half are done (pvh_done[h]); it arrives on ready[h]
//     after each half.
// Returns false when the group left early (a timeout here or elsewhere).
template <int F, int D, bool LO>
__device__ __noinline__ bool dequant_loop(const uint8_t* __restrict__ q_plane, const uint16_t* __restrict__ s_plane,
                                          const int32_t* __restrict__ pt_row, int n_pages_row, int num_pages,
                                          int hkv, int g, int key_end, int n_kv, int jg0, int t0, bool is_k,
                                          uint8_t* dst_hi0, uint8_t* dst_lo0, uint8_t* dst_hi1, uint8_t* dst_lo1,
                                          uint64_t* free_bars, uint64_t* ready, int bar_id,
                                          volatile int* abort_flag, unsigned int* err) {
  bool ok = true;
  // page ids of key half (j, h); the bounds check happens at load time
  auto pid_of = [&](int pg) { return ldg_s32_or(pt_row + pg, pg < n_pages_row && pg * kPage < key_end, kNoPage); };
  auto valid_of = [&](int j, int h) { return key_end - j * kChunkN - h * (kChunkN / 2); };
  // one half: wait until its destination is free, convert, publish
  // buffers and barrier phases follow the CTA's running KV-tile count jg0 + j
  auto process = [&](const HalfRaw<F, D>& r, int j, int h) -> bool {
    const int jg = jg0 + j;
    if (is_k) {
      if (h == 0 && jg > 1) ok = mbar_wait(&free_bars[jg & 1], (uint32_t)(((jg - 2) >> 1) & 1), err) && ok;
    } else {
      if (jg > 0) ok = mbar_wait(&free_bars[h], (uint32_t)((jg - 1) & 1), err) && ok;
    }
    tc_fence_after();
    const bool b1 = is_k && (jg & 1);
    convert_half<F, D, LO>(r, b1 ? dst_hi1 : dst_hi0, b1 ? dst_lo1 : dst_lo0, h, t0);
    fence_proxy_async_smem();
    if (bar_any(bar_id, 128, !ok || *abort_flag)) {  // one decision for the group
      *abort_flag = 1;
      return false;
    }
    if (t0 == 0) {
      if (!is_k) mbar_arrive(&ready[h]);
      else if (h == 1) mbar_arrive(&ready[jg & 1]);
    }
    return true;
  };
  HalfRaw<F, D> ra, rb;
  int pa = pid_of(0), pb = pid_of(1);
  load_half<F, D>(ra, q_plane, s_plane, pa, pb, num_pages, hkv, g, valid_of(0, 0), t0, err);
  pa = pid_of(2);
  pb = pid_of(3);
  for (int j = 0; j < n_kv; ++j) {
    // half 0 of tile j is in ra; fetch half 1 into rb meanwhile
    load_half<F, D>(rb, q_plane, s_plane, pa, pb, num_pages, hkv, g, valid_of(j, 1), t0, err);
    pa = pid_of(4 * (j + 1));
    pb = pid_of(4 * (j + 1) + 1);
    if (!process(ra, j, 0)) return false;
    // half 1 is in rb; fetch half 0 of tile j+1 into ra meanwhile
    if (j + 1 < n_kv) load_half<F, D>(ra, q_plane, s_plane, pa, pb, num_pages, hkv, g, valid_of(j + 1, 0), t0, err);
    pa = pid_of(4 * (j + 1) + 2);
    pb = pid_of(4 * (j + 1) + 3);
    if (!process(rb, j, 1)) return false;
  }
  return ok;
}

// Tile k of chunk CTA c among C chunk CTAs: a snake over the heaviest-first
// tile list (c, 2C-1-c, 2C+c, ...), so every CTA gets a similar share of work;
// -1 where the snake runs past the last tile.
__device__ __forceinline__ int chunk_tile_of(int c, int k, int C, int n) {
  const int idx = (k & 1) ? (k + 1) * C - 1 - c : k * C + c;
  return idx < n ? idx : -1;
}

// Chunk CTA c of C: walks its chunk tiles (chunk_tile_of) one after the other.
// A tile is 128 rows (128/G query tokens x G heads of kv head `t.kvh`) against
// the keys they can see, in 128-key KV tiles.  Roles:
//   K group (warps 4-7): loads the raw K bytes of each KV tile straight from the
//     cache planes (one 64-key half ahead of their use) and dequantises them
//     into operand buffer jg%2 once QK(jg-2) has released it;
//   V group (warps 8-11): the same for V, into a single buffer, key half h once
//     the PV MMAs of the previous KV tile that read that half are done;
//   softmax group (warps 0-3, thread i = TMEM lane i = query row i): reads
//     S[jg%2] twice (row max, then P = 2^(s - m) as fp16 into the P columns,
//     each key half once the previous PV MMAs reading that half are done),
//     rescales O when the row max moved; after a tile's last scores it writes
//     the next tile's Q, then stores this tile's O;
//   MMA warp (warp 12, one thread): issues QK(jg) into S[jg%2] once K(jg) is
//     written (and, on a tile's first KV tile, its Q), then PV(jg-1), each key
//     half as soon as its V half is written.
// jg counts the KV tiles the CTA has walked, across its tiles: buffers and
// barrier phases follow it, so the next tile's loads, dequantisation and first
// QK overlap this tile's last softmax and its epilogue.  The MMA issue blocks
// its thread for about the MMA's duration, which is why one warp does nothing
// else.  TMEM: Q | P (A operands, fp16) | S0 | S1 | O (fp32).  Every wait is
// bounded; a timeout in any role makes all of them leave their loops.
template <int FK, int FV, int D>
__device__ __forceinline__ void chunk_cta(const AttnParams& p, int cta, int n_ctas, uint8_t* smem_raw,
                                          unsigned int* err) {
  using L = ChunkSmem<FK, FV, D>;
  constexpr uint32_t kTmemCols = 512;
  constexpr uint32_t kQCol = 0, kPCol = 64, kSCol0 = 128, kSCol1 = 256, kOCol = 384;
  constexpr int kGroup = 128;          // threads per warp group
  constexpr int kBarSoftmax = 1, kBarK = 2, kBarV = 3;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* kdeq = bars;                   // [2] K(jg) written to buffer jg%2
  uint64_t* vdeq = kdeq + 2;               // [2] V half h of the current KV tile written
  uint64_t* pvh_done = vdeq + 2;           // [2] the PV MMAs reading V half h are done
  uint64_t* qk_done = pvh_done + 2;        // [2] S[st] holds the scores of the KV tile
  uint64_t* pv_done = qk_done + 2;         // [2] PV of the KV tile done
  uint64_t* sm_done = pv_done + 2;         // [2] P of the KV tile written, O rescaled
  uint64_t* q_ready = sm_done + 2;         // [1] Q of the CTA's next tile is in TMEM
  uint64_t* mma_fin = q_ready + 1;         // [1] every MMA of the CTA done
  constexpr int kNumBars = 14;
  static_assert(kNumBars * 8 + 8 <= L::kBarBytes, "barrier area too small");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + kNumBars) + 1;

  const int tid = threadIdx.x, warp = tid >> 5;
  const int G = p.group, lg = p.log2_group;
  const int n_rounds = (p.n_chunk_tiles + n_ctas - 1) / n_ctas;

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) mbar_init(bars + i, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int row = tid & 127;  // softmax group: TMEM lane = query row
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;

  constexpr uint32_t kIdescQK = idesc_f16_f32(128, kChunkN, false, false);
  constexpr uint32_t kIdescPV = idesc_f16_f32(128, D, false, true);
  // operand descriptors, split into words: K tiles K-major (SBO 1024 B between
  // 8-key groups), V tiles MN-major (LBO = one 64-column slab, 128 keys x 128 B)
  const uint32_t dK0 = (uint32_t)sw128_desc(smem_u32(smem + L::kK0), 16, 1024);
  const uint32_t dK1 = (uint32_t)sw128_desc(smem_u32(smem + L::kK1), 16, 1024);
  const uint32_t dHiK = (uint32_t)(sw128_desc(0, 16, 1024) >> 32);
  const uint32_t dV = (uint32_t)sw128_desc(smem_u32(smem + L::kVh), kChunkN * 128, 1024);
  const uint32_t dHiV = (uint32_t)(sw128_desc(0, kChunkN * 128, 1024) >> 32);
  bool ok = true;

  if (tid >= kGroup && tid < 3 * kGroup) {
    // =========== K group (warps 4-7) and V group (warps 8-11): dequantisation ===========
    const bool is_k = tid < 2 * kGroup;
    int jg0 = 0;
    bool alive = true;
    for (int k = 0; alive && k < n_rounds; ++k) {
      const int idx = chunk_tile_of(cta, k, n_ctas, p.n_chunk_tiles);
      if (idx < 0) continue;
      const TileDesc t = p.tiles[idx];
      const RowInfo ri = p.rows[t.row];
      const int n_pages_row = (ri.seq_len + kPage - 1) / kPage;
      const int key_end = min(ri.seq_len, ri.q_offset + t.begin + t.count);
      const int kv0 = t.kv0, n_kv = t.kv1 - t.kv0;
      const int32_t* pt_row = p.page_table + (int64_t)t.row * p.max_pages + kv0 * kPagesPerKvTile;
      alive = is_k ? dequant_loop<FK, D, L::kKLo>(p.k_quant, p.k_scale, pt_row, n_pages_row - kv0 * kPagesPerKvTile,
                                                  p.num_pages, p.hkv, t.kvh, key_end - kv0 * kChunkN, n_kv, jg0,
                                                  tid - kGroup, true, smem + L::kK0, smem + L::kK0 + L::kTile,
                                                  smem + L::kK1, smem + L::kK1 + L::kTile, qk_done, kdeq, kBarK,
                                                  abort_flag, err)
                   : dequant_loop<FV, D, L::kVLo>(p.v_quant, p.v_scale, pt_row, n_pages_row - kv0 * kPagesPerKvTile,
                                                  p.num_pages, p.hkv, t.kvh, key_end - kv0 * kChunkN, n_kv, jg0,
                                                  tid - 2 * kGroup, false, smem + L::kVh, smem + L::kVl,
                                                  smem + L::kVh, smem + L::kVl, pvh_done, vdeq, kBarV, abort_flag,
                                                  err);
      jg0 += n_kv;
    }
    if (!alive) *abort_flag = 1;
  } else if (tid < kGroup) {
    // ======================= softmax group =======================
    const float sl2 = p.scale_log2;
    const uint32_t ninf = __float_as_uint(-CUDART_INF_F);
    const int tok = row >> lg;
    // Q rows of chunk tile idx -> TMEM (the A operand of QK), two fp16 per
    // column; then the MMA warp may issue the tile's QK
    auto write_q = [&](int idx) {
      const TileDesc t = p.tiles[idx];
      const RowInfo ri = p.rows[t.row];
      const uint16_t* src = static_cast<const uint16_t*>(p.q) +
                            ((int64_t)(ri.q_start + t.begin + min(tok, t.count - 1)) * p.hq + (int64_t)t.kvh * G +
                             (row & (G - 1))) * D;
#pragma unroll
      for (int ch = 0; ch < D / 64; ++ch) {
        uint32_t v[32];
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const uint4 w = tok < t.count ? ldg_u128(src + 64 * ch + 8 * q4) : make_uint4(0u, 0u, 0u, 0u);
          v[4 * q4] = w.x;
          v[4 * q4 + 1] = w.y;
          v[4 * q4 + 2] = w.z;
          v[4 * q4 + 3] = w.w;
        }
        tmem_st32(tmem + lane_base + kQCol + 32 * ch, v);
      }
      tmem_wait_st();
      tc_fence_before();
      bar_any(kBarSoftmax, kGroup, false);
      if (tid == 0) mbar_arrive(q_ready);
    };
    auto next_round = [&](int k) {  // the first round >= k that holds a tile of this CTA
      while (k < n_rounds && chunk_tile_of(cta, k, n_ctas, p.n_chunk_tiles) < 0) ++k;
      return k;
    };
    int k = next_round(0);
    if (k < n_rounds) write_q(chunk_tile_of(cta, k, n_ctas, p.n_chunk_tiles));
    int jg0 = 0;
    for (; k < n_rounds && !*abort_flag; k = next_round(k + 1)) {
      const int idx = chunk_tile_of(cta, k, n_ctas, p.n_chunk_tiles);
      const TileDesc t = p.tiles[idx];
      const RowInfo ri = p.rows[t.row];
      const int g = t.kvh;
      const bool row_valid = tok < t.count;
      const int pos = ri.q_offset + t.begin + min(tok, t.count - 1);
      const int kv0 = t.kv0, n_kv = t.kv1 - t.kv0;
      float m_run = -CUDART_INF_F, l_run = 0.f;
      for (int j = 0; j < n_kv; ++j) {
        const int jg = jg0 + j;
        const int st = jg & 1;
        const uint32_t ph = (uint32_t)((jg >> 1) & 1);
        const uint32_t s_base = st ? kSCol1 : kSCol0;
        const uint32_t s_col = tmem + lane_base + s_base;
        ok = mbar_wait(&qk_done[st], ph, err) && ok;
        tc_fence_after();
        const int kbase = (kv0 + j) * kChunkN;
        // causal mask: only a warp whose tile crosses the diagonal pays for it
        const bool diag = __any_sync(0xFFFFFFFFu, kbase + kChunkN - 1 > pos);
        uint32_t a[32];
        // pass 1: the row max of the tile's 128 scores, 32 at a time
        float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          tmem_ld32(s_col + 32 * c, a);
          tmem_wait_ld();
          if (diag) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (kbase + 32 * c + e > pos) a[e] = ninf;
          }
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            mx0 = fmax3(mx0, __uint_as_float(a[e]), __uint_as_float(a[e + 1]));
            mx1 = fmax3(mx1, __uint_as_float(a[e + 2]), __uint_as_float(a[e + 3]));
          }
        }
        // running max in log2 units (the score scale is positive, so it commutes with max)
        const float m_new = fmaxf(m_run, fmaxf(mx0, mx1) * sl2);
        // a row can see none of a piece's first keys (a later piece of a cut tile):
        // everything stays zero until its first visible key
        const bool none = m_new == -CUDART_INF_F;
        const float alpha = none ? 1.f : ex2(m_run - m_new);
        const float neg_m = none ? 0.f : -m_new;
        // pass 2: P = 2^(s*scale - m) as fp16 into the P columns (keys 32c.. of
        // chunk c), each key half once the PV(j-1) MMAs reading that half of
        // P(j-1) are done; row sums in fp32.  The scale-and-shift and the sums run
        // on fp32 pairs.
        const uint64_t sl2x2 = f2_pack(sl2, sl2), negm2 = f2_pack(neg_m, neg_m);
        uint64_t sum_a = f2_pack(0.f, 0.f), sum_b = sum_a;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          tmem_ld32(s_col + 32 * c, a);
          tmem_wait_ld();
          if (diag) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (kbase + 32 * c + e > pos) a[e] = ninf;
          }
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            float x0, x1, x2, x3;
            f2_unpack(ffma2(f2_pack(__uint_as_float(a[e]), __uint_as_float(a[e + 1])), sl2x2, negm2), x0, x1);
            f2_unpack(ffma2(f2_pack(__uint_as_float(a[e + 2]), __uint_as_float(a[e + 3])), sl2x2, negm2), x2, x3);
            const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
            sum_a = fadd2(sum_a, f2_pack(p0, p1));
            sum_b = fadd2(sum_b, f2_pack(p2, p3));
            pk[e >> 1] = pack_f16x2(p0, p1);
            pk[(e >> 1) + 1] = pack_f16x2(p2, p3);
          }
          if (jg > 0 && (c & 1) == 0) {
            ok = mbar_wait(&pvh_done[c >> 1], (uint32_t)((jg - 1) & 1), err) && ok;
            tc_fence_after();
          }
          tmem_st16(tmem + lane_base + kPCol + 16 * c, pk);
        }
        float sum0, sum1, sum2, sum3;
        f2_unpack(sum_a, sum0, sum1);
        f2_unpack(sum_b, sum2, sum3);
        sum0 += sum2;
        sum1 += sum3;
        l_run = l_run * alpha + (sum0 + sum1);
        m_run = m_new;
        // the running O: PV(j-1) has finished with it (its last half was waited above)
        if (j > 0) {
          if (__any_sync(0xFFFFFFFFu, alpha != 1.0f)) {
#pragma unroll 1
            for (int ch = 0; ch < D / 32; ++ch) {
              tmem_ld32(tmem + lane_base + kOCol + 32 * ch, a);
              tmem_wait_ld();
              const uint64_t al2 = f2_pack(alpha, alpha);
#pragma unroll
              for (int e = 0; e < 32; e += 2) {
                float y0, y1;
                f2_unpack(fmul2(f2_pack(__uint_as_float(a[e]), __uint_as_float(a[e + 1])), al2), y0, y1);
                a[e] = __float_as_uint(y0);
                a[e + 1] = __float_as_uint(y1);
              }
              tmem_st32(tmem + lane_base + kOCol + 32 * ch, a);
            }
          }
        }
        tmem_wait_st();
        tc_fence_before();
        if (bar_any(kBarSoftmax, kGroup, !ok || *abort_flag)) {  // one decision for the group
          *abort_flag = 1;
          break;
        }
        if (tid == 0) mbar_arrive(&sm_done[st]);  // P(jg) written, O rescaled
      }
      // the next tile's Q: this tile's last QK is done (its scores were read above)
      const int kn = next_round(k + 1);
      if (kn < n_rounds && !*abort_flag) write_q(chunk_tile_of(cta, kn, n_ctas, p.n_chunk_tiles));
      // ---- epilogue of this tile, while the MMA warp starts the next ----
      const bool done = !*abort_flag;
      const int jl = jg0 + n_kv - 1;  // the tile's last KV tile
      if (done && n_kv > 0) ok = mbar_wait(&pv_done[jl & 1], (uint32_t)((jl >> 1) & 1), err) && ok;
      tc_fence_after();
      uint16_t* dst = static_cast<uint16_t*>(p.o) +
                      ((int64_t)(ri.q_start + t.begin + tok) * p.hq + (int64_t)g * G + (row & (G - 1))) * D;
      if (t.nsplit == 1) {
        const float inv_l = (l_run > 0.f) ? 1.f / l_run : 0.f;
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + kOCol + 32 * ch, v);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            pk[e >> 1] = pack_f16x2(__uint_as_float(v[e]) * inv_l, __uint_as_float(v[e + 1]) * inv_l);
          if (row_valid && ok && done) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              *reinterpret_cast<uint4*>(dst + 32 * ch + 8 * q4) =
                  make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
          }
        }
      } else {
        // a piece of a cut tile: leave (m, l, unnormalised O) of its rows; the last
        // piece to finish merges them (log-sum-exp) and writes O
        const int64_t n_o = (int64_t)p.n_chunk_tiles * kChunkM * D;  // the O partials come first
        float* o_part = p.chunk_partials + ((int64_t)idx * kChunkM + row) * D;
        float* ml_part = p.chunk_partials + n_o + ((int64_t)idx * kChunkM + row) * 2;
        ml_part[0] = m_run;
        ml_part[1] = l_run;
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + kOCol + 32 * ch, v);
          tmem_wait_ld();
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4)
            *reinterpret_cast<uint4*>(o_part + 32 * ch + 4 * q4) =
                make_uint4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
        }
        __threadfence();
        __shared__ int s_last_piece;
        bar_any(kBarSoftmax, kGroup, false);
        const int first = idx - t.part;  // the tile's pieces are consecutive
        if (tid == 0) s_last_piece = atomicAdd(&p.chunk_counters[first], 1u) == (unsigned)(t.nsplit - 1);
        bar_any(kBarSoftmax, kGroup, false);
        if (s_last_piece) {
          __threadfence();
          float m_all = -CUDART_INF_F;
          for (int q = 0; q < t.nsplit; ++q)
            m_all = fmaxf(m_all, __ldcg(p.chunk_partials + n_o + ((int64_t)(first + q) * kChunkM + row) * 2));
          float l_all = 0.f;
          for (int q = 0; q < t.nsplit; ++q) {
            const float* ml = p.chunk_partials + n_o + ((int64_t)(first + q) * kChunkM + row) * 2;
            const float mq = __ldcg(ml);
            l_all += mq == -CUDART_INF_F ? 0.f : __ldcg(ml + 1) * ex2(mq - m_all);
          }
          const float inv_l = (l_all > 0.f) ? 1.f / l_all : 0.f;
#pragma unroll 1
          for (int d0 = 0; d0 < D; d0 += 8) {
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int q = 0; q < t.nsplit; ++q) {
              const float mq = __ldcg(p.chunk_partials + n_o + ((int64_t)(first + q) * kChunkM + row) * 2);
              if (mq == -CUDART_INF_F) continue;
              const float w = ex2(mq - m_all);
              const float* op = p.chunk_partials + ((int64_t)(first + q) * kChunkM + row) * D + d0;
              const float4 x0 = __ldcg(reinterpret_cast<const float4*>(op));
              const float4 x1 = __ldcg(reinterpret_cast<const float4*>(op + 4));
              acc[0] += w * x0.x; acc[1] += w * x0.y; acc[2] += w * x0.z; acc[3] += w * x0.w;
              acc[4] += w * x1.x; acc[5] += w * x1.y; acc[6] += w * x1.z; acc[7] += w * x1.w;
            }
            if (row_valid && ok && done)
              *reinterpret_cast<uint4*>(dst + d0) =
                  make_uint4(pack_f16x2(acc[0] * inv_l, acc[1] * inv_l), pack_f16x2(acc[2] * inv_l, acc[3] * inv_l),
                             pack_f16x2(acc[4] * inv_l, acc[5] * inv_l), pack_f16x2(acc[6] * inv_l, acc[7] * inv_l));
          }
        }
      }
      jg0 += n_kv;
    }
  } else if (tid == 3 * kGroup) {
    // ============ MMA warp (warp 12, one thread): issues every tcgen05.mma ============
    // Order on the tensor pipe: QK(0), QK(1), PV(0), QK(2), PV(1), ... over the
    // CTA's KV tiles, the first QK of a tile once its Q is in TMEM.
    int jg0 = 0, nt = 0;
    for (int k = 0; k < n_rounds && ok; ++k) {
      const int idx = chunk_tile_of(cta, k, n_ctas, p.n_chunk_tiles);
      if (idx < 0) continue;
      const TileDesc t = p.tiles[idx];
      const int n_kv = t.kv1 - t.kv0;
      ok = mbar_wait(q_ready, (uint32_t)(nt & 1), err) && ok;  // this tile's Q written
      ++nt;
      if (!ok) break;
      tc_fence_after();
      for (int j = 0; j <= n_kv; ++j) {
        if (j < n_kv) {
          const int jg = jg0 + j, st = jg & 1;
          const uint32_t s_col = tmem + (st ? kSCol1 : kSCol0);
          ok = mbar_wait(&kdeq[st], (uint32_t)((jg >> 1) & 1), err) && ok;  // K(jg) written to buffer st
          // S[st] is free: the softmax of KV tile jg-2 read it before PV(jg-2) was issued
          if (!ok) break;
          tc_fence_after();
          const uint32_t kd = st ? dK1 : dK0;  // low descriptor word of K buffer st
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = (uint32_t)((ks >> 2) * (kChunkN * 128) + (ks & 3) * 32) >> 4;
            if (ks == 0) tc_mma_ts_w<0>(s_col, tmem + kQCol, kd + off, dHiK, kIdescQK);
            else tc_mma_ts_w<1>(s_col, tmem + kQCol + 8 * ks, kd + off, dHiK, kIdescQK);
            if (L::kKLo) tc_mma_ts_w<1>(s_col, tmem + kQCol + 8 * ks, kd + (L::kTile >> 4) + off, dHiK, kIdescQK);
          }
          tc_commit(&qk_done[st]);
        }
        if (j > 0) {
          const int jp = jg0 + j - 1, sp = jp & 1;
          ok = mbar_wait(&sm_done[sp], (uint32_t)((jp >> 1) & 1), err) && ok;  // P(jp) written, O rescaled
          const uint32_t p_col = tmem + kPCol;
#pragma unroll
          for (int hv = 0; hv < 2; ++hv) {
            ok = mbar_wait(&vdeq[hv], (uint32_t)(jp & 1), err) && ok;  // V half hv of KV tile jp written
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 4 * hv; kk < 4 * hv + 4; ++kk) {
              const uint32_t pa = p_col + 8 * kk;  // P columns of keys 16kk..16kk+15
              const uint32_t boff = (uint32_t)(kk * 16 * 128) >> 4;
              // the tile's first PV overwrites O (the softmax group has stored the last tile's)
              if (kk == 0) tc_mma_ts_w(tmem + kOCol, pa, dV + boff, dHiV, kIdescPV, j > 1 ? 1u : 0u);
              else tc_mma_ts_w<1>(tmem + kOCol, pa, dV + boff, dHiV, kIdescPV);
              if (L::kVLo) tc_mma_ts_w<1>(tmem + kOCol, pa, dV + (L::kTile >> 4) + boff, dHiV, kIdescPV);
            }
            tc_commit(&pvh_done[hv]);
          }
          if (!ok) break;
          tc_commit(&pv_done[sp]);
        }
        if (*abort_flag) {
          ok = false;
          break;
        }
      }
      jg0 += n_kv;
    }
    if (!ok) *abort_flag = 1;
    // nothing this thread started may still run when TMEM is released
    tc_commit(mma_fin);
    mbar_wait(mma_fin, 0u, err);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Stages of a decode warp's ring inside the fused launch (which sizes its shared
// memory for the chunk role).
template <int FK, int FV, int D>
struct FusedSmem {
  using DS = DecodeSmem<FK, FV, D>;
  // two decode tiles per CTA (one per half of its warps) where two rings of two
  // stages fit, else one
  static constexpr bool kTwoDecode = 2 * DS::total(2) <= 227 * 1024;
  static constexpr int kDecodePerCta = kTwoDecode ? 2 : 1;
  static constexpr int kDecNeed = kDecodePerCta * DS::total(2);
  static constexpr int kNeed = ChunkSmem<FK, FV, D>::kTotal > kDecNeed ? ChunkSmem<FK, FV, D>::kTotal : kDecNeed;
  static constexpr int kBytes = (kNeed + 255) / 256 * 256;
  static constexpr int kHalfBytes = kBytes / kDecodePerCta;  // one decode tile's share (a multiple of 128)
  static constexpr int kDecodeStages = DS::stages_for(kHalfBytes - 16);
  static_assert(DS::total(kDecodeStages) <= kHalfBytes, "decode tile does not fit");
};

template <int FK, int FV, int D>
__global__ void __launch_bounds__(kFusedThreads, 1) mixed_attention_kernel(AttnParams p, unsigned int* err) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tile = blockIdx.x;
  if (tile < p.n_chunk_ctas) {
    chunk_cta<FK, FV, D>(p, tile, p.n_chunk_ctas, smem, err);
  } else {
    // two decode tiles per CTA where they fit, one on each half of its warps and
    // shared memory; else one on the first half
    using FS = FusedSmem<FK, FV, D>;
    const int half = threadIdx.x >= kThreads ? 1 : 0;
    if (half && !FS::kTwoDecode) return;
    const int d = FS::kDecodePerCta * (tile - p.n_chunk_ctas) + half;
    if (d >= p.n_decode_tiles) return;
    decode_tile<FK, FV, D, FS::kDecodeStages>(p, p.tiles[p.n_chunk_tiles + d], d, smem + half * FS::kHalfBytes, err,
                                              half);
  }
}

template <int FK, int FV, int D, int MINB, int NS>
__global__ void __launch_bounds__(kThreads, MINB) decode_attention_kernel(AttnParams p, unsigned int* err) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tile = blockIdx.x + p.n_chunk_tiles;
  decode_tile<FK, FV, D, NS>(p, p.tiles[tile], blockIdx.x, smem, err, 0);
}

// Chunk tiles whose mean KV-tile count is below this are walked by persistent
// CTAs.
constexpr int kPersistMaxKvTiles = 64;

// SMs of the current device, read once per device (a very large count when it
// cannot be read: then every chunk tile gets its own CTA).
inline int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1 << 30;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1 << 30;
    cached[dev] = n;
  }
  return cached[dev];
}

template <int FK, int FV, int D>
cudaError_t launch_attention_t(const AttnParams& p, unsigned int* err, cudaStream_t s) {
  using DS = DecodeSmem<FK, FV, D>;
  const int n_tiles = p.n_chunk_tiles + p.n_decode_tiles;
  if (n_tiles == 0) return cudaSuccess;
  constexpr int kPer = FusedSmem<FK, FV, D>::kDecodePerCta;  // decode tiles per fused CTA
  // short chunk tiles run on at most one CTA per SM, each walking several (the
  // next tile's loads and first MMAs then overlap this tile's last softmax and
  // its epilogue, ~15k cycles a tile); long ones, where that overlap is worth
  // little, one per CTA
  AttnParams q = p;
  const bool persist = p.n_chunk_tiles > 0 && p.chunk_kv_tiles < kPersistMaxKvTiles * p.n_chunk_tiles;
  q.n_chunk_ctas = persist ? std::min(p.n_chunk_tiles, sm_count()) : p.n_chunk_tiles;
  const int n_fused_ctas = q.n_chunk_ctas + (p.n_decode_tiles + kPer - 1) / kPer;
  constexpr int kDec = DS::kTotal;
  constexpr int kFused = FusedSmem<FK, FV, D>::kBytes;
  auto* dec_kernel = decode_attention_kernel<FK, FV, D, DS::kSoloMinBlocks, DS::kSoloStages>;
  static bool configured = false;  // the attribute is per function, once per process
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(dec_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDec);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(mixed_attention_kernel<FK, FV, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kFused);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  if (p.n_chunk_tiles == 0) {
    dec_kernel<<<p.n_decode_tiles, kThreads, kDec, s>>>(p, err);
  } else {
    mixed_attention_kernel<FK, FV, D><<<n_fused_ctas, kFusedThreads, kFused, s>>>(q, err);
  }
  return cudaGetLastError();
}

}  // namespace mixattn
