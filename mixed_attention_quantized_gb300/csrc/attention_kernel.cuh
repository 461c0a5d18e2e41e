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
// range of one (row, kv head); each warp streams its pages with 16-byte-class
// vector loads straight into registers and runs QK^T and PV on mma.sync
// m16n8k16 with the G query heads in the N=8 dimension.  Quantised codes are
// turned into exact fp16 integers by a byte permute (no rounding); the Q8_0 /
// Q4_0 scales are applied in fp32: per key and 32-d block on the scores, and
// folded into P per key and block on the values.  Warp partials are merged in
// shared memory, split partials by the last CTA of the (row, kv head) to
// finish (atomic ticket, no spin).
//
// Chunk tiles (tensor-bound): a CTA owns 128 rows = 128/G query tokens x G
// heads of one kv head.  K/V pages arrive raw through 1-D bulk copies (TMA
// engine) into a stage whose refill overlaps the math of the previous tile.
// They are dequantised into 128-byte-swizzled fp16 tiles -- an exact hi/lo
// pair for quantised formats, since d*q needs up to 18 significant bits --
// and S = Q K^T and O += P V run on tcgen05.mma (one MMA per half) with the
// accumulators in TMEM.  The softmax threads own one TMEM lane (one query row)
// each and write P as fp16 back into TMEM, where the PV MMA reads it.
#pragma once

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
  static constexpr int kNb = D / kBlock;
  static constexpr int kKqPage = kPage * (FK == MIXATTN_KV_F16 ? 2 * D : (FK == MIXATTN_KV_Q8_0 ? D : D / 2));
  static constexpr int kKsPage = FK == MIXATTN_KV_F16 ? 0 : kPage * kNb * 2;
  static constexpr int kVqPage = kPage * (FV == MIXATTN_KV_F16 ? 2 * D : (FV == MIXATTN_KV_Q8_0 ? D : D / 2));
  static constexpr int kVsPage = FV == MIXATTN_KV_F16 ? 0 : kPage * kNb * 2;
  static constexpr int kPagesPerTile = kChunkN / kPage;  // 4
  // quantised formats carry an exact low half: d*q = hi + lo, both fp16
  static constexpr bool kKLo = FK != MIXATTN_KV_F16;
  static constexpr bool kVLo = FV != MIXATTN_KV_F16;
  // raw stage: [Kq x4][Ks x4][Vq x4][Vs x4]
  static constexpr int kRawKq = 0;
  static constexpr int kRawKs = kRawKq + kPagesPerTile * kKqPage;
  static constexpr int kRawVq = kRawKs + kPagesPerTile * kKsPage;
  static constexpr int kRawVs = kRawVq + kPagesPerTile * kVqPage;
  static constexpr int kRawBytes = (kRawVs + kPagesPerTile * kVsPage + 1023) / 1024 * 1024;
  static constexpr int kTile = kChunkN * D * 2;             // one fp16 operand tile
  static constexpr int kQ = 0;                              // [D/64][128 rows][128 B]
  static constexpr int kKh = kQ + kChunkM * D * 2;          // [D/64][128 keys][128 B]
  static constexpr int kKl = kKh + kTile;
  static constexpr int kVh = kKl + (kKLo ? kTile : 0);
  static constexpr int kVl = kVh + kTile;
  static constexpr int kRaw = kVl + (kVLo ? kTile : 0);
  static constexpr int kBar = kRaw + kRawBytes;
  static constexpr int kTotal = kBar + 64 + 1024;           // + slack for 1024-B alignment
  static_assert(kTotal <= 227 * 1024, "chunk tile does not fit in shared memory");
};

// Merge scratch of a decode tile: per warp m[8], l[8], O[8][D].
template <int D>
struct DecodeSmem {
  static constexpr int kPerWarp = 16 + kMaxGroup * D;
  static constexpr int kTotal = kWarps * kPerWarp * 4 + 16;
};

// ===========================================================================
// Decode tiles
// ===========================================================================

// Byte offset of token `key` (0..31) of a page-plane row, for K/V row bytes.
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

template <int FK, int FV, int D>
__device__ __forceinline__ void decode_tile(const AttnParams& p, const TileDesc& t, int dec_idx, uint8_t* smem,
                                            unsigned int* err) {
  constexpr int NB = D / kBlock;   // scale blocks per row
  constexpr int KS = D / 16;       // k-steps of QK / M-tiles of PV
  constexpr int RBK = row_bytes<FK, D>();
  constexpr int RBV = row_bytes<FV, D>();

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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

  // ---- Q as the B operand of S^T = K Q^T (heads in N) ----------------------
  uint32_t qf[KS][2];
  {
    const bool real = r < G;
    const uint16_t* qrow =
        static_cast<const uint16_t*>(p.q) + ((int64_t)ri.q_start * p.hq + (int64_t)g * G + (real ? r : 0)) * D;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      if (FK == MIXATTN_KV_Q4_0) {
        uint2 lo = real ? ldg_u64(qrow + 32 * b + 4 * c) : make_uint2(0u, 0u);
        uint2 hi = real ? ldg_u64(qrow + 32 * b + 16 + 4 * c) : make_uint2(0u, 0u);
        qf[2 * b][0] = lo.x;
        qf[2 * b][1] = lo.y;
        qf[2 * b + 1][0] = hi.x;
        qf[2 * b + 1][1] = hi.y;
      } else {
        uint4 v = real ? ldg_u128(qrow + 32 * b + 8 * c) : make_uint4(0u, 0u, 0u, 0u);
        qf[2 * b][0] = v.x;
        qf[2 * b][1] = v.y;
        qf[2 * b + 1][0] = v.z;
        qf[2 * b + 1][1] = v.w;
      }
    }
  }

  float o_acc[KS][4];
#pragma unroll
  for (int i = 0; i < KS; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
  float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F};
  float l_run[2] = {0.f, 0.f};
  const float sl2 = p.scale_log2;

  const uint8_t* kq_base = p.k_quant + (int64_t)g * kPage * RBK;
  const uint8_t* vq_base = p.v_quant + (int64_t)g * kPage * RBV;
  const uint16_t* ks_base = p.k_scale + (int64_t)g * kPage * NB;
  const uint16_t* vs_base = p.v_scale + (int64_t)g * kPage * NB;
  const int64_t kq_page_stride = (int64_t)p.hkv * kPage * RBK;
  const int64_t vq_page_stride = (int64_t)p.hkv * kPage * RBV;
  const int64_t sc_page_stride = (int64_t)p.hkv * kPage * NB;
  const int32_t* pt_row = p.page_table + (int64_t)t.row * p.max_pages;

  for (int pg = wp0; pg < wp1; ++pg) {
    const int pid = pt_row[pg];
    if (pid < 0 || pid >= p.num_pages) {
      if (lane == 0) set_device_error(err, MIXATTN_DEVERR_PAGE_ID);
      continue;
    }
    const uint8_t* kq = kq_base + (int64_t)pid * kq_page_stride;
    const uint8_t* vq = vq_base + (int64_t)pid * vq_page_stride;
    const uint16_t* ksc = ks_base + (int64_t)pid * sc_page_stride;
    const uint16_t* vsc = vs_base + (int64_t)pid * sc_page_stride;
    const int key0 = pg * kPage;

    // ---------------- S^T = K Q^T for the page's 32 keys ----------------
    float s[2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const int k_lo = 16 * mt + r, k_hi = k_lo + 8;  // the lane's two key rows
      s[mt][0] = s[mt][1] = s[mt][2] = s[mt][3] = 0.f;
      float dk_lo[NB], dk_hi[NB];
      if (FK != MIXATTN_KV_F16) {
        if (NB == 4) {
          uint2 a = ldg_u64(ksc + k_lo * NB), b2 = ldg_u64(ksc + k_hi * NB);
          dk_lo[0] = __half2float(__ushort_as_half(a.x & 0xFFFF));
          dk_lo[1] = __half2float(__ushort_as_half(a.x >> 16));
          dk_lo[2 % NB] = __half2float(__ushort_as_half(a.y & 0xFFFF));
          dk_lo[3 % NB] = __half2float(__ushort_as_half(a.y >> 16));
          dk_hi[0] = __half2float(__ushort_as_half(b2.x & 0xFFFF));
          dk_hi[1] = __half2float(__ushort_as_half(b2.x >> 16));
          dk_hi[2 % NB] = __half2float(__ushort_as_half(b2.y & 0xFFFF));
          dk_hi[3 % NB] = __half2float(__ushort_as_half(b2.y >> 16));
        } else {
          uint32_t a = ldg_u32(ksc + k_lo * NB), b2 = ldg_u32(ksc + k_hi * NB);
          dk_lo[0] = __half2float(__ushort_as_half(a & 0xFFFF));
          dk_lo[1 % NB] = __half2float(__ushort_as_half(a >> 16));
          dk_hi[0] = __half2float(__ushort_as_half(b2 & 0xFFFF));
          dk_hi[1 % NB] = __half2float(__ushort_as_half(b2 >> 16));
        }
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        uint32_t a0[4], a1[4];  // A fragments of k-steps 2b and 2b+1
        if (FK == MIXATTN_KV_Q8_0) {
          const uint2 wl = ldg_u64(kq + k_lo * RBK + 32 * b + 8 * c);
          const uint2 wh = ldg_u64(kq + k_hi * RBK + 32 * b + 8 * c);
          s8x4_to_f16x2x2(wl.x, a0[0], a0[2]);
          s8x4_to_f16x2x2(wh.x, a0[1], a0[3]);
          s8x4_to_f16x2x2(wl.y, a1[0], a1[2]);
          s8x4_to_f16x2x2(wh.y, a1[1], a1[3]);
        } else if (FK == MIXATTN_KV_Q4_0) {
          const uint32_t yl = ldg_u32(kq + k_lo * RBK + 16 * b + 4 * c);
          const uint32_t yh = ldg_u32(kq + k_hi * RBK + 16 * b + 4 * c);
          u4x4_to_f16x2x2(yl & 0x0F0F0F0Fu, a0[0], a0[2]);
          u4x4_to_f16x2x2(yh & 0x0F0F0F0Fu, a0[1], a0[3]);
          u4x4_to_f16x2x2((yl >> 4) & 0x0F0F0F0Fu, a1[0], a1[2]);
          u4x4_to_f16x2x2((yh >> 4) & 0x0F0F0F0Fu, a1[1], a1[3]);
        } else {
          const uint4 wl = ldg_u128(kq + k_lo * RBK + 2 * (32 * b + 8 * c));
          const uint4 wh = ldg_u128(kq + k_hi * RBK + 2 * (32 * b + 8 * c));
          a0[0] = wl.x; a0[1] = wh.x; a0[2] = wl.y; a0[3] = wh.y;
          a1[0] = wl.z; a1[1] = wh.z; a1[2] = wl.w; a1[3] = wh.w;
        }
        if (FK == MIXATTN_KV_F16) {
          mma_16816(s[mt], a0, qf[2 * b]);
          mma_16816(s[mt], a1, qf[2 * b + 1]);
        } else {
          float tmp[4] = {0.f, 0.f, 0.f, 0.f};
          mma_16816(tmp, a0, qf[2 * b]);
          mma_16816(tmp, a1, qf[2 * b + 1]);
          s[mt][0] = fmaf(dk_lo[b], tmp[0], s[mt][0]);
          s[mt][1] = fmaf(dk_lo[b], tmp[1], s[mt][1]);
          s[mt][2] = fmaf(dk_hi[b], tmp[2], s[mt][2]);
          s[mt][3] = fmaf(dk_hi[b], tmp[3], s[mt][3]);
        }
      }
    }

    // ---------------- online softmax over the page ----------------
    float pmax[2] = {-CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const bool v_lo = key0 + 16 * mt + r < ri.seq_len;
      const bool v_hi = key0 + 16 * mt + r + 8 < ri.seq_len;
      s[mt][0] = v_lo ? s[mt][0] * sl2 : -CUDART_INF_F;
      s[mt][1] = v_lo ? s[mt][1] * sl2 : -CUDART_INF_F;
      s[mt][2] = v_hi ? s[mt][2] * sl2 : -CUDART_INF_F;
      s[mt][3] = v_hi ? s[mt][3] * sl2 : -CUDART_INF_F;
      pmax[0] = fmaxf(pmax[0], fmaxf(s[mt][0], s[mt][2]));
      pmax[1] = fmaxf(pmax[1], fmaxf(s[mt][1], s[mt][3]));
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      pmax[0] = fmaxf(pmax[0], __shfl_xor_sync(0xFFFFFFFFu, pmax[0], o));
      pmax[1] = fmaxf(pmax[1], __shfl_xor_sync(0xFFFFFFFFu, pmax[1], o));
    }
    float alpha[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float mn = fmaxf(m_run[h], pmax[h]);
      alpha[h] = ex2(m_run[h] - mn);
      m_run[h] = mn;
      l_run[h] *= alpha[h];
    }
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      s[mt][0] = ex2(s[mt][0] - m_run[0]);
      s[mt][1] = ex2(s[mt][1] - m_run[1]);
      s[mt][2] = ex2(s[mt][2] - m_run[0]);
      s[mt][3] = ex2(s[mt][3] - m_run[1]);
      l_run[0] += s[mt][0] + s[mt][2];
      l_run[1] += s[mt][1] + s[mt][3];
    }
#pragma unroll
    for (int i = 0; i < KS; ++i) {
      o_acc[i][0] *= alpha[0];
      o_acc[i][1] *= alpha[1];
      o_acc[i][2] *= alpha[0];
      o_acc[i][3] *= alpha[1];
    }

    // ---------------- O^T += V^T P for the page ----------------
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      // P (keys x heads) from the S^T fragment layout to the B-operand layout:
      // this lane needs P[key 2c, 2c+1, 2c+8, 2c+9][head r].
      const int src0 = 8 * c + (r >> 1), src1 = src0 + 4;
      float f0[4], f1[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        f0[i] = __shfl_sync(0xFFFFFFFFu, s[mt][i], src0);
        f1[i] = __shfl_sync(0xFFFFFFFFu, s[mt][i], src1);
      }
      const bool odd = r & 1;
      const float p0 = odd ? f0[1] : f0[0];   // key 2c
      const float p1 = odd ? f1[1] : f1[0];   // key 2c+1
      const float p8 = odd ? f0[3] : f0[2];   // key 2c+8
      const float p9 = odd ? f1[3] : f1[2];   // key 2c+9
      const int kk0 = 16 * mt + 2 * c;        // the lane's four keys: kk0, kk0+1, kk0+8, kk0+9

      // V words of the four keys, per block
      uint32_t bfr[NB][2];
      if (FV == MIXATTN_KV_F16) {
        bfr[0][0] = pack_f16x2(p0, p1);
        bfr[0][1] = pack_f16x2(p8, p9);
      } else {
        float dv[4][NB];
        const int keys[4] = {kk0, kk0 + 1, kk0 + 8, kk0 + 9};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (NB == 4) {
            uint2 a = ldg_u64(vsc + keys[k] * NB);
            dv[k][0] = __half2float(__ushort_as_half(a.x & 0xFFFF));
            dv[k][1] = __half2float(__ushort_as_half(a.x >> 16));
            dv[k][2 % NB] = __half2float(__ushort_as_half(a.y & 0xFFFF));
            dv[k][3 % NB] = __half2float(__ushort_as_half(a.y >> 16));
          } else {
            uint32_t a = ldg_u32(vsc + keys[k] * NB);
            dv[k][0] = __half2float(__ushort_as_half(a & 0xFFFF));
            dv[k][1 % NB] = __half2float(__ushort_as_half(a >> 16));
          }
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          // p == 0 (masked or underflowed) stays 0 whatever the scale holds
          bfr[b][0] = pack_f16x2(p0 != 0.f ? p0 * dv[0][b] : 0.f, p1 != 0.f ? p1 * dv[1][b] : 0.f);
          bfr[b][1] = pack_f16x2(p8 != 0.f ? p8 * dv[2][b] : 0.f, p9 != 0.f ? p9 * dv[3][b] : 0.f);
        }
      }

#pragma unroll
      for (int b = 0; b < NB; ++b) {
        uint32_t a_u0[4], a_u1[4];  // A fragments of M-tiles 2b (u=0) and 2b+1 (u=1)
        const uint32_t* bb = (FV == MIXATTN_KV_F16) ? bfr[0] : bfr[b];
        if (FV == MIXATTN_KV_Q8_0) {
          const uint32_t w0 = ldg_u32(vq + (kk0)*RBV + 32 * b + 4 * r);
          const uint32_t w1 = ldg_u32(vq + (kk0 + 1) * RBV + 32 * b + 4 * r);
          const uint32_t w8 = ldg_u32(vq + (kk0 + 8) * RBV + 32 * b + 4 * r);
          const uint32_t w9 = ldg_u32(vq + (kk0 + 9) * RBV + 32 * b + 4 * r);
          s8x4_to_f16x2x2(prmt(w0, w1, 0x5140u), a_u0[0], a_u0[1]);
          s8x4_to_f16x2x2(prmt(w8, w9, 0x5140u), a_u0[2], a_u0[3]);
          s8x4_to_f16x2x2(prmt(w0, w1, 0x7362u), a_u1[0], a_u1[1]);
          s8x4_to_f16x2x2(prmt(w8, w9, 0x7362u), a_u1[2], a_u1[3]);
        } else if (FV == MIXATTN_KV_Q4_0) {
          const uint32_t h0 = ldg_u16(vq + (kk0)*RBV + 16 * b + 2 * r);
          const uint32_t h1 = ldg_u16(vq + (kk0 + 1) * RBV + 16 * b + 2 * r);
          const uint32_t h8 = ldg_u16(vq + (kk0 + 8) * RBV + 16 * b + 2 * r);
          const uint32_t h9 = ldg_u16(vq + (kk0 + 9) * RBV + 16 * b + 2 * r);
          const uint32_t x01 = prmt(h0, h1, 0x5140u), x89 = prmt(h8, h9, 0x5140u);
          u4x4_to_f16x2x2(x01 & 0x0F0F0F0Fu, a_u0[0], a_u0[1]);
          u4x4_to_f16x2x2(x89 & 0x0F0F0F0Fu, a_u0[2], a_u0[3]);
          u4x4_to_f16x2x2((x01 >> 4) & 0x0F0F0F0Fu, a_u1[0], a_u1[1]);
          u4x4_to_f16x2x2((x89 >> 4) & 0x0F0F0F0Fu, a_u1[2], a_u1[3]);
        } else {
          // fp16 values: zero the words of keys past the row so stale data never reaches the MMA
          const bool v0 = key0 + kk0 < ri.seq_len, v1 = key0 + kk0 + 1 < ri.seq_len;
          const bool v8 = key0 + kk0 + 8 < ri.seq_len, v9 = key0 + kk0 + 9 < ri.seq_len;
          uint2 e0 = ldg_u64(vq + (kk0)*RBV + 2 * (32 * b + 4 * r));
          uint2 e1 = ldg_u64(vq + (kk0 + 1) * RBV + 2 * (32 * b + 4 * r));
          uint2 e8 = ldg_u64(vq + (kk0 + 8) * RBV + 2 * (32 * b + 4 * r));
          uint2 e9 = ldg_u64(vq + (kk0 + 9) * RBV + 2 * (32 * b + 4 * r));
          if (!v0) e0 = make_uint2(0u, 0u);
          if (!v1) e1 = make_uint2(0u, 0u);
          if (!v8) e8 = make_uint2(0u, 0u);
          if (!v9) e9 = make_uint2(0u, 0u);
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
  }

  // ---------------- warp partial -> shared memory ----------------
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    l_run[0] += __shfl_xor_sync(0xFFFFFFFFu, l_run[0], o);
    l_run[1] += __shfl_xor_sync(0xFFFFFFFFu, l_run[1], o);
  }
  float* ws = reinterpret_cast<float*>(smem);
  float* wm = ws + warp * DecodeSmem<D>::kPerWarp;  // m[8], l[8], O[8][D]
  const int h0 = 2 * c, h1 = 2 * c + 1;
  if (r == 0) {
    if (h0 < G) { wm[h0] = m_run[0]; wm[8 + h0] = l_run[0]; }
    if (h1 < G) { wm[h1] = m_run[1]; wm[8 + h1] = l_run[1]; }
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
  __syncthreads();

  // ---------------- merge the 8 warps ----------------
  const int n_out = G * D;
  const int n_warps_used = min(kWarps, (t.count + ppw - 1) / ppw);
  const bool single = ri.n_splits == 1;
  float* part = p.partials + (int64_t)dec_idx * G * (D + 2);
  for (int idx = tid; idx < n_out; idx += kThreads) {
    const int h = idx / D, d = idx - h * D;
    float mmax = -CUDART_INF_F;
    for (int w = 0; w < n_warps_used; ++w) mmax = fmaxf(mmax, ws[w * DecodeSmem<D>::kPerWarp + h]);
    float lsum = 0.f, osum = 0.f;
    for (int w = 0; w < n_warps_used; ++w) {
      const float* x = ws + w * DecodeSmem<D>::kPerWarp;
      const float sc = ex2(x[h] - mmax);
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
  __syncthreads();
  __shared__ int s_last;
  if (tid == 0) {
    const unsigned prev = atomicAdd(&p.counters[(int64_t)t.row * p.hkv + g], 1u);
    s_last = (prev == (unsigned)(ri.n_splits - 1));
  }
  __syncthreads();
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
      const float sc = ex2(__ldcg(x + G * D + 2 * h) - mmax);
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
  lo = hfma2_u32(v, s, hi ^ 0x80008000u);
}

// Dequantise one 128-key x D tile from the raw stage into swizzled fp16 tiles
// (hi, and lo for quantised formats).  Keys at or past `valid_keys` (relative
// to the tile) are written as zeros.
template <int F, int D, bool LO>
__device__ __forceinline__ void dequant_tile(const uint8_t* raw_q, const uint8_t* raw_s, uint8_t* dst_hi,
                                             uint8_t* dst_lo, int valid_keys) {
  constexpr int NB = D / kBlock;
  constexpr int CPR = D / 8;  // 16-byte fp16 chunks per key row
  constexpr int RB = F == MIXATTN_KV_F16 ? 2 * D : (F == MIXATTN_KV_Q8_0 ? D : D / 2);
  constexpr int PAGE_Q = kPage * RB;
  constexpr int PAGE_S = kPage * NB * 2;
  for (int k = threadIdx.x; k < kChunkN * CPR; k += kThreads) {
    const int key = k / CPR, dc = k - key * CPR;
    const int pj = key >> 5, kr = key & 31;
    uint4 hi = make_uint4(0u, 0u, 0u, 0u), lo = make_uint4(0u, 0u, 0u, 0u);
    if (key < valid_keys) {
      const uint8_t* qrow = raw_q + pj * PAGE_Q + kr * RB;
      if (F == MIXATTN_KV_F16) {
        hi = *reinterpret_cast<const uint4*>(qrow + 16 * dc);
      } else {
        const int b = dc >> 2;
        const uint16_t sh = *reinterpret_cast<const uint16_t*>(raw_s + pj * PAGE_S + (kr * NB + b) * 2);
        const uint32_t s2 = (uint32_t)sh | ((uint32_t)sh << 16);
        uint32_t h0, h1, h2, h3;
        if (F == MIXATTN_KV_Q8_0) {
          const uint2 w = *reinterpret_cast<const uint2*>(qrow + 8 * dc);
          s8x4_to_f16x2x2(w.x, h0, h1);
          s8x4_to_f16x2x2(w.y, h2, h3);
        } else {
          const int e = dc & 3;  // 8-element group of the block: 0,1 low nibbles; 2,3 high nibbles
          const uint2 w = *reinterpret_cast<const uint2*>(qrow + 16 * b + 8 * (e & 1));
          const int shift = (e >> 1) * 4;
          u4x4_to_f16x2x2((w.x >> shift) & 0x0F0F0F0Fu, h0, h1);
          u4x4_to_f16x2x2((w.y >> shift) & 0x0F0F0F0Fu, h2, h3);
        }
        split_hilo(h0, s2, hi.x, lo.x);
        split_hilo(h1, s2, hi.y, lo.y);
        split_hilo(h2, s2, hi.z, lo.z);
        split_hilo(h3, s2, hi.w, lo.w);
      }
    }
    const int half = dc >> 3, cc = dc & 7;
    const uint32_t off = half * (kChunkN * 128) + sw128_off(key, cc);
    *reinterpret_cast<uint4*>(dst_hi + off) = hi;
    if (LO) *reinterpret_cast<uint4*>(dst_lo + off) = lo;
  }
}

template <int FK, int FV, int D>
__device__ __forceinline__ void chunk_tile(const AttnParams& p, const TileDesc& t, uint8_t* smem_raw,
                                           unsigned int* err) {
  using L = ChunkSmem<FK, FV, D>;
  constexpr int NB = D / kBlock;
  constexpr uint32_t kTmemCols = 256;  // S: 128 columns (P, fp16, overwrites its first 64); O: D columns
  constexpr uint32_t kSCol = 0, kOCol = 128;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* s_done = full + 1;
  uint64_t* o_done = full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(full + 3);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int G = p.group, lg = p.log2_group;
  const int g = t.kvh;
  const RowInfo ri = p.rows[t.row];
  const int n_pages_row = (ri.seq_len + kPage - 1) / kPage;
  // keys this tile can see: up to the position of its last query
  const int key_end = min(ri.seq_len, ri.q_offset + t.begin + t.count);
  const int n_kv = (key_end + kChunkN - 1) / kChunkN;
  const int32_t* pt_row = p.page_table + (int64_t)t.row * p.max_pages;

  if (tid == 0) {
    mbar_init(full, 1);
    mbar_init(s_done, 1);
    mbar_init(o_done, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }

  // ---- Q tile: row i = token (i >> lg), head (i & (G-1)) -> swizzled fp16 ----
  {
    constexpr int CPR = D / 8;
    for (int k = tid; k < kChunkM * CPR; k += kThreads) {
      const int row = k / CPR, dc = k - row * CPR;
      const int tok = row >> lg, h = row & (G - 1);
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (tok < t.count) {
        const uint16_t* src = static_cast<const uint16_t*>(p.q) +
                              ((int64_t)(ri.q_start + t.begin + tok) * p.hq + (int64_t)g * G + h) * D + 8 * dc;
        v = ldg_u128(src);
      }
      *reinterpret_cast<uint4*>(smem + L::kQ + (dc >> 3) * (kChunkM * 128) + sw128_off(row, dc & 7)) = v;
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // ---- producer: raw pages of KV tile jj into the stage ----
  auto issue_raw = [&](int jj) {
    uint8_t* raw = smem + L::kRaw;
    uint32_t bytes = 0;
    int pids[L::kPagesPerTile];
#pragma unroll
    for (int pj = 0; pj < L::kPagesPerTile; ++pj) {
      const int pg = jj * L::kPagesPerTile + pj;
      int pid = -1;
      if (pg < n_pages_row && pg * kPage < key_end) {
        pid = pt_row[pg];
        if (pid < 0 || pid >= p.num_pages) {
          set_device_error(err, MIXATTN_DEVERR_PAGE_ID);
          pid = -1;
        }
      }
      pids[pj] = pid;
      if (pid >= 0) bytes += L::kKqPage + L::kKsPage + L::kVqPage + L::kVsPage;
    }
    mbar_arrive_expect_tx(full, bytes);
#pragma unroll
    for (int pj = 0; pj < L::kPagesPerTile; ++pj) {
      const int pid = pids[pj];
      if (pid < 0) continue;
      const int64_t prow = ((int64_t)pid * p.hkv + g) * kPage;  // first plane row of (page, head)
      bulk_g2s(raw + L::kRawKq + pj * L::kKqPage, p.k_quant + prow * (L::kKqPage / kPage), L::kKqPage, full);
      if (L::kKsPage) bulk_g2s(raw + L::kRawKs + pj * L::kKsPage, p.k_scale + prow * NB, L::kKsPage, full);
      bulk_g2s(raw + L::kRawVq + pj * L::kVqPage, p.v_quant + prow * (L::kVqPage / kPage), L::kVqPage, full);
      if (L::kVsPage) bulk_g2s(raw + L::kRawVs + pj * L::kVsPage, p.v_scale + prow * NB, L::kVsPage, full);
    }
  };

  const int issuer = 128;  // warp 4, lane 0: copies and MMAs
  int raw_issued = 0, raw_consumed = 0;
  if (tid == issuer) {
    issue_raw(0);
    raw_issued = 1;
  }

  // softmax state: thread i < 128 owns row i (TMEM lane i)
  const int row = tid & 127;
  const int tok = row >> lg;
  const bool row_valid = tid < 128 && tok < t.count;
  const int pos = ri.q_offset + t.begin + min(tok, t.count - 1);
  float m_run = -CUDART_INF_F, l_run = 0.f;
  const float sl2 = p.scale_log2;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  bool ok = true;
  int pv_issued = 0;

  constexpr uint32_t kIdescQK = idesc_f16_f32(128, kChunkN, false, false);
  constexpr uint32_t kIdescPV = idesc_f16_f32(128, D, false, true);
  const uint32_t sQ = smem_u32(smem + L::kQ);
  const uint32_t sKh = smem_u32(smem + L::kKh), sKl = smem_u32(smem + L::kKl);
  const uint32_t sVh = smem_u32(smem + L::kVh), sVl = smem_u32(smem + L::kVl);

  for (int j = 0; j < n_kv; ++j) {
    ok = mbar_wait(full, (uint32_t)(j & 1), err) && ok;
    raw_consumed = j + 1;
    if (j > 0) ok = mbar_wait(o_done, (uint32_t)((j - 1) & 1), err) && ok;
    tc_fence_after();
    const uint8_t* raw = smem + L::kRaw;
    const int valid_keys = key_end - j * kChunkN;
    dequant_tile<FK, D, L::kKLo>(raw + L::kRawKq, raw + L::kRawKs, smem + L::kKh, smem + L::kKl, valid_keys);
    dequant_tile<FV, D, L::kVLo>(raw + L::kRawVq, raw + L::kRawVs, smem + L::kVh, smem + L::kVl, valid_keys);
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == issuer) {
      if (j + 1 < n_kv) {  // the stage is free again: the copy overlaps this tile's math
        issue_raw(j + 1);
        raw_issued = j + 2;
      }
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t off = (uint32_t)((ks >> 2) * (128 * 128) + (ks & 3) * 32);
        const uint64_t qd = sw128_desc(sQ + off, 16, 1024);
        tc_mma_ss(tmem + kSCol, qd, sw128_desc(sKh + off, 16, 1024), kIdescQK, ks > 0 ? 1u : 0u);
        if (L::kKLo) tc_mma_ss(tmem + kSCol, qd, sw128_desc(sKl + off, 16, 1024), kIdescQK, 1u);
      }
      tc_commit(s_done);
    }
    if (tid < 128) {
      ok = mbar_wait(s_done, (uint32_t)(j & 1), err) && ok;
      tc_fence_after();
      const int kbase = j * kChunkN;
      // pass 1: row max of the scaled, masked scores
      float mx = -CUDART_INF_F;
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + kSCol + 32 * ch, v);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int key = kbase + 32 * ch + e;
          const float x = key <= pos ? __uint_as_float(v[e]) * sl2 : -CUDART_INF_F;
          mx = fmaxf(mx, x);
        }
      }
      const float m_new = fmaxf(m_run, mx);
      const float alpha = ex2(m_run - m_new);
      // pass 2: P = 2^(s - m) as fp16 into TMEM over the consumed scores, row sums
      float sum = 0.f;
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + kSCol + 32 * ch, v);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int key = kbase + 32 * ch + e;
          const float x0 = key <= pos ? __uint_as_float(v[e]) * sl2 : -CUDART_INF_F;
          const float x1 = key + 1 <= pos ? __uint_as_float(v[e + 1]) * sl2 : -CUDART_INF_F;
          const float p0 = ex2(x0 - m_new), p1 = ex2(x1 - m_new);
          sum += p0 + p1;
          pk[e >> 1] = pack_f16x2(p0, p1);
        }
        tmem_st16(tmem + lane_base + kSCol + 16 * ch, pk);
      }
      l_run = l_run * alpha + sum;
      m_run = m_new;
      // rescale the running O (TMEM) when this row's max moved
      if (j > 0 && __any_sync(0xFFFFFFFFu, alpha != 1.0f)) {
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + kOCol + 32 * ch, v);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
          tmem_st32(tmem + lane_base + kOCol + 32 * ch, v);
        }
      }
      tmem_wait_st();
    }
    tc_fence_before();
    if (!__syncthreads_and(ok)) {  // a bounded wait gave up somewhere: leave together
      ok = false;
      break;
    }
    if (tid == issuer) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kChunkN / 16; ++kk) {
        const uint32_t pa = tmem + kSCol + 8 * kk;  // P columns of keys 16kk..16kk+15
        const uint32_t boff = (uint32_t)(kk * 16 * 128);
        const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
        tc_mma_ts(tmem + kOCol, pa, sw128_desc(sVh + boff, kChunkN * 128, 1024), kIdescPV, acc);
        if (L::kVLo) tc_mma_ts(tmem + kOCol, pa, sw128_desc(sVl + boff, kChunkN * 128, 1024), kIdescPV, 1u);
      }
      tc_commit(o_done);
      ++pv_issued;
    }
  }

  // ---- epilogue: O / l -> fp16 ----
  if (tid == issuer) {
    // nothing the issuer started may still be running when TMEM and the stage are released
    if (pv_issued > 0) mbar_wait(o_done, (uint32_t)((pv_issued - 1) & 1), err);
    if (raw_issued > raw_consumed) mbar_wait(full, (uint32_t)((raw_issued - 1) & 1), err);
  }
  if (tid < 128 && ok) ok = mbar_wait(o_done, (uint32_t)((n_kv - 1) & 1), err);
  if (tid < 128) {
    tc_fence_after();
    const float inv_l = (l_run > 0.f) ? 1.f / l_run : 0.f;
    uint16_t* dst = static_cast<uint16_t*>(p.o) +
                    ((int64_t)(ri.q_start + t.begin + tok) * p.hq + (int64_t)g * G + (row & (G - 1))) * D;
#pragma unroll 1
    for (int ch = 0; ch < D / 32; ++ch) {
      uint32_t v[32];
      tmem_ld32(tmem + lane_base + kOCol + 32 * ch, v);
      tmem_wait_ld();
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 32; e += 2)
        pk[e >> 1] = pack_f16x2(__uint_as_float(v[e]) * inv_l, __uint_as_float(v[e + 1]) * inv_l);
      if (row_valid && ok) {
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          *reinterpret_cast<uint4*>(dst + 32 * ch + 8 * q4) =
              make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ===========================================================================
// Kernels
// ===========================================================================
template <int FK, int FV, int D>
__global__ void __launch_bounds__(kThreads, 1) mixed_attention_kernel(AttnParams p, unsigned int* err) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tile = blockIdx.x;
  if (tile < p.n_chunk_tiles) {
    chunk_tile<FK, FV, D>(p, p.tiles[tile], smem, err);
  } else {
    decode_tile<FK, FV, D>(p, p.tiles[tile], tile - p.n_chunk_tiles, smem, err);
  }
}

template <int FK, int FV, int D>
__global__ void __launch_bounds__(kThreads, 1) decode_attention_kernel(AttnParams p, unsigned int* err) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tile = blockIdx.x + p.n_chunk_tiles;
  decode_tile<FK, FV, D>(p, p.tiles[tile], blockIdx.x, smem, err);
}

template <int FK, int FV, int D>
cudaError_t launch_attention_t(const AttnParams& p, unsigned int* err, cudaStream_t s) {
  const int n_tiles = p.n_chunk_tiles + p.n_decode_tiles;
  if (n_tiles == 0) return cudaSuccess;
  if (p.n_chunk_tiles == 0) {
    const size_t sm = DecodeSmem<D>::kTotal;
    decode_attention_kernel<FK, FV, D><<<p.n_decode_tiles, kThreads, sm, s>>>(p, err);
    return cudaGetLastError();
  }
  const size_t sm = ChunkSmem<FK, FV, D>::kTotal;
  static bool configured = false;  // per process; the attribute is per function
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(mixed_attention_kernel<FK, FV, D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  mixed_attention_kernel<FK, FV, D><<<n_tiles, kThreads, sm, s>>>(p, err);
  return cudaGetLastError();
}

}  // namespace mixattn
