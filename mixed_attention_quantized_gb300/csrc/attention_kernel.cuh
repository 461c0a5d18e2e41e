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
// XOR swizzle so the ldmatrix reads are conflict free) and runs QK^T and PV on
// mma.sync m16n8k16 with the G query heads in rows of QK's A and the N=8
// dimension of PV.  Quantised codes reach the tensor cores as exact fp16
// subnormals (one or two logic ops per pair of codes, the code offset taken out
// through the accumulator start and one extra MMA per block); the Q8_0 / Q4_0
// scales are applied in fp32: per key and 32-d block on the scores, and folded
// into P per key and block on the values.  Warp partials are merged in shared
// memory, split partials by the last CTA of the (row, kv head) to finish
// (atomic ticket, no spin).
//
// Chunk tiles (tensor-bound): a CTA of 16 warps owns 128 rows = 128/G query
// tokens x G heads of one kv head.  Two dequant warp groups load the raw K and V
// bytes straight from the cache and write 128-byte-swizzled fp16 operand tiles
// -- an exact hi/lo pair for quantised formats, since d*q needs up to 18
// significant bits; one thread issues every tcgen05.mma (S = Q K^T and O += P V,
// one MMA per half, Q, S, P and O in TMEM); a softmax warp group, one TMEM lane
// (query row) per thread, turns S into P in place.  K, S and P are double-buffered,
// so QK of the next tile, the dequantisation and the next softmax overlap this
// tile's PV.
#pragma once

#include <algorithm>
#include <atomic>
#include <mutex>

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
// 128-byte line index mod 8), so every ldmatrix read (8 keys x one 16-byte
// chunk) hits 8 distinct bank groups; then the 16 keys' raw K and V scale rows.
// Beside its ring each warp keeps the scales of the M-tile it is working on as
// fp32, [K | V][block][lane quad c][4]: the quad c = 0..3 holding keys 2c, 2c+1,
// 2c+8, 2c+9 reads its four scales of one block with one 16-byte load.
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
  // fp32 scales of the current M-tile, per warp: K then V, 16 keys x D/32 blocks each
  static constexpr int kFsK = FK == MIXATTN_KV_F16 ? 0 : 64 * kNb;
  static constexpr int kFs = kFsK + (FV == MIXATTN_KV_F16 ? 0 : 64 * kNb);
  __host__ __device__ static constexpr int kWarpBytes(int ns) { return ns * kStage + kFs; }
  // after the rings, shared by the tile's warps, [16-byte word j][lane]: the lanes' Q
  // fragments (D/16 k-steps x 2 words), score-accumulator starts (4 floats),
  // one-hot words of the value correction (4) and the K-scale multiplier (1 float)
  static constexpr int kQBytes = (kNb + 3) * 512;
  __host__ __device__ static constexpr int q_off(int ns) { return kWarps * kWarpBytes(ns); }
  static constexpr int stages_for(int budget) {
    return (budget - kWarps * kFs - kQBytes) / (kWarps * kStage) > 8
               ? 8
               : ((budget - kWarps * kFs - kQBytes) / (kWarps * kStage) < 2
                      ? 2
                      : (budget - kWarps * kFs - kQBytes) / (kWarps * kStage));
  }
  // after the page loop the same memory holds the warp partials: m[8], l[8], O[8][D]
  static constexpr int kPerWarp = 16 + kMaxGroup * D;
  static constexpr int kMerge = kWarps * kPerWarp * 4;
  static constexpr int total(int ns) {
    return (q_off(ns) + kQBytes > kMerge ? q_off(ns) + kQBytes : kMerge) + 16;
  }
  // decode-only launches: two CTAs per SM when two stages per warp fit in 113 KB
  // (half an SM's shared memory less the per-CTA reserve), else one CTA per SM
  // with a deeper ring
  static constexpr int kPairBudget = 113 * 1024;
  static constexpr bool kTwoPerSm = kWarps * kWarpBytes(2) + kQBytes <= kPairBudget;
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

// Four 8x8 b16 matrices from shared memory; the rows of matrix m are the 16-byte
// rows at the addresses of lanes 8m .. 8m+7.  Lane 4i + j receives elements
// (i, 2j) and (i, 2j+1) of each matrix; with .trans, elements (2j, i) and
// (2j+1, i).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// ldmatrix plan of one 16-key M-tile of `RB`-byte rows: its 2 x RB/16 tiles
// (n-tile nt = keys 8nt..8nt+7, 16-byte chunk ch), tile t = nt * kCh + ch, go
// four to a load; load L covers tiles 4L .. 4L+3.
template <int RB>
struct LdsmPlan {
  static constexpr int kCh = RB / 16;                     // chunks per key row
  static constexpr int kGroups = kCh >= 4 ? kCh / 4 : 1;  // loads per n-tile (1 load for both when kCh == 2)
  static constexpr int kLoads = kCh >= 4 ? kCh / 2 : 1;
  // the n-tile 1 load of a group sits 8 rows further, the same swizzle phase
  static constexpr bool kNtAdds = (8 * RB) % 1024 == 0;
  static constexpr int kOffs = kNtAdds || kCh < 4 ? kGroups : 2 * kGroups;
  // the lane's row address (offset in the staged region) for load L
  static __device__ __forceinline__ int lane_off(int L, int lane) {
    const int t = 4 * L + (lane >> 3);
    const int nt = t / kCh, ch = t - nt * kCh;
    return swz((8 * nt + (lane & 7)) * RB + 16 * ch);
  }
};

// Words of chunks 4h .. 4h+3 of both n-tiles (kCh == 2: chunks 0, 1 of both,
// in w0[0..1] and w1[0..1]).
template <int RB, bool TRANS>
__device__ __forceinline__ void ldsm_group(uint32_t base, const int (&off)[LdsmPlan<RB>::kOffs], int h,
                                           uint32_t (&w0)[4], uint32_t (&w1)[4]) {
  using P = LdsmPlan<RB>;
  if (P::kCh < 4) {
    uint32_t r[4];
    if (TRANS) ldsm_x4_t(base + off[0], r); else ldsm_x4(base + off[0], r);
    w0[0] = r[0]; w0[1] = r[1]; w1[0] = r[2]; w1[1] = r[3];
    w0[2] = w0[3] = w1[2] = w1[3] = 0u;
  } else {
    const uint32_t a0 = base + off[h];
    const uint32_t a1 = P::kNtAdds ? a0 + 8 * RB : base + off[P::kGroups + h];
    if (TRANS) { ldsm_x4_t(a0, w0); ldsm_x4_t(a1, w1); } else { ldsm_x4(a0, w0); ldsm_x4(a1, w1); }
  }
}

// Quantised codes -> fp16 subnormals: the 16-bit pattern holding a small
// unsigned integer u (< 1024) is the fp16 number u * 2^-24, exactly.
//   Q8_0: bytes 0 and 2 (even) or 1 and 3 (odd) of a word, sign bit flipped:
//         u = q + 128
//   Q4_0: low (u = n) or high (u = 16 n) nibble of bytes 0 and 2 (even) or 1 and 3 (odd)
__device__ __forceinline__ uint32_t q8_even(uint32_t w) { return (w ^ 0x80808080u) & 0x00FF00FFu; }
__device__ __forceinline__ uint32_t q8_odd(uint32_t w) { return ((w >> 8) ^ 0x00800080u) & 0x00FF00FFu; }
__device__ __forceinline__ uint32_t q4_lo_even(uint32_t w) { return w & 0x000F000Fu; }
__device__ __forceinline__ uint32_t q4_lo_odd(uint32_t w) { return (w >> 8) & 0x000F000Fu; }
__device__ __forceinline__ uint32_t q4_hi_even(uint32_t w) { return w & 0x00F000F0u; }
__device__ __forceinline__ uint32_t q4_hi_odd(uint32_t w) { return (w >> 8) & 0x00F000F0u; }

// Code offset of a format as an fp16 subnormal pair, negated: -128 * 2^-24
// (Q8_0) or -8 * 2^-24 (Q4_0).
template <int F>
__device__ __forceinline__ constexpr uint32_t neg_offset_pair() {
  return F == MIXATTN_KV_Q8_0 ? 0x80808080u : 0x80088008u;
}

// Head dimension held by row `rr` (0..15) of PV M-tile t.
//   quantised V: 32-d block t/2, half t%2, element 2(rr%8) + rr/8 of the half
//   fp16 V:      16t + rr
template <int FV>
__device__ __forceinline__ int pv_row_to_d(int t, int rr) {
  if (FV == MIXATTN_KV_F16) return 16 * t + rr;
  return 16 * t + 2 * (rr & 7) + (rr >> 3);
}

// Barrier over the 8 warps of a decode tile (a fused-launch CTA runs one tile
// on each half of its 16 warps, each half on its own named barrier).
__device__ __forceinline__ void decode_sync(int half) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + half), "n"(kThreads) : "memory");
}

__device__ __forceinline__ float h2f_lo(uint32_t x) { return __half2float(__ushort_as_half((unsigned short)(x & 0xFFFFu))); }
__device__ __forceinline__ float h2f_hi(uint32_t x) { return __half2float(__ushort_as_half((unsigned short)(x >> 16))); }

// One decode tile: a page range of one (row, kv head), 8 warps, each warp
// walking its own pages 16 keys (one M-tile) at a time.
//
// Quantised K and V reach the tensor cores as fp16 subnormals: the 16-bit
// pattern of a small unsigned integer u is the fp16 number u * 2^-24 exactly,
// so one or two logic ops per pair of codes make an exact operand (Q8_0:
// u = q + 128; Q4_0: u = n, or 16 n for the high nibble, which the matching Q
// entries take as q / 16 or the epilogue divides out).  The code offset is
// taken out exactly where it is cheapest:
//   scores: the block's accumulator starts at -offset * sum(q over the block) * 2^-24,
//           so the MMA ends on sum q * (u - offset) * 2^-24;
//   values: O += V_u^T P' per block, and one more MMA per block with a one-hot
//           A row of -offset * 2^-24 sums the same fp16 P' into row b of `corr`,
//           added to the block's rows at the end.
// The 2^24 is folded into the softmax scale (scores) and the epilogue (values).
template <int FK, int FV, int D, int NS>
__device__ __forceinline__ void decode_tile(const AttnParams& p, const TileDesc& t, uint8_t* smem, unsigned int* err,
                                            int half) {
  using S = DecodeSmem<FK, FV, D>;
  constexpr int NB = D / kBlock;   // scale blocks per row
  constexpr int KS = D / 16;       // k-steps of QK / M-tiles of PV
  constexpr int RBK = row_bytes<FK, D>();
  constexpr int RBV = row_bytes<FV, D>();
  constexpr bool QK = FK != MIXATTN_KV_F16;
  constexpr bool QV = FV != MIXATTN_KV_F16;
  using PK = LdsmPlan<RBK>;
  using PV = LdsmPlan<RBV>;
  constexpr float kTwo24 = 16777216.f;
  constexpr float kTwoM24 = 5.9604644775390625e-8f;

  // `half`: which 8 warps of the CTA run this tile (a fused-launch CTA runs two)
  const int tid = threadIdx.x - half * kThreads, warp = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, c = lane & 3;
  const int G = p.group;
  const int g = t.kvh;
  const RowInfo ri = p.rows[t.row];
  const int split = t.part;
  // The tile's R = nq * G rows are (query, head) pairs: row rr is query qg0 + rr / G of
  // the row (position q_offset + that) and head rr % G of kv head g.  A decode row has
  // one query; a short chunk row (speculative verify) has up to 8 / G per tile.
  const int qg0 = t.kv1, nq = t.nsplit, R = nq * G;
  const int my_q = qg0 + (r < R ? (r >> p.log2_group) : 0), my_h = r & (G - 1);
  const int pos = ri.q_offset + my_q;                // this lane's row sees keys lo .. pos
  const int lo = window_first_key(pos, p.window);    // (a sliding window starts at lo)
  // an M-tile needs masks when it reaches past the group's earliest query or
  // before its latest window start (the same bounds for every lane)
  const int mask_hi = ri.q_offset + qg0 + 1;
  const int mask_lo = window_first_key(ri.q_offset + qg0 + nq - 1, p.window);
  // the tile's pages spread evenly over its 8 warps (runs differing by at most one
  // page, each at most ppw), so a row's shorter last split also keeps every warp busy
  const int pg_base = t.count / kWarps, pg_rem = t.count - pg_base * kWarps;
  const int wp0 = t.begin + warp * pg_base + min(warp, pg_rem);
  const int wp1 = wp0 + pg_base + (warp < pg_rem ? 1 : 0);
  const int n_mt = wp1 > wp0 ? 2 * (wp1 - wp0) : 0;  // the warp's M-tiles (16 keys each)

  // ---- Q as the A operand of S = Q K^T: tile row r in M row r (rows 8..15 zero) ----
  // quantised K: k-step 2b+j covers dims 32b + 16j + 4c + {0, 2} (a0) and {1, 3}
  //   (a2), the order of the subnormal pairs of one K word; for Q4_0 the j = 1
  //   k-step (high nibbles, 16 n) takes q * sigma / 16 (see below)
  // fp16 K: k-step ks covers dims 16ks + 2c + {0, 1} (a0) and {8, 9} (a2)

  float o_acc[KS][4];
#pragma unroll
  for (int i = 0; i < KS; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
  float corr[4] = {0.f, 0.f, 0.f, 0.f};  // quantised V: row b, tile rows 2c, 2c+1
  float m_run = -CUDART_INF_F, l_run = 0.f;  // tile row r, in log2 units

  const int32_t* pt_row = p.page_table + (int64_t)t.row * p.max_pages;
  const uint32_t ring_s = smem_u32(smem) + warp * S::kWarpBytes(NS);
  const uint32_t fs_s = ring_s + NS * S::kStage;  // fp32 scales of the current M-tile
  int offk[PK::kOffs], offv[PV::kOffs];
#pragma unroll
  for (int i = 0; i < PK::kOffs; ++i) offk[i] = PK::lane_off(i, lane);
#pragma unroll
  for (int i = 0; i < PV::kOffs; ++i) offv[i] = PV::lane_off(i, lane);
  // cp.async destinations: chunk lane + 32k of a region sits at cpo[k & 1] + 512 (k & ~1)
  // (the swizzle repeats every 1024 bytes)
  const int cpo0 = swz(16 * lane), cpo1 = swz(16 * lane + 512);

  // The warp's page ids, lane j holding page wp0 + j (at most 32 a warp); a page
  // outside the cache is flagged once and skipped.
  const int n_pg = wp1 > wp0 ? wp1 - wp0 : 0;
  int my_pid = lane < n_pg ? pt_row[wp0 + lane] : 0;
  const bool pid_ok = my_pid >= 0 && my_pid < p.num_pages;
  const uint32_t page_ok = __ballot_sync(0xFFFFFFFFu, pid_ok);
  if (lane < n_pg && !pid_ok) set_device_error(err, MIXATTN_DEVERR_PAGE_ID);

  // Issue the copies of the warp's M-tile i into its stage, then close the group
  // (an empty group for i past the end keeps the group count uniform).
  int st_issue = 0;  // ring stage of the next M-tile to issue (M-tile i -> stage i % NS)
  auto issue = [&](int i) {
    if (i < n_mt) {
      const int mt = i & 1;
      const int pid = __shfl_sync(0xFFFFFFFFu, my_pid, i >> 1);
      if ((page_ok >> (i >> 1)) & 1u) {
        const uint32_t st = ring_s + st_issue * S::kStage;
        const int64_t prow = (int64_t)pid * p.hkv + g;  // (page, kv head) plane
        const uint8_t* kq = p.k_quant + prow * (kPage * RBK) + (16 * mt * RBK + 16 * lane);
        const uint8_t* vq = p.v_quant + prow * (kPage * RBV) + (16 * mt * RBV + 16 * lane);
#pragma unroll
        for (int k = 0; k < RBK / 32; ++k)
          cp_async16_s(st + S::kK + ((k & 1) ? cpo1 : cpo0) + 512 * (k & ~1), kq + 512 * k);
#pragma unroll
        for (int k = 0; k < RBV / 32; ++k)
          cp_async16_s(st + S::kV + ((k & 1) ? cpo1 : cpo0) + 512 * (k & ~1), vq + 512 * k);
        constexpr int SC = S::kSc / 16;  // 16-byte chunks of one scale slice
        const int64_t so = prow * (kPage * NB * 2) + 16 * mt * NB * 2;
        if (FK != MIXATTN_KV_F16 && lane < SC)
          cp_async16_s(st + S::kKs + 16 * lane, reinterpret_cast<const uint8_t*>(p.k_scale) + so + 16 * lane);
        if (FV != MIXATTN_KV_F16 && lane >= 16 && lane < 16 + SC)
          cp_async16_s(st + S::kVs + 16 * (lane - 16),
                       reinterpret_cast<const uint8_t*>(p.v_scale) + so + 16 * (lane - 16));
      }
    }
    cp_async_commit();
    st_issue = st_issue + 1 == NS ? 0 : st_issue + 1;
  };

#pragma unroll
  for (int i = 0; i < NS - 1; ++i) issue(i);

  // (after the first copies are under way) written once by warp 0 into the tile's Q
  // block: word j (j < NB) of a lane holds the
  // fragments of k-steps 2j, 2j+1 (a0, a2 each), word NB the four block starts, word
  // NB + 1 the one-hot words of the value correction
  const uint32_t q_s = smem_u32(smem) + S::q_off(NS);
  if (warp == 0) {
    uint32_t qa[KS][2];
    float cb[4] = {0.f, 0.f, 0.f, 0.f};  // start of block b's score accumulator (tile row r)
    const bool real = r < R;
    const uint16_t* qrow =
        static_cast<const uint16_t*>(p.q) + ((int64_t)(ri.q_start + my_q) * p.hq + (int64_t)g * G + my_h) * D;
    // Q4_0 K: the high-nibble k-steps take q / 16, an fp16 subnormal (losing bits) for
    // |q| below ~1e-3.  The tile's queries are scaled by one power of two sigma (exact)
    // that puts their largest element in [1024, 2048); 1 / sigma joins the K scales
    // when they are converted to fp32 (below), so the loop pays four multiplies per
    // 16 keys.  Other formats keep sigma = 1.
    float sig = 1.f;
    if (FK == MIXATTN_KV_Q4_0) {
      float mx = 0.f;
      if (real) {
#pragma unroll
        for (int b = 0; b < NB; ++b)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const uint2 v = ldg_u64(qrow + 32 * b + 16 * j + 4 * c);
            mx = fmax3(mx, fabsf(h2f_lo(v.x)), fabsf(h2f_hi(v.x)));
            mx = fmax3(mx, fabsf(h2f_lo(v.y)), fabsf(h2f_hi(v.y)));
          }
      }
#pragma unroll
      for (int sh = 1; sh < 32; sh <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, sh));
      // mx is 0 or an fp16 magnitude (exponent -24 .. 15): sigma = 2^(10 - exponent)
      if (mx > 0.f) sig = __uint_as_float((uint32_t)(264 - (int)((__float_as_uint(mx) >> 23) & 0xFF)) << 23);
    }
    if (!QK) {
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qa[ks][0] = real ? ldg_u32(qrow + 16 * ks + 2 * c) : 0u;
        qa[ks][1] = real ? ldg_u32(qrow + 16 * ks + 8 + 2 * c) : 0u;
      }
    } else {
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        float qs = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          uint2 v = ldg_u64(qrow + 32 * b + 16 * j + 4 * c);
          if (!real) v = make_uint2(0u, 0u);
          if (FK == MIXATTN_KV_Q4_0) {  // q * sigma, exact (a power of two into the normal range)
            v.x = pack_f16x2(h2f_lo(v.x) * sig, h2f_hi(v.x) * sig);
            v.y = pack_f16x2(h2f_lo(v.y) * sig, h2f_hi(v.y) * sig);
          }
          qs += (h2f_lo(v.x) + h2f_hi(v.x)) + (h2f_lo(v.y) + h2f_hi(v.y));
          uint32_t e = prmt(v.x, v.y, 0x5410u), o = prmt(v.x, v.y, 0x7632u);
          if (FK == MIXATTN_KV_Q4_0 && j == 1) {
            e = hmul2_u32(e, 0x2C002C00u);  // x 1/16
            o = hmul2_u32(o, 0x2C002C00u);
          }
          qa[2 * b + j][0] = e;
          qa[2 * b + j][1] = o;
        }
        qs += __shfl_xor_sync(0xFFFFFFFFu, qs, 1);
        qs += __shfl_xor_sync(0xFFFFFFFFu, qs, 2);
        cb[b] = qs * (FK == MIXATTN_KV_Q8_0 ? -128.f : -8.f) * kTwoM24;
      }
    }
#pragma unroll
    for (int j = 0; j < NB; ++j)
      sts128_s(q_s + 512 * j + 16 * lane, make_uint4(qa[2 * j][0], qa[2 * j][1], qa[2 * j + 1][0], qa[2 * j + 1][1]));
    sts128_s(q_s + 512 * NB + 16 * lane,
             make_uint4(__float_as_uint(cb[0]), __float_as_uint(cb[1]), __float_as_uint(cb[2]), __float_as_uint(cb[3])));
    const uint32_t off = neg_offset_pair<FV>();
    sts128_s(q_s + 512 * (NB + 1) + 16 * lane,
             make_uint4(r == 0 ? off : 0u, r == 1 ? off : 0u, r == 2 ? off : 0u, r == 3 ? off : 0u));
    if (FK == MIXATTN_KV_Q4_0 && lane == 0) sts32f_s(q_s + 512 * (NB + 2), 1.f / sig);  // a power of two: exact
  }
  decode_sync(half);

  // score scale (log2 units): 1/sqrt(D) and, for quantised K, the 2^24 of the subnormal codes
  const float sl2 = QK ? p.scale_log2 * kTwo24 : p.scale_log2;

  // scale conversion: lanes 0-15 take the K scales of key lane, lanes 16-31 the V scales
  // of key lane - 16, into slot (key & 1) + 2 (key >> 3) of quad (key & 7) / 2
  const bool sc_lane = lane >= 16 ? QV : QK;
  const int sc_src = (lane >= 16 ? S::kVs : S::kKs) + (lane & 15) * NB * 2;
  const uint32_t sc_dst =
      fs_s + (lane >= 16 ? S::kFsK : 0) + 4 * ((((lane & 7) >> 1) << 2) + (lane & 1) + (((lane >> 3) & 1) << 1));
  const int kv0 = 2 * c;  // the lane's keys in an M-tile: kv0, kv0+1 (n-tile 0), kv0+8, kv0+9 (n-tile 1)
  int st_cons = 0;
  for (int i = 0; i < n_mt; ++i) {
    issue(i + NS - 1);        // refills the stage consumed in the previous step
    cp_async_wait<NS - 1>();  // this lane's copies of M-tile i have landed
    __syncwarp();             // ... and every other lane's
    const uint32_t st_s = ring_s + st_cons * S::kStage;
    st_cons = st_cons + 1 == NS ? 0 : st_cons + 1;
    if ((page_ok >> (i >> 1)) & 1u) {
      const int key0 = (wp0 + (i >> 1)) * kPage + 16 * (i & 1);  // first key of the M-tile
      // some key of the M-tile lies outside some row's range
      const bool partial = key0 + 16 > mask_hi || key0 < mask_lo;
      auto seen = [&](int k) { return k <= pos && k >= lo; };  // visible to this lane's row

      // ---------------- scales of the M-tile -> fp32, one key per lane ----------------
      if (QK || QV) {
        if (sc_lane) {
          const uint32_t src = st_s + sc_src;
          const uint32_t dst = sc_dst;
          // multiplier of the converted scales: 1 / sigma for Q4_0 K, else 1 (read here, not
          // kept in a register across the loop)
          const float sc_mul = (FK == MIXATTN_KV_Q4_0 && lane < 16) ? lds32f_s(q_s + 512 * (NB + 2)) : 1.f;
          if (NB == 4) {
            const uint2 x = lds64_s(src);
            sts32f_s(dst, h2f_lo(x.x) * sc_mul);
            sts32f_s(dst + 64, h2f_hi(x.x) * sc_mul);
            sts32f_s(dst + 128, h2f_lo(x.y) * sc_mul);
            sts32f_s(dst + 192, h2f_hi(x.y) * sc_mul);
          } else {
            const uint32_t x = lds32_s(src);
            sts32f_s(dst, h2f_lo(x) * sc_mul);
            sts32f_s(dst + 64, h2f_hi(x) * sc_mul);
          }
        }
        __syncwarp();
      }

      // ---------------- S = Q K^T: head r x keys kv0, kv0+1 (s01), kv0+8, kv0+9 (s89) ----------------
      uint64_t s01, s89;
      if (QK) {
        s01 = s89 = 0ull;
        const float4 cbv = lds128f_s(q_s + 512 * NB + 16 * lane);
        // blocks per ldmatrix group: Q8_0 two chunks a block, Q4_0 one
        constexpr int BPG = FK == MIXATTN_KV_Q8_0 ? 2 : (NB < 4 ? NB : 4);
#pragma unroll
        for (int h = 0; h < PK::kGroups; ++h) {
          uint32_t w0[4], w1[4];  // K words of n-tiles 0 and 1 (keys r and r+8)
          ldsm_group<RBK, false>(st_s + S::kK, offk, h, w0, w1);
#pragma unroll
          for (int bb = 0; bb < BPG; ++bb) {
            const int b = h * BPG + bb;
            uint32_t k0[2][2], k1[2][2];  // [k-step 2b+j][b0, b1]
            if (FK == MIXATTN_KV_Q8_0) {
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                k0[j][0] = q8_even(w0[2 * bb + j]);
                k0[j][1] = q8_odd(w0[2 * bb + j]);
                k1[j][0] = q8_even(w1[2 * bb + j]);
                k1[j][1] = q8_odd(w1[2 * bb + j]);
              }
            } else {
              k0[0][0] = q4_lo_even(w0[bb]);
              k0[0][1] = q4_lo_odd(w0[bb]);
              k0[1][0] = q4_hi_even(w0[bb]);
              k0[1][1] = q4_hi_odd(w0[bb]);
              k1[0][0] = q4_lo_even(w1[bb]);
              k1[0][1] = q4_lo_odd(w1[bb]);
              k1[1][0] = q4_hi_even(w1[bb]);
              k1[1][1] = q4_hi_odd(w1[bb]);
            }
            const uint4 qv = lds128_s(q_s + 512 * b + 16 * lane);
            const float cbb = (b == 0 ? cbv.x : (b == 1 ? cbv.y : (b == 2 ? cbv.z : cbv.w)));
            const uint32_t a0[4] = {qv.x, 0u, qv.y, 0u};
            const uint32_t a1[4] = {qv.z, 0u, qv.w, 0u};
            float u0[4], u1[4];  // sum q (u - offset) 2^-24 over the block, keys kv0.. | kv0+8..
            mma_16816_c(u0, a0, k0[0], cbb, cbb, 0.f, 0.f);
            mma_16816(u0, a1, k0[1]);
            mma_16816_c(u1, a0, k1[0], cbb, cbb, 0.f, 0.f);
            mma_16816(u1, a1, k1[1]);
            const float4 dk = lds128f_s(fs_s + b * 64 + c * 16);
            s01 = ffma2(f2_pack(dk.x, dk.y), f2_pack(u0[0], u0[1]), s01);
            s89 = ffma2(f2_pack(dk.z, dk.w), f2_pack(u1[0], u1[1]), s89);
          }
        }
      } else {
        float u0[4] = {0.f, 0.f, 0.f, 0.f}, u1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int h = 0; h < PK::kGroups; ++h) {
          uint32_t w0[4], w1[4];  // chunks 4h .. 4h+3 = k-steps 2h, 2h+1
          ldsm_group<RBK, false>(st_s + S::kK, offk, h, w0, w1);
          const uint4 qv = lds128_s(q_s + 512 * h + 16 * lane);  // k-steps 2h, 2h+1
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const uint32_t a[4] = {j ? qv.z : qv.x, 0u, j ? qv.w : qv.y, 0u};
            const uint32_t b0[2] = {w0[2 * j], w0[2 * j + 1]};
            const uint32_t b1[2] = {w1[2 * j], w1[2 * j + 1]};
            mma_16816(u0, a, b0);
            mma_16816(u1, a, b1);
          }
        }
        s01 = f2_pack(u0[0], u0[1]);
        s89 = f2_pack(u1[0], u1[1]);
      }

      // ---------------- online softmax over the 16 keys (head r) ----------------
      float s[4];
      f2_unpack(s01, s[0], s[1]);
      f2_unpack(s89, s[2], s[3]);
      if (partial) {
        s[0] = seen(key0 + kv0) ? s[0] : -CUDART_INF_F;
        s[1] = seen(key0 + kv0 + 1) ? s[1] : -CUDART_INF_F;
        s[2] = seen(key0 + kv0 + 8) ? s[2] : -CUDART_INF_F;
        s[3] = seen(key0 + kv0 + 9) ? s[3] : -CUDART_INF_F;
      }
      // The reference m_run (per head, log2 units) follows the running maximum
      // lazily: it moves, and O, corr and l are rescaled, only when a score passes it
      // by more than kSlack.  Weights then stay <= 2^kSlack, so P' = p x scale stays
      // finite in fp16 for every scale a format can hold (Q4_0 |d| <= 8188, Q8_0
      // |d| <= 516), and the common M-tile needs one vote instead of a quad maximum.
      constexpr float kSlack = FV == MIXATTN_KV_Q4_0 ? 2.f : (FV == MIXATTN_KV_Q8_0 ? 6.f : 8.f);
      float pm = fmax3(s[0], s[1], fmaxf(s[2], s[3])) * sl2;  // this lane's maximum (scale > 0)
      if (__any_sync(0xFFFFFFFFu, pm > m_run + kSlack)) {  // also the first valid key (m_run = -inf)
        pm = fmaxf(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, 1));
        pm = fmaxf(pm, __shfl_xor_sync(0xFFFFFFFFu, pm, 2));
        const bool grow = pm > m_run + kSlack;
        const float alpha = grow ? ex2(m_run - pm) : 1.f;
        m_run = grow ? pm : m_run;
        l_run *= alpha;
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
        corr[0] *= a_even;
        corr[1] *= a_odd;
      }
      const float mref = m_run == -CUDART_INF_F ? 0.f : m_run;
      const float p0 = ex2(fmaf(s[0], sl2, -mref)), p1 = ex2(fmaf(s[1], sl2, -mref));
      const float p8 = ex2(fmaf(s[2], sl2, -mref)), p9 = ex2(fmaf(s[3], sl2, -mref));
      l_run += (p0 + p1) + (p8 + p9);

      // ---------------- O^T += V^T P' for the 16 keys ----------------
      // P is already in the B-operand layout: this lane holds P[key kv0.., kv0+9][head r];
      // quantised V takes P' = P x (the key's scale of the block) per block.
      uint32_t bq[QV ? NB : 1][2];
      if (QV) {
        const uint4 ohv = lds128_s(q_s + 512 * (NB + 1) + 16 * lane);  // one-hot rows of corr
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          const float4 dv = lds128f_s(fs_s + S::kFsK + b * 64 + c * 16);
          float x0, x1, x8, x9;
          f2_unpack(fmul2(f2_pack(p0, p1), f2_pack(dv.x, dv.y)), x0, x1);
          f2_unpack(fmul2(f2_pack(p8, p9), f2_pack(dv.z, dv.w)), x8, x9);
          if (partial) {  // p == 0 (a key past the row) stays 0 whatever its scale slot holds
            x0 = p0 != 0.f ? x0 : 0.f;
            x1 = p1 != 0.f ? x1 : 0.f;
            x8 = p8 != 0.f ? x8 : 0.f;
            x9 = p9 != 0.f ? x9 : 0.f;
          }
          bq[b][0] = pack_f16x2(x0, x1);
          bq[b][1] = pack_f16x2(x8, x9);
          // row b of corr += (-offset 2^-24) x sum over the keys of this fp16 P'
          const uint32_t oh = b == 0 ? ohv.x : (b == 1 ? ohv.y : (b == 2 ? ohv.z : ohv.w));
          const uint32_t ao[4] = {oh, 0u, oh, 0u};
          mma_16816(corr, ao, bq[b]);
        }
      } else {
        bq[0][0] = pack_f16x2(p0, p1);
        bq[0][1] = pack_f16x2(p8, p9);
      }

#pragma unroll
      for (int h = 0; h < PV::kGroups; ++h) {
        uint32_t w0[4], w1[4];  // transposed V words of n-tiles 0 and 1: keys (kv0, kv0+1) | (kv0+8, kv0+9)
        ldsm_group<RBV, true>(st_s + S::kV, offv, h, w0, w1);
        if (FV == MIXATTN_KV_Q8_0) {
          // chunk 4h+m is M-tile 4h+m: rows r, r+8 = its bytes 2r, 2r+1
          constexpr int MT = PV::kCh < 4 ? PV::kCh : 4;
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const int tt = 4 * h + m;
            const uint32_t a[4] = {q8_even(w0[m]), q8_odd(w0[m]), q8_even(w1[m]), q8_odd(w1[m])};
            mma_16816(o_acc[tt], a, bq[tt >> 1]);
          }
        } else if (FV == MIXATTN_KV_Q4_0) {
          // chunk b is block b: low nibbles M-tile 2b, high nibbles (16 n) M-tile 2b+1
          constexpr int BPG = NB < 4 ? NB : 4;
#pragma unroll
          for (int bb = 0; bb < BPG; ++bb) {
            const int b = h * BPG + bb;
            const uint32_t a_lo[4] = {q4_lo_even(w0[bb]), q4_lo_odd(w0[bb]), q4_lo_even(w1[bb]), q4_lo_odd(w1[bb])};
            const uint32_t a_hi[4] = {q4_hi_even(w0[bb]), q4_hi_odd(w0[bb]), q4_hi_even(w1[bb]), q4_hi_odd(w1[bb])};
            mma_16816(o_acc[2 * b], a_lo, bq[b]);
            mma_16816(o_acc[2 * b + 1], a_hi, bq[b]);
          }
        } else {
          // fp16: chunks 4h..4h+3 (8 dims each) are rows 0-7 / 8-15 of M-tiles 2h, 2h+1
          uint32_t mk0 = 0xFFFFFFFFu, mk1 = 0xFFFFFFFFu;
          if (partial) {  // zero the keys no row sees, so stale data never reaches the MMA
            const int lo_first = window_first_key(ri.q_offset + qg0, p.window);
            auto any_row = [&](int k) { return k < ri.seq_len && k >= lo_first; };
            mk0 = (any_row(key0 + kv0) ? 0x0000FFFFu : 0u) | (any_row(key0 + kv0 + 1) ? 0xFFFF0000u : 0u);
            mk1 = (any_row(key0 + kv0 + 8) ? 0x0000FFFFu : 0u) | (any_row(key0 + kv0 + 9) ? 0xFFFF0000u : 0u);
          }
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const uint32_t a[4] = {w0[2 * j] & mk0, w0[2 * j + 1] & mk0, w1[2 * j] & mk1, w1[2 * j + 1] & mk1};
            mma_16816(o_acc[2 * h + j], a, bq[0]);
          }
        }
      }
    }
    __syncwarp();  // every lane is done with this stage before it is refilled
  }
  cp_async_wait<0>();

  // ---------------- quantised V: take out the code offset and the 2^-24 ----------------
  if (QV) {
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float c0 = __shfl_sync(0xFFFFFFFFu, corr[0], 4 * b + c);
      const float c1 = __shfl_sync(0xFFFFFFFFu, corr[1], 4 * b + c);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int tt = 2 * b + u;
        const float f = (FV == MIXATTN_KV_Q4_0 && u == 1) ? 0.0625f : 1.f;
        o_acc[tt][0] = fmaf(o_acc[tt][0], f, c0) * kTwo24;
        o_acc[tt][1] = fmaf(o_acc[tt][1], f, c1) * kTwo24;
        o_acc[tt][2] = fmaf(o_acc[tt][2], f, c0) * kTwo24;
        o_acc[tt][3] = fmaf(o_acc[tt][3], f, c1) * kTwo24;
      }
    }
  }

  // ---------------- warp partial -> shared memory ----------------
  l_run += __shfl_xor_sync(0xFFFFFFFFu, l_run, 1);
  l_run += __shfl_xor_sync(0xFFFFFFFFu, l_run, 2);
  decode_sync(half);  // the staging rings are no longer needed: reuse them as merge scratch
  float* ws = reinterpret_cast<float*>(smem);
  float* wm = ws + warp * S::kPerWarp;  // m[8], l[8], O[8][D]
  const int h0 = 2 * c, h1 = 2 * c + 1;  // O columns: tile rows 2c, 2c+1
  if (c == 0 && r < R) {
    wm[r] = m_run;
    wm[8 + r] = l_run;
  }
#pragma unroll
  for (int tt = 0; tt < KS; ++tt) {
    const int d_lo = pv_row_to_d<FV>(tt, r), d_hi = pv_row_to_d<FV>(tt, r + 8);
    if (h0 < R) {
      wm[16 + h0 * D + d_lo] = o_acc[tt][0];
      wm[16 + h0 * D + d_hi] = o_acc[tt][2];
    }
    if (h1 < R) {
      wm[16 + h1 * D + d_lo] = o_acc[tt][1];
      wm[16 + h1 * D + d_hi] = o_acc[tt][3];
    }
  }
  decode_sync(half);

  // ---------------- merge the 8 warps ----------------
  // output of tile row rr: query qg0 + rr / G, head g * G + rr % G
  auto out_of = [&](int rr) {
    return static_cast<uint16_t*>(p.o) +
           ((int64_t)(ri.q_start + qg0 + (rr >> p.log2_group)) * p.hq + (int64_t)g * G + (rr & (G - 1))) * D;
  };
  const int n_out = R * D;
  const int n_warps_used = min(kWarps, t.count);
  const bool single = ri.n_splits == 1;
  const int slot_rows = p.slot_rows > 0 ? p.slot_rows : G;  // rows per partial slot
  // split partial: O [slot_rows][D], then (m, l) [slot_rows][2]; t.kv0 is the slot of split 0
  float* part = p.partials + (int64_t)(t.kv0 + split) * slot_rows * (D + 2);
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
      out_of(h)[d] = f16_out(osum / lsum);
    } else {
      part[h * D + d] = osum;
      if (d == 0) {
        part[slot_rows * D + 2 * h] = mmax;
        part[slot_rows * D + 2 * h + 1] = lsum;
      }
    }
  }
  if (single) return;

  // ---------------- the last CTA of the group's splits merges them ----------------
  __threadfence();
  decode_sync(half);
  __shared__ int s_last_of[2];
  int& s_last = s_last_of[half];
  if (tid == 0) {
    const unsigned prev = atomicAdd(&p.counters[t.kv0], 1u);  // one ticket per split group
    s_last = (prev == (unsigned)(ri.n_splits - 1));
  }
  decode_sync(half);
  if (!s_last) return;
  __threadfence();
  const int first = t.kv0;
  const int ns = ri.n_splits;
  const int64_t stride = (int64_t)slot_rows * (D + 2);
  for (int idx = tid; idx < n_out; idx += kThreads) {
    const int h = idx / D, d = idx - h * D;
    float mmax = -CUDART_INF_F;
    for (int s2 = 0; s2 < ns; ++s2) {
      const float* x = p.partials + (first + s2) * stride;
      mmax = fmaxf(mmax, __ldcg(x + slot_rows * D + 2 * h));
    }
    float lsum = 0.f, osum = 0.f;
    for (int s2 = 0; s2 < ns; ++s2) {
      const float* x = p.partials + (first + s2) * stride;
      const float mx = __ldcg(x + slot_rows * D + 2 * h);
      const float sc = mx == -CUDART_INF_F ? 0.f : ex2(mx - mmax);
      lsum += sc * __ldcg(x + slot_rows * D + 2 * h + 1);
      osum += sc * __ldcg(x + h * D + d);
    }
    out_of(h)[d] = f16_out(osum / lsum);
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
//
// CLAMP (Q8_0): a block whose largest magnitude is 65504 gets the scale
// fp16(65504/127) = 516, and 127 * 516 = 65532 rounds to infinity in fp16.
// hi is then clamped to +-65504 (the largest finite fp16, sign kept, one
// instruction); lo = 65532 - 65504 = 28 is still exact (a multiple of the
// scale's ulp, 0.5, far inside the fp16 range), so hi + lo == v*s holds for
// every code and scale.  Q4_0 needs no clamp: |q - 8| * |d| <= 8 * 8188 = 65504.
template <bool CLAMP>
__device__ __forceinline__ void split_hilo(uint32_t v, uint32_t s, uint32_t& hi, uint32_t& lo) {
  hi = hmul2_u32(v, s);
  if (CLAMP) asm("min.xorsign.abs.f16x2 %0, %0, %1;" : "+r"(hi) : "r"(0x7BFF7BFFu));
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
      constexpr bool kClamp = F == MIXATTN_KV_Q8_0;
      split_hilo<kClamp>(h0, sc, hi.x, lo.x);
      split_hilo<kClamp>(h1, sc, hi.y, lo.y);
      split_hilo<kClamp>(h2, sc, hi.z, lo.z);
      split_hilo<kClamp>(h3, sc, hi.w, lo.w);
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
//     S[jg%2] twice (row max, then P = 2^(s - m) as fp16 written over the scores
//     it has read, so P is double-buffered with S and never waits for a PV),
//     rescales O when the row max moved (then, and only then, after PV(jg-1));
//     after a tile's last scores it writes the next tile's Q, then stores this
//     tile's O;
//   MMA warp (warp 12, one thread): issues QK(jg) into S[jg%2] once K(jg) is
//     written (and, on a tile's first KV tile, its Q), then PV(jg-1), each key
//     half as soon as its V half is written.
// jg counts the KV tiles the CTA has walked, across its tiles: buffers and
// barrier phases follow it, so the next tile's loads, dequantisation and first
// QK overlap this tile's last softmax and its epilogue.  The MMA issue blocks
// its thread for about the MMA's duration, which is why one warp does nothing
// else.  TMEM: Q (A operand, fp16) | S0 / P0 | S1 / P1 | O (fp32): P(jg) lies over
// S[jg%2], PV(jg) reads it there, and QK(jg+2), the next writer of S[jg%2], is
// issued after PV(jg) by the same thread (the MMAs of one thread run in issue
// order).  Every wait is bounded; a timeout in any role makes all of them leave
// their loops.
template <int FK, int FV, int D>
__device__ __forceinline__ void chunk_cta(const AttnParams& p, int cta, int n_ctas, uint8_t* smem_raw,
                                          unsigned int* err) {
  using L = ChunkSmem<FK, FV, D>;
  constexpr uint32_t kTmemCols = 512;
  constexpr uint32_t kQCol = 0, kSCol0 = 128, kSCol1 = 256, kOCol = 384;  // P(j) lies over S[j % 2]
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
    // Every branch of this group that leads to a named barrier is taken by all of its
    // 128 threads: the abort flag, which other roles may set at any time, is read
    // through a group vote (bar_any) wherever a barrier follows, never thread by thread.
    auto group_abort = [&]() { return bar_any(kBarSoftmax, kGroup, *abort_flag != 0); };
    int k = next_round(0);
    if (k < n_rounds) write_q(chunk_tile_of(cta, k, n_ctas, p.n_chunk_tiles));
    int jg0 = 0;
    for (; k < n_rounds && !group_abort(); k = next_round(k + 1)) {
      const int idx = chunk_tile_of(cta, k, n_ctas, p.n_chunk_tiles);
      const TileDesc t = p.tiles[idx];
      const RowInfo ri = p.rows[t.row];
      const int g = t.kvh;
      const bool row_valid = tok < t.count;
      const int pos = ri.q_offset + t.begin + min(tok, t.count - 1);
      const int lo = window_first_key(pos, p.window);  // the row's first visible key
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
        // causal (and window) mask: only a warp whose tile crosses the diagonal (or the
        // window's start) pays for it
        const bool diag = __any_sync(0xFFFFFFFFu, kbase + kChunkN - 1 > pos || kbase < lo);
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
              if (kbase + 32 * c + e > pos || kbase + 32 * c + e < lo) a[e] = ninf;
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
        // pass 2: P = 2^(s*scale - m) as fp16, written over the tile's own scores
        // (S is double-buffered, so P is too: nothing here waits for PV(j-1)); row sums
        // in fp32.  The scale-and-shift and the sums run on fp32 pairs.
        const uint64_t sl2x2 = f2_pack(sl2, sl2), negm2 = f2_pack(neg_m, neg_m);
        uint64_t sum_a = f2_pack(0.f, 0.f), sum_b = sum_a;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          tmem_ld32(s_col + 32 * c, a);
          tmem_wait_ld();
          if (diag) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (kbase + 32 * c + e > pos || kbase + 32 * c + e < lo) a[e] = ninf;
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
          // P over the scores already read (words 16c.. of the row = columns 16c.. of
          // S[st]; chunks up to c are read by now): PV(jg) reads P there, and QK(jg+2),
          // the next writer of S[st], is issued after PV(jg) by the same thread
          tmem_st16(s_col + 16 * c, pk);
        }
        float sum0, sum1, sum2, sum3;
        f2_unpack(sum_a, sum0, sum1);
        f2_unpack(sum_b, sum2, sum3);
        sum0 += sum2;
        sum1 += sum3;
        l_run = l_run * alpha + (sum0 + sum1);
        m_run = m_new;
        // the running O, once PV(j-1) has finished with it; only a warp with a row whose
        // maximum moved waits for that
        if (j > 0) {
          if (__any_sync(0xFFFFFFFFu, alpha != 1.0f)) {
            ok = mbar_wait(&pv_done[(jg - 1) & 1], (uint32_t)(((jg - 1) >> 1) & 1), err) && ok;
            tc_fence_after();
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
      if (kn < n_rounds && !group_abort()) write_q(chunk_tile_of(cta, kn, n_ctas, p.n_chunk_tiles));
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
            pk[e >> 1] = pack_f16x2_out(__uint_as_float(v[e]) * inv_l, __uint_as_float(v[e + 1]) * inv_l);
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
                  make_uint4(pack_f16x2_out(acc[0] * inv_l, acc[1] * inv_l), pack_f16x2_out(acc[2] * inv_l, acc[3] * inv_l),
                             pack_f16x2_out(acc[4] * inv_l, acc[5] * inv_l), pack_f16x2_out(acc[6] * inv_l, acc[7] * inv_l));
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
          // S[st] holds P(jg-2), which PV(jg-2) reads; this thread issued PV(jg-2) before,
          // and the MMAs of one thread run in issue order
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
          const uint32_t p_col = tmem + (sp ? kSCol1 : kSCol0);  // P(jp) lies over S(jp)
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
    decode_tile<FK, FV, D, FS::kDecodeStages>(p, p.tiles[p.n_chunk_tiles + d], smem + half * FS::kHalfBytes, err, half);
  }
}

template <int FK, int FV, int D, int MINB, int NS>
__global__ void __launch_bounds__(kThreads, MINB) decode_attention_kernel(AttnParams p, unsigned int* err) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tile = blockIdx.x + p.n_chunk_tiles;
  decode_tile<FK, FV, D, NS>(p, p.tiles[tile], smem, err, 0);
}

// Chunk tiles whose mean KV-tile count is below this are walked by persistent
// CTAs.
constexpr int kPersistMaxKvTiles = 64;

// SMs of the current device, read once per device (a very large count when it
// cannot be read: then every chunk tile gets its own CTA).
inline int sm_count() {
  static std::atomic<int> cached[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1 << 30;
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
  // The shared-memory limit is an attribute of the function in the current
  // device's context: set it once per device (under a lock, host threads may
  // launch concurrently).
  {
    static std::mutex mu;
    static bool configured[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!configured[dev]) {
      e = cudaFuncSetAttribute(dec_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDec);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mixed_attention_kernel<FK, FV, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kFused);
      if (e != cudaSuccess) return e;
      configured[dev] = true;
    }
  }
  if (p.n_chunk_tiles == 0) {
    dec_kernel<<<p.n_decode_tiles, kThreads, kDec, s>>>(p, err);
  } else {
    mixed_attention_kernel<FK, FV, D><<<n_fused_ctas, kFusedThreads, kFused, s>>>(q, err);
  }
  return cudaGetLastError();
}

}  // namespace mixattn
