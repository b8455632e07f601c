// Short-query attention kernels (decode, speculative verify, and any request
// of at most 32 packed rows, in one tile of 8, 16 or 32 rows: query row x
// head of the GQA group), against the paged KV. Bandwidth-bound: every K/V byte is read
// exactly once, the online softmax is kept in fp32.
//
// Work item = (request tile, kv head, key chunk). One producer warp streams
// the item's live keys through a ring of stages in shared memory: per page
// of a stage it issues one cp.async.bulk.tensor box of K and one of V (4-D
// maps over [pages, slot, kv head, dim]), and for an item's first stage its
// q rows by plain bulk copy into a q buffer. mbarriers hand the stages to the
// consumer warps and back; each stage carries an 80-byte header with the
// item's geometry, so consumer warps read no global memory before they write
// the output. The producer runs ahead across work items, so the ring stays
// full through item boundaries.
//
// Two consumers:
//   DecodeMmaWarp  the GQA contraction on the warp-level tensor cores:
//                  S = Q K^T with the item's packed rows (padded to the 16
//                  rows of mma.m16n8k16), then O += P V. Stages are 64-column
//                  halves in 128B swizzle, so ldmatrix reads them without bank
//                  conflicts; needs boxes of at least 8 slots.
//   DecodeWarp     CUDA cores, for decode with smaller boxes (page sizes
//                  1, 2, 4): 16 lanes per key, a shuffle reduce-scatter of
//                  the G heads' dot products.
// At the end of an item the consumer warps' (max, sum, o) states are merged
// in shared memory, in rounds of 8 rows.
//
// Mask [P1 "Why window_size_right stays -1"], [P2 "Summary"]: key j of
// query row i is kept when (!causal || j <= i + Lk - Lq) &&
// (wl < 0 || j + Lq + wl >= Lk + i). Stages outside the item's live range
// are never loaded; the per-element test runs only on stages that straddle
// a bound.
//   [P1] "Route non-causal windowed prefill to AITER's masked kernel" (#339)
//   [P2] "Support speculative-decode verify on ROCm, and stop auto routing
//         short-query prefill to AITER" (#362)
#pragma once

#include <climits>
#include <type_traits>

#include "tma.cuh"

namespace fi {
namespace {

constexpr int kMaxRows = 32;  // packed rows per item (the row stride of the merge arrays)

// Header of one stage, written by the producer before it arms the stage's
// barrier. Keys [lo, hi) are live for some row of the item, keys
// [lo_full, hi_full) for every row; diff = Lk - Lq of the request.
// kStMaskOnes: the custom mask keeps every key of the stage for every row
enum : int32_t { kStFirst = 1, kStLast = 2, kStEnd = 4, kStNoKeys = 8, kStMaskOnes = 16 };
struct alignas(16) StageHdr {
  int32_t flags, k0, lo, hi;
  int32_t lo_full, hi_full, token0, kv_head;  // token0: global token of query row i0
  int32_t row0, n_rows, diff, chunk;          // first packed row, rows, Lk - Lq, chunk (-1: direct)
  int32_t num_chunks, partial_base, i0, lk;
  int32_t pad2, lq, pad0, pad1;               // Lq
};

// Write rows [r0, r0 + 8) of an item: sm_o holds those rows' o summed over
// the consumer warps (in MB partial sums of 8 rows each, added here in a
// fixed order), each warp's share already scaled to the row's common max;
// sm_m / sm_l hold each warp's row max (log2 domain) and sum.
template <int D, int G, bool BF16, int NWARP, int MB>
__device__ __forceinline__ void write_rows(const AttnParams& p, const StageHdr& h, int r0,
                                           float* tmp_o, float* tmp_lse, int tid, float* sm_o,
                                           float (*sm_m)[kMaxRows], float (*sm_l)[kMaxRows]) {
  using DT = Dt<BF16>;
  using T = typename DT::T;
  const int Hq = p.num_qo_heads;
  for (int idx = tid; idx < 8 * (D / 4); idx += NWARP * 32) {
    const int rl = idx / (D / 4);
    const int c = (idx % (D / 4)) * 4;
    const int r = r0 + rl;
    if (r >= h.n_rows) continue;
    float4 num = *reinterpret_cast<const float4*>(sm_o + rl * D + c);
    if (MB == 2) {  // (warps 0 + 1) + (warps 2 + 3)
      const float4 b = *reinterpret_cast<const float4*>(sm_o + (8 + rl) * D + c);
      num.x += b.x; num.y += b.y; num.z += b.z; num.w += b.w;
    }
    float M = neg_inf();
#pragma unroll
    for (int w = 0; w < NWARP; ++w) M = fmaxf(M, sm_m[w][r]);
    const float Mu = (M == neg_inf()) ? 0.f : M;
    float den = 0.f;
#pragma unroll
    for (int w = 0; w < NWARP; ++w) den += ex2(sm_m[w][r] - Mu) * sm_l[w][r];
    const float inv = den > 0.f ? 1.f / den : 0.f;
    const float lse = den > 0.f ? (M + __log2f(den)) * kLn2 : neg_inf();
    const int pr = h.row0 + r;
    const int ti = pr / G - h.i0;  // query row within the tile
    const int head = h.kv_head * G + pr % G;
    if (h.chunk < 0) {
      T* op = static_cast<T*>(p.out) + (int64_t(h.token0 + ti) * Hq + head) * D + c;
      uint2 pk;
      pk.x = DT::pack(num.x * inv, num.y * inv);
      pk.y = DT::pack(num.z * inv, num.w * inv);
      *reinterpret_cast<uint2*>(op) = pk;
      if (c == 0 && p.lse) p.lse[int64_t(h.token0 + ti) * Hq + head] = lse;
    } else {
      const int slot = h.partial_base + ti * h.num_chunks + h.chunk;
      *reinterpret_cast<float4*>(tmp_o + (int64_t(slot) * Hq + head) * D + c) =
          make_float4(num.x * inv, num.y * inv, num.z * inv, num.w * inv);
      if (c == 0) tmp_lse[int64_t(slot) * Hq + head] = lse;
    }
  }
}

// Common max of row r over the warps (0 when every warp's max is -inf).
template <int NWARP>
__device__ __forceinline__ float row_max(float (*sm_m)[kMaxRows], int r) {
  float M = neg_inf();
#pragma unroll
  for (int w = 0; w < NWARP; ++w) M = fmaxf(M, sm_m[w][r]);
  return (M == neg_inf()) ? 0.f : M;
}

// ------------------------------------------------------- shuffle consumer

// One consumer warp on CUDA cores, decode only (the item's rows are the G
// heads of one query token): q of the G heads pre-scaled into the exp2
// domain (fp32 pairs for the packed FMA), o of every head on this lane's 8
// dims, and the running max / sum of the head whose score this lane holds
// after the reduce-scatter.
template <int D, int G, bool BF16, int NWARP, int KT>
struct DecodeWarp {
  using DT = Dt<BF16>;
  using T = typename DT::T;
  static constexpr int LPK = D / 8;          // lanes per key
  static constexpr int KPS = 32 / LPK;       // keys per warp step
  static constexpr int KPW = KT / NWARP;     // keys per warp per stage
  static constexpr int STEPS = KPW / KPS;    // warp steps per stage
  static constexpr int ROUNDS = 1;           // G <= 8 rows: one merge round
  static_assert(KPW % KPS == 0, "a warp's keys of a stage are whole warp steps");
  static_assert(G <= 8, "one merge round");
  static constexpr bool kSwizzled = false;  // reads K/V stages as plain [KT][D] rows
  static constexpr int ROWS = 16;           // q buffer rows
  static constexpr bool kPair = false;

  int warp, lane, kg, dl;
  int myh;          // head whose score this lane holds after the reduce-scatter
  int src_of[G];    // lane (within this key's lane group) holding head h's score
  float2 q2[G][4];  // slot s holds head (myh ^ s)
  float2 o2[G][4];
  float m_me, l_me;
  float m_h[G];     // per-head max and sum of the warp (after publish)

  __device__ __forceinline__ void setup(int warp_, int lane_) {
    warp = warp_;
    lane = lane_;
    kg = lane / LPK;
    dl = lane % LPK;
    myh = 0;
    int cnt = G;
#pragma unroll
    for (int off = LPK / 2; off >= 1; off >>= 1) {
      if (cnt > 1) {
        cnt >>= 1;
        if (lane & off) myh += cnt;
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      int l_in = 0, c = G, rem = h;
#pragma unroll
      for (int off = LPK / 2; off >= 1; off >>= 1) {
        if (c > 1) {
          c >>= 1;
          if (rem >= c) {
            l_in |= off;
            rem -= c;
          }
        }
      }
      src_of[h] = (lane & ~(LPK - 1)) | l_in;
    }
  }

  // q of the G heads staged in shared memory as rows 0..G-1 of [16][D].
  // Slot s holds head (myh ^ s): at each level of the reduce-scatter a lane
  // then keeps its first half of the slots and sends the second, with no
  // per-lane selection.
  __device__ __forceinline__ void begin(const T* qs, int n_rows, float sm_scale_log2) {
    (void)n_rows;
#pragma unroll
    for (int sl = 0; sl < G; ++sl) {
      const uint4 r = *reinterpret_cast<const uint4*>(qs + (myh ^ sl) * D + dl * 8);
      const uint32_t wv[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        q2[sl][e] = make_float2(DT::lo(wv[e]) * sm_scale_log2, DT::hi(wv[e]) * sm_scale_log2);
    }
    m_me = neg_inf();
    l_me = 0.f;
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < 4; ++e) o2[h][e] = make_float2(0.f, 0.f);
  }

  __device__ __forceinline__ void stage(T* cK, T* cV, const StageHdr& h, int causal, int wl,
                                        const uint32_t* smask) {
    (void)causal;
    (void)wl;
    (void)smask;  // decode plans carry no custom mask
    stage_keys(cK, cV, h.k0, h.lo, h.hi);
  }

  // Consume one stage: keys k0 .. k0+KT-1 in rows 0..KT-1 of cK / cV, of
  // which [lo, hi) are live. Rows outside the live range may hold anything
  // (a neighbour's page slots): their scores are masked to -inf and their V
  // rows are read as zero, so no value there reaches o.
  __device__ __forceinline__ void stage_keys(T* cK, T* cV, int k0, int lo, int hi) {
    const bool full_tile = k0 >= lo && k0 + KT <= hi;
    float s[STEPS];  // this lane's (key, head) score per step
#pragma unroll
    for (int u = 0; u < STEPS; ++u) {
      const int key = warp * KPW + u * KPS + kg;
      const uint4 kr = *reinterpret_cast<const uint4*>(cK + key * D + dl * 8);
      const uint32_t wv[4] = {kr.x, kr.y, kr.z, kr.w};
      float2 k2[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) k2[e] = make_float2(DT::lo(wv[e]), DT::hi(wv[e]));
      float part[G];  // slot order: part[s] belongs to head myh ^ s
#pragma unroll
      for (int sl = 0; sl < G; ++sl) {
        float2 acc = __fmul2_rn(q2[sl][0], k2[0]);
#pragma unroll
        for (int e = 1; e < 4; ++e) acc = __ffma2_rn(q2[sl][e], k2[e], acc);
        part[sl] = acc.x + acc.y;
      }
      // reduce-scatter over the key's LPK lanes: at each of the first
      // log2(G) levels keep the first half of the slots and add the
      // partner's second half (which holds the same heads), then a plain
      // butterfly
      int cnt = G;
#pragma unroll
      for (int off = LPK / 2; off >= 1; off >>= 1) {
        if (cnt > 1) {
          const int half = cnt >> 1;
#pragma unroll
          for (int i = 0; i < half; ++i) part[i] += __shfl_xor_sync(0xffffffffu, part[half + i], off);
          cnt = half;
        } else {
          part[0] += __shfl_xor_sync(0xffffffffu, part[0], off);
        }
      }
      const int kk = k0 + key;
      s[u] = (full_tile || (kk >= lo && kk < hi)) ? part[0] : neg_inf();
    }
    // stage max of my head over the warp's keys
    float mx = s[0];
#pragma unroll
    for (int u = 1; u < STEPS; ++u) mx = fmaxf(mx, s[u]);
#pragma unroll
    for (int off = LPK; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    // lazy max: the reference moves only when the stage max exceeds it by
    // more than 2^8 (p stays <= 256), so o is rarely rescaled
    float mn = m_me;
    if (mx > m_me + 8.f || (m_me == neg_inf() && mx != neg_inf())) mn = mx;
    const float corr_me = (mn == m_me) ? 1.f : ex2(m_me - mn);
    const float mu = (mn == neg_inf()) ? 0.f : mn;
    m_me = mn;
    float pu[STEPS];
    float psum = 0.f;
#pragma unroll
    for (int u = 0; u < STEPS; ++u) {
      pu[u] = ex2(s[u] - mu);
      psum += pu[u];
    }
    l_me = l_me * corr_me + psum;
    // rescale o of every head by that head's correction
    if (__any_sync(0xffffffffu, corr_me != 1.f)) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float c = __shfl_sync(0xffffffffu, corr_me, src_of[h]);
        const float2 c2 = make_float2(c, c);
#pragma unroll
        for (int e = 0; e < 4; ++e) o2[h][e] = __fmul2_rn(o2[h][e], c2);
      }
    }
#pragma unroll
    for (int u = 0; u < STEPS; ++u) {
      const int key = warp * KPW + u * KPS + kg;
      uint4 vr = *reinterpret_cast<const uint4*>(cV + key * D + dl * 8);
      if (!full_tile) {
        const int kk = k0 + key;
        if (kk < lo || kk >= hi) vr = make_uint4(0u, 0u, 0u, 0u);
      }
      const uint32_t wv[4] = {vr.x, vr.y, vr.z, vr.w};
      float2 v2[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) v2[e] = make_float2(DT::lo(wv[e]), DT::hi(wv[e]));
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float ph = __shfl_sync(0xffffffffu, pu[u], src_of[h]);
        const float2 p2 = make_float2(ph, ph);
#pragma unroll
        for (int e = 0; e < 4; ++e) o2[h][e] = __ffma2_rn(p2, v2[e], o2[h][e]);
      }
    }
  }

  // Reduce the warp's key groups and publish each head's max / sum.
  __device__ __forceinline__ void publish_ml(float (*sm_m)[kMaxRows], float (*sm_l)[kMaxRows]) {
    float l_h[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m_h[h] = __shfl_sync(0xffffffffu, m_me, src_of[h]);
      l_h[h] = __shfl_sync(0xffffffffu, l_me, src_of[h]);
    }
#pragma unroll
    for (int off = LPK; off < 32; off <<= 1) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        l_h[h] += __shfl_xor_sync(0xffffffffu, l_h[h], off);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          o2[h][e].x += __shfl_xor_sync(0xffffffffu, o2[h][e].x, off);
          o2[h][e].y += __shfl_xor_sync(0xffffffffu, o2[h][e].y, off);
        }
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        sm_m[warp][h] = m_h[h];
        sm_l[warp][h] = l_h[h];
      }
    }
  }

  // Store (first) or add this warp's o, scaled to each head's common max,
  // into sm_o (rows = heads); the warps take turns in a fixed order. The
  // lanes of key group 0 hold the warp's sums.
  __device__ __forceinline__ void add_o(int round, int n_rows, bool first, float* sm_o,
                                        float (*sm_m)[kMaxRows]) {
    (void)round;
    (void)n_rows;
    if (kg != 0) return;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float sc = ex2(m_h[h] - row_max<NWARP>(sm_m, h));
      float4* dst = reinterpret_cast<float4*>(sm_o + h * D + dl * 8);
      float4 v0 = make_float4(o2[h][0].x * sc, o2[h][0].y * sc, o2[h][1].x * sc, o2[h][1].y * sc);
      float4 v1 = make_float4(o2[h][2].x * sc, o2[h][2].y * sc, o2[h][3].x * sc, o2[h][3].y * sc);
      if (!first) {
        const float4 a0 = dst[0], a1 = dst[1];
        v0.x += a0.x; v0.y += a0.y; v0.z += a0.z; v0.w += a0.w;
        v1.x += a1.x; v1.y += a1.y; v1.z += a1.z; v1.w += a1.w;
      }
      dst[0] = v0;
      dst[1] = v1;
    }
  }
};

// ------------------------------------------------------- tensor-core consumer

// One consumer warp on the warp-level tensor cores. The GQA group is a dense
// contraction: S = Q K^T with the item's packed rows (query row x head,
// padded to 16) against the warp's KPW keys of a stage, then O += P V. RH
// fragment row halves are live: 1 when the items have at most 8 rows (decode
// with G <= 8), else 2. Lane l holds rows l / 4 and l / 4 + 8; its running
// max / sum live in the lane's quad. About 80 instructions per warp-stage
// for 16 keys, against about 900 for the shuffle consumer.
template <int D, int G, bool BF16, int NWARP, int KT, int RH>
struct DecodeMmaWarp {
  using DT = Dt<BF16>;
  using T = typename DT::T;
  static constexpr int KPW = KT / NWARP;  // keys per warp per stage
  static constexpr int NT = KPW / 8;      // n8 score tiles per warp
  static constexpr int KD = D / 16;       // k16 steps over the head dim
  static constexpr int HALF = KT * 128;   // bytes of one 64-column half of a stage
  static constexpr int ROUNDS = RH;
  static_assert(KPW % 16 == 0, "a warp's keys are whole k16 steps of P V");
  static_assert(RH == 1 || RH == 2, "one or two live row halves");
  static constexpr bool kSwizzled = true;
  static constexpr int ROWS = 16;
  static constexpr bool kPair = false;

  int warp, lane, qr, qc;
  uint32_t qa[KD][4];   // A fragments (rows qr, qr + 8; the padding rows are zero)
  float o[D / 8][4];    // rows qr (o[.][0..1]) and qr + 8 (o[.][2..3])
  float m[RH], l[RH];   // running max / sum of rows qr (+ 8)
  float scale;

  // byte offset of 16-byte chunk c of row r in a swizzled stage
  __device__ __forceinline__ static uint32_t swz(int r, int c) {
    return uint32_t((c >> 3) * HALF + r * 128 + (((c & 7) ^ (r & 7)) << 4));
  }

  __device__ __forceinline__ void setup(int warp_, int lane_) {
    warp = warp_;
    lane = lane_;
    qr = lane >> 2;
    qc = lane & 3;
  }

  // q of the item's rows staged in shared memory as [16][D]
  __device__ __forceinline__ void begin(const T* qs, int n_rows, float sm_scale_log2) {
#pragma unroll
    for (int kd = 0; kd < KD; ++kd) {
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int r = qr + 8 * hr;
        uint32_t lo = 0u, hi = 0u;
        if (hr < RH && r < n_rows) {
          lo = *reinterpret_cast<const uint32_t*>(qs + r * D + kd * 16 + qc * 2);
          hi = *reinterpret_cast<const uint32_t*>(qs + r * D + kd * 16 + 8 + qc * 2);
        }
        qa[kd][hr] = lo;
        qa[kd][2 + hr] = hi;
      }
    }
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
#pragma unroll
    for (int hr = 0; hr < RH; ++hr) {
      m[hr] = neg_inf();
      l[hr] = 0.f;
    }
    scale = sm_scale_log2;
  }

  // Consume one stage (keys h.k0 .. + KT). Where the stage is not inside
  // every row's range (or a custom mask drops a key of it) the per-element
  // mask runs; where it is not inside the item's live range the warp first
  // zeroes its V rows outside it (they may hold anything, a neighbour's
  // slots, and 0 * NaN would reach o). smask: the stage's custom-mask bits,
  // KT / 32 words per query row of the item (null: no custom mask).
  __device__ __forceinline__ void stage(T* cK, T* cV, const StageHdr& h, int causal, int wl,
                                        const uint32_t* smask) {
    const uint32_t sk = smem_u32(cK), sv = smem_u32(cV);
    const int kb = warp * KPW;  // this warp's first key in the stage
    const int k0 = h.k0;
    if (!(k0 >= h.lo && k0 + KT <= h.hi)) {
      // lane l zeroes chunks l, l+32, ... of the warp's dead rows
      for (int idx = lane; idx < KPW * (D / 8); idx += 32) {
        const int r = kb + idx / (D / 8), c = idx % (D / 8);
        const int kk = k0 + r;
        if (kk < h.lo || kk >= h.hi)
          *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(cV) + swz(r, c)) =
              make_uint4(0u, 0u, 0u, 0u);
      }
      // these generic-proxy writes are ordered before the slot's next TMA fill
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
    }
    const bool full_tile = k0 >= h.lo_full && k0 + KT <= h.hi_full &&
                           (!smask || (h.flags & kStMaskOnes));
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int kd = 0; kd < KD; ++kd) {
#pragma unroll
      for (int nt = 0; nt < NT; nt += 2) {
        const int r = kb + nt * 8 + (lane & 7) + (lane >> 4) * 8;
        const int c = kd * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sk + swz(r, c), b0, b1, b2, b3);
        mma16816<BF16>(s[nt], qa[kd], b0, b1);
        mma16816<BF16>(s[nt + 1], qa[kd], b2, b3);
      }
    }
    // s[nt][2*hr + e]: row qr + 8*hr, key kb + nt*8 + qc*2 + e
    float corr[RH];
#pragma unroll
    for (int hr = 0; hr < RH; ++hr) {
      const int r = qr + 8 * hr;
      const int i = (h.row0 + r) / G;  // query row of the request
      float mx = neg_inf();
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float x = s[nt][2 * hr + e] * scale;
          if (!full_tile) {
            const int kk = k0 + kb + nt * 8 + qc * 2 + e;
            bool ok = r < h.n_rows && kk >= h.lo && kk < h.hi;
            if (causal && kk > i + h.diff) ok = false;
            if (wl >= 0 && kk + wl < h.diff + i) ok = false;
            // custom mask (ANDed), as staged by the producer
            if (ok && smask) {
              const int kl = kb + nt * 8 + qc * 2 + e;
              if (!((smask[(i - h.i0) * (KT / 32) + (kl >> 5)] >> (kl & 31)) & 1u)) ok = false;
            }
            if (!ok) x = neg_inf();
          }
          s[nt][2 * hr + e] = x;
          mx = fmaxf(mx, x);
        }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      // lazy max: moves only when the stage max exceeds it by more than 2^8
      float mn = m[hr];
      if (mx > m[hr] + 8.f || (m[hr] == neg_inf() && mx != neg_inf())) mn = mx;
      corr[hr] = (mn == m[hr]) ? 1.f : ex2(m[hr] - mn);
      const float mu = (mn == neg_inf()) ? 0.f : mn;
      m[hr] = mn;
      float psum = 0.f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          s[nt][2 * hr + e] = ex2(s[nt][2 * hr + e] - mu);
          psum += s[nt][2 * hr + e];
        }
      l[hr] = l[hr] * corr[hr] + psum;
    }
    bool any = corr[0] != 1.f;
    if (RH == 2) any = any || corr[RH - 1] != 1.f;
    if (__any_sync(0xffffffffu, any)) {
#pragma unroll
      for (int i = 0; i < D / 8; ++i)
#pragma unroll
        for (int hr = 0; hr < RH; ++hr) {
          o[i][2 * hr] *= corr[hr];
          o[i][2 * hr + 1] *= corr[hr];
        }
    }
#pragma unroll
    for (int kk = 0; kk < KPW / 16; ++kk) {
      uint32_t pa[4];
      pa[0] = DT::pack(s[2 * kk][0], s[2 * kk][1]);
      pa[2] = DT::pack(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[1] = RH == 2 ? DT::pack(s[2 * kk][2], s[2 * kk][3]) : 0u;
      pa[3] = RH == 2 ? DT::pack(s[2 * kk + 1][2], s[2 * kk + 1][3]) : 0u;
#pragma unroll
      for (int dn = 0; dn < D / 16; ++dn) {
        const int r = kb + kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int c = dn * 2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(sv + swz(r, c), b0, b1, b2, b3);
        mma16816<BF16>(o[2 * dn], pa, b0, b1);
        mma16816<BF16>(o[2 * dn + 1], pa, b2, b3);
      }
    }
  }

  __device__ __forceinline__ void publish_ml(float (*sm_m)[kMaxRows], float (*sm_l)[kMaxRows]) {
#pragma unroll
    for (int hr = 0; hr < RH; ++hr) {
      float lr = l[hr];
      lr += __shfl_xor_sync(0xffffffffu, lr, 1);
      lr += __shfl_xor_sync(0xffffffffu, lr, 2);
      if (qc == 0) {
        sm_m[warp][qr + 8 * hr] = m[hr];
        sm_l[warp][qr + 8 * hr] = lr;
      }
    }
  }

  // Store (first) or add this warp's o of rows [8*round, 8*round + 8),
  // scaled to each row's common max, into sm_o (8 rows). The warps take
  // turns in a fixed order, so the sum is the same on every run.
  __device__ __forceinline__ void add_o(int round, int n_rows, bool first, float* sm_o,
                                        float (*sm_m)[kMaxRows]) {
#pragma unroll
    for (int hr = 0; hr < RH; ++hr) {
      if (hr != round) continue;
      const int r = qr + 8 * hr;
      if (r >= n_rows) continue;
      const float sc = ex2(m[hr] - row_max<NWARP>(sm_m, r));
      float2* dst = reinterpret_cast<float2*>(sm_o + qr * D + qc * 2);
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        float2 v = make_float2(o[i][2 * hr] * sc, o[i][2 * hr + 1] * sc);
        if (!first) {
          const float2 a = dst[i * 4];
          v.x += a.x;
          v.y += a.y;
        }
        dst[i * 4] = v;
      }
    }
  }
};

// Two warp pairs on the warp-level tensor cores for items of 17 to 32 packed
// rows, so the item's keys are read once (two 16-row items would each read
// them). Warp w runs M tile w / 2 (rows 16 (w / 2) ..) against key half w % 2
// of every stage (KT / 2 keys); the two warps of an M tile hold that tile's
// rows over complementary keys, and their states meet in the item-end merge.
template <int D, int G, bool BF16, int NWARP, int KT>
struct DecodeMmaPairWarp {
  using DT = Dt<BF16>;
  using T = typename DT::T;
  static constexpr int KPW = KT / 2;      // keys per warp per stage
  static constexpr int NT = KPW / 8;      // n8 score tiles per warp
  static constexpr int KD = D / 16;       // k16 steps over the head dim
  static constexpr int HALF = KT * 128;   // bytes of one 64-column half of a stage
  static constexpr int ROUNDS = 4;        // merge rounds of 8 rows
  static constexpr int ROWS = 32;
  static constexpr bool kSwizzled = true;
  static constexpr bool kPair = true;
  static_assert(NWARP == 4, "two M tiles x two key halves");
  static_assert(KPW % 16 == 0, "a warp's keys are whole k16 steps of P V");

  int warp, lane, qr, qc, mt, kh;
  uint32_t qa[KD][4];   // A fragments of rows 16 mt + qr (+ 8)
  float o[D / 8][4];
  float m[2], l[2];     // running max / sum of rows 16 mt + qr (+ 8)
  float scale;

  __device__ __forceinline__ static uint32_t swz(int r, int c) {
    return uint32_t((c >> 3) * HALF + r * 128 + (((c & 7) ^ (r & 7)) << 4));
  }

  __device__ __forceinline__ void setup(int warp_, int lane_) {
    warp = warp_;
    lane = lane_;
    qr = lane >> 2;
    qc = lane & 3;
    mt = warp >> 1;
    kh = warp & 1;
  }

  // q of the item's rows staged in shared memory as [32][D]
  __device__ __forceinline__ void begin(const T* qs, int n_rows, float sm_scale_log2) {
#pragma unroll
    for (int kd = 0; kd < KD; ++kd) {
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int r = 16 * mt + qr + 8 * hr;
        uint32_t lo = 0u, hi = 0u;
        if (r < n_rows) {
          lo = *reinterpret_cast<const uint32_t*>(qs + r * D + kd * 16 + qc * 2);
          hi = *reinterpret_cast<const uint32_t*>(qs + r * D + kd * 16 + 8 + qc * 2);
        }
        qa[kd][hr] = lo;
        qa[kd][2 + hr] = hi;
      }
    }
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    m[0] = m[1] = neg_inf();
    l[0] = l[1] = 0.f;
    scale = sm_scale_log2;
  }

  // Consume this warp's key half of one stage (see DecodeMmaWarp::stage:
  // the same masking, zeroing of dead V rows, lazy max and P V product).
  __device__ __forceinline__ void stage(T* cK, T* cV, const StageHdr& h, int causal, int wl,
                                        const uint32_t* smask) {
    const uint32_t sk = smem_u32(cK), sv = smem_u32(cV);
    const int kb = kh * KPW;
    const int k0 = h.k0;
    if (!(k0 >= h.lo && k0 + KT <= h.hi)) {
      for (int idx = lane; idx < KPW * (D / 8); idx += 32) {
        const int r = kb + idx / (D / 8), c = idx % (D / 8);
        const int kk = k0 + r;
        if (kk < h.lo || kk >= h.hi)
          *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(cV) + swz(r, c)) =
              make_uint4(0u, 0u, 0u, 0u);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
    }
    const bool full_tile = k0 >= h.lo_full && k0 + KT <= h.hi_full &&
                           (!smask || (h.flags & kStMaskOnes));
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int kd = 0; kd < KD; ++kd) {
#pragma unroll
      for (int nt = 0; nt < NT; nt += 2) {
        const int r = kb + nt * 8 + (lane & 7) + (lane >> 4) * 8;
        const int c = kd * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sk + swz(r, c), b0, b1, b2, b3);
        mma16816<BF16>(s[nt], qa[kd], b0, b1);
        mma16816<BF16>(s[nt + 1], qa[kd], b2, b3);
      }
    }
    float corr[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int r = 16 * mt + qr + 8 * hr;
      const int i = (h.row0 + r) / G;
      float mx = neg_inf();
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float x = s[nt][2 * hr + e] * scale;
          if (!full_tile) {
            const int kk = k0 + kb + nt * 8 + qc * 2 + e;
            bool ok = r < h.n_rows && kk >= h.lo && kk < h.hi;
            if (causal && kk > i + h.diff) ok = false;
            if (wl >= 0 && kk + wl < h.diff + i) ok = false;
            if (ok && smask) {
              const int kl = kb + nt * 8 + qc * 2 + e;
              if (!((smask[(i - h.i0) * (KT / 32) + (kl >> 5)] >> (kl & 31)) & 1u)) ok = false;
            }
            if (!ok) x = neg_inf();
          }
          s[nt][2 * hr + e] = x;
          mx = fmaxf(mx, x);
        }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      float mn = m[hr];
      if (mx > m[hr] + 8.f || (m[hr] == neg_inf() && mx != neg_inf())) mn = mx;
      corr[hr] = (mn == m[hr]) ? 1.f : ex2(m[hr] - mn);
      const float mu = (mn == neg_inf()) ? 0.f : mn;
      m[hr] = mn;
      float psum = 0.f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          s[nt][2 * hr + e] = ex2(s[nt][2 * hr + e] - mu);
          psum += s[nt][2 * hr + e];
        }
      l[hr] = l[hr] * corr[hr] + psum;
    }
    if (__any_sync(0xffffffffu, corr[0] != 1.f || corr[1] != 1.f)) {
#pragma unroll
      for (int i = 0; i < D / 8; ++i)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          o[i][2 * hr] *= corr[hr];
          o[i][2 * hr + 1] *= corr[hr];
        }
    }
#pragma unroll
    for (int kk = 0; kk < KPW / 16; ++kk) {
      uint32_t pa[4];
      pa[0] = DT::pack(s[2 * kk][0], s[2 * kk][1]);
      pa[2] = DT::pack(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[1] = DT::pack(s[2 * kk][2], s[2 * kk][3]);
      pa[3] = DT::pack(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int dn = 0; dn < D / 16; ++dn) {
        const int r = kb + kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int c = dn * 2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(sv + swz(r, c), b0, b1, b2, b3);
        mma16816<BF16>(o[2 * dn], pa, b0, b1);
        mma16816<BF16>(o[2 * dn + 1], pa, b2, b3);
      }
    }
  }

  // Row max / sum of this warp's 16 rows; the other M tile's rows get
  // (-inf, 0), so every per-row reduction over the four warps sees only the
  // two warps that hold the row.
  __device__ __forceinline__ void publish_ml(float (*sm_m)[kMaxRows], float (*sm_l)[kMaxRows]) {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      float lr = l[hr];
      lr += __shfl_xor_sync(0xffffffffu, lr, 1);
      lr += __shfl_xor_sync(0xffffffffu, lr, 2);
      if (qc == 0) {
        sm_m[warp][16 * mt + qr + 8 * hr] = m[hr];
        sm_l[warp][16 * mt + qr + 8 * hr] = lr;
        sm_m[warp][16 * (1 - mt) + qr + 8 * hr] = neg_inf();
        sm_l[warp][16 * (1 - mt) + qr + 8 * hr] = 0.f;
      }
    }
  }

  // Round r merges rows [8 r, 8 r + 8): M tile r / 2, row half r % 2. Its
  // key-half-0 warp stores (first), then its key-half-1 warp adds, each
  // share scaled to the row's common max; the other M tile's warps idle.
  __device__ __forceinline__ void add_o(int round, int n_rows, bool first, float* sm_o,
                                        float (*sm_m)[kMaxRows]) {
    if (mt != (round >> 1)) return;
    const int hr = round & 1;
    const int r = 16 * mt + qr + 8 * hr;
    if (r >= n_rows) return;
    const float sc = ex2(m[hr] - row_max<NWARP>(sm_m, r));
    float2* dst = reinterpret_cast<float2*>(sm_o + qr * D + qc * 2);
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      float2 v = make_float2(o[i][2 * hr] * sc, o[i][2 * hr + 1] * sc);
      if (!first) {
        const float2 a = dst[i * 4];
        v.x += a.x;
        v.y += a.y;
      }
      dst[i * 4] = v;
    }
  }
};

// ------------------------------------------------------------ TMA kernel

// Ring geometry: NCW consumer warps of KPW keys each per stage (D = 128;
// twice as many keys at D = 64, so a stage is always the same bytes), NS
// stages, MINB CTAs per SM. Measured on the batch-64 decode (page 16): the
// tensor-core consumer is fastest with 3 stages at 2 CTAs per SM (6300
// GB/s; 2 stages at 3 CTAs per SM: 5930, and it spills), the CUDA-core
// consumer with 2 stages at 3 CTAs per SM (5760; 3 stages at 2 CTAs: 5045).
template <int D, bool MMA, int ROWS_ = 16>
struct TmaCfg {
  static constexpr int ROWS = ROWS_;  // q rows of an item
  static constexpr int NCW = 4;
  static constexpr int KPW = 16;
  static constexpr int KT = NCW * KPW * (128 / D);  // keys per stage (a power of two)
  static constexpr int NS = MMA ? 3 : 2;
  static constexpr int MINB = MMA ? 2 : 3;
  static constexpr int THREADS = (NCW + 1) * 32;
  static constexpr int STAGE = KT * D;             // elements per stage, K or V
  static constexpr int RING_BYTES = NS * STAGE * 2 * 2;
  static constexpr int NBAR = 2 * NS + 2;          // full, empty per slot; q free; merge
  // dynamic shared memory: K/V ring | merge rows | per-warp row max, sum |
  // q rows | stage headers | barriers, abort flag | custom-mask bits
  // merge buffers of 8 rows: two (a pairwise merge, 3 barriers per round)
  // where shared memory allows, else one (warps take turns; the 32-row
  // consumer's two warps of a row, 3 barriers)
  static constexpr int MB = (MMA && ROWS == 16) ? 2 : 1;
  static_assert(!MMA || NCW == 4, "the pairwise merge pairs four warps");
  static constexpr int O_OFF = RING_BYTES;
  static constexpr int ML_OFF = O_OFF + MB * 8 * D * 4;
  static constexpr int Q_OFF = ML_OFF + 2 * NCW * kMaxRows * 4;
  static constexpr int HDR_OFF = Q_OFF + ROWS * D * 2;
  static constexpr int BAR_OFF = HDR_OFF + NS * int(sizeof(StageHdr));
  // custom-mask bits of each stage (tensor-core consumer): KT / 32 words per
  // query row of the item, written by the producer with the stage header
  static constexpr int MASKW = KT / 32;
  static constexpr int MASK_OFF = BAR_OFF + NBAR * 8 + 16;
  static constexpr int SMEM = MASK_OFF + (MMA ? NS * ROWS * MASKW * 4 : 0);
  static_assert((KT & (KT - 1)) == 0, "keys per stage is a power of two");
  static_assert(MINB * (SMEM + 1024) <= 233472, "MINB CTAs fit one SM's shared memory");
};

// The producer warp of decode_tma_kernel (see there). Kept out of line, so
// its registers are allocated apart from the consumer warps' path.
template <int D, int G, bool BF16, bool MMA, class W>
__device__ __noinline__ void decode_producer(const AttnParams& p, const CUtensorMap* tkp,
                                             const CUtensorMap* tvp, int box_rows, uint8_t* dsmem,
                                             int lane, int causal, int window_left,
                                             volatile WaitCtl* ctl) {
  using C = TmaCfg<D, MMA, W::ROWS>;
  constexpr int NCW = C::NCW, KT = C::KT, NS = C::NS, STAGE = C::STAGE;
  using T = typename W::T;
  const WsHeader* hdr = static_cast<const WsHeader*>(p.ws);
  T* sK = reinterpret_cast<T*>(dsmem);
  T* sV = sK + NS * STAGE;
  T* sQ = reinterpret_cast<T*>(dsmem + C::Q_OFF);
  StageHdr* sH = reinterpret_cast<StageHdr*>(dsmem + C::HDR_OFF);
  const uint32_t bar0 = smem_u32(dsmem + C::BAR_OFF);
  auto FULL = [&](int s) { return bar0 + 8u * uint32_t(s); };
  auto EMPTY = [&](int s) { return bar0 + 8u * uint32_t(NS + s); };
  const uint32_t QFREE = bar0 + 8u * uint32_t(2 * NS);
  (void)NCW;
  // ------------------------------------------------------------ producer
  // Stage c of this CTA's sequence goes to slot c % NS; its (c / NS)-th
  // fill waits for the consumers' release of the previous one. The q
  // buffer of item n waits for the consumers' release of item n - 1's q.
  // Everything a stage needs from global memory (the item's metadata, the
  // page indices) is loaded before those waits, so a full ring hides it.
  // The start of the chain before the first K/V bytes move: the tensor maps'
  // descriptors are prefetched, and the CTA's first item (at a fixed offset,
  // and the plan always holds at least a grid's worth of items) loads in the
  // same round trip as the header; an item carries its request's metadata,
  // so the page-table read comes next.
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tkp)) : "memory");
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tvp)) : "memory");
  const WorkItem* items = ws_ptr<const WorkItem>(p.ws, kItemsOffset);
  WorkItem next_it = items[blockIdx.x];
  const int n_items = hdr->n_items;
  const int tile_rows = hdr->tile_rows;
  const int n_boxes = KT / box_rows;  // a stage is n_boxes boxes of box_rows slots of one page
  const uint32_t box_bytes = uint32_t(box_rows) * D * 2;
  constexpr int BPL = (KT + 31) / 32;  // boxes per lane, at most
  int c = 0, n_item = 0;
  bool ok = true;
  uint32_t last_par[NS];
  bool armed[NS];
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    armed[s] = false;
    last_par[s] = 0;
  }
  constexpr int MW = C::MASKW;
  uint32_t* sMask = reinterpret_cast<uint32_t*>(dsmem + C::MASK_OFF);
  // claim slot st for stage c (and, for an item's first stage, the q
  // buffer): wait for their release, then write the stage's custom-mask
  // words (lanes below n_mask: lane = query row of the item), the header,
  // and arm the slot's barrier for `bytes` (lane 0); false once the CTA
  // aborts. Every armed phase is recorded (the end-of-work stage too), so the
  // drain below waits on each slot's latest phase.
  auto claim = [&](int st, uint32_t par, const StageHdr& h, uint32_t bytes, bool first,
                   int n_mask, const uint32_t* mw) {
    bool okl = true;
    if (lane == 0) {
      if (c >= NS) okl = mbar_wait(EMPTY(st), par ^ 1u, ctl);
      if (okl && first && n_item > 0)
        okl = mbar_wait(QFREE, uint32_t(n_item - 1) & 1u, ctl);
    }
    okl = __shfl_sync(0xffffffffu, okl, 0) != 0;
    if (okl && n_mask > 0) {
      if (lane < n_mask) {
#pragma unroll
        for (int w = 0; w < MW; ++w) sMask[(st * C::ROWS + lane) * MW + w] = mw[w];
      }
      __syncwarp();  // ordered before lane 0's arrive (release) below
    }
    if (okl && lane == 0) {
      sH[st] = h;
      mbar_expect_tx(FULL(st), bytes);
    }
    if (okl) {
#pragma unroll
      for (int s = 0; s < NS; ++s)
        if (s == st) {
          armed[s] = true;
          last_par[s] = par;
        }
    }
    return okl;
  };
  for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
    const WorkItem it = next_it;
    // the CTA's next item loads while this one streams
    if (w + int(gridDim.x) < n_items) next_it = items[w + gridDim.x];
    if (it.b < 0) continue;  // schedule padding
    // item geometry: packed rows [row0, row0 + n_rows) = query rows
    // i0..i1 of request b, and the key ranges their masks leave
    const int tok_b = it.tok0;
    const int lq = it.lq;
    const int lk = it.lk;
    const int n_rows = min(tile_rows, lq * G - it.row0);
    const int i0 = it.row0 / G, i1 = (it.row0 + n_rows) / G - 1;
    const int diff = lk - lq;
    const int hi_t = causal ? min(lk, i1 + diff + 1) : lk;
    const int lo_t = window_left >= 0 ? max(0, diff + i0 - window_left) : 0;
    const int lo = max(it.kv_begin, lo_t), hi = min(it.kv_end, hi_t);
    StageHdr h;
    h.lo = lo;
    h.hi = hi;
    h.lo_full = max(lo, window_left >= 0 ? diff + i1 - window_left : 0);
    h.hi_full = min(hi, causal ? i0 + diff + 1 : hi);
    h.token0 = tok_b + i0;
    h.kv_head = it.kv_head;
    h.row0 = it.row0;
    h.n_rows = n_rows;
    h.diff = diff;
    h.chunk = it.chunk;
    h.num_chunks = it.num_chunks;
    h.partial_base = it.partial_base;
    h.i0 = i0;
    h.lk = lk;
    h.lq = lq;
    h.pad2 = h.pad0 = h.pad1 = 0;
    // custom mask: request b's bits (row-major, bit i * Lk + j) start on
    // byte mask_base; the producer stages each stage's KT bits per query row
    const bool masked = MMA && p.custom_mask != nullptr;
    const uint8_t* mseg =
        masked ? p.custom_mask + it.mask_base : nullptr;
    const int n_mask = masked ? i1 - i0 + 1 : 0;
    const int start = lo & ~(box_rows - 1);
    const int n_tiles = hi > lo ? (hi - start + KT - 1) / KT : 0;
    const int kv_start = it.kv_start;  // ragged: first row; paged: first page-table entry
    const int32_t* pages = p.ragged ? nullptr : p.kv_indices + kv_start;
    const int n_st = max(n_tiles, 1);  // an item without keys still writes its output
    for (int t = 0; t < n_st; ++t, ++c) {
      const int st = c % NS;
      const uint32_t par = uint32_t(c / NS) & 1u;
      const int k0 = start + t * KT;
      const int n_live = n_tiles ? min(n_boxes, (hi - k0 + box_rows - 1) / box_rows) : 0;
      int page[BPL], slot[BPL];
#pragma unroll
      for (int j = 0; j < BPL; ++j) {
        const int i = lane + 32 * j;
        page[j] = 0;
        slot[j] = 0;
        if (i < n_live) {
          const int kb = k0 + i * box_rows;
          if (p.ragged) {  // one logical page: the slot is the row
            slot[j] = kv_start + kb;
          } else {
            int pi;
            if (p.page_shift >= 0) {
              pi = kb >> p.page_shift;
              slot[j] = kb & ((1 << p.page_shift) - 1);
            } else {
              pi = kb / p.page_size;
              slot[j] = kb - pi * p.page_size;
            }
            page[j] = __ldg(pages + pi);
          }
        }
      }
      h.flags = (t == 0 ? kStFirst : 0) | (t == n_st - 1 ? kStLast : 0) |
                (n_tiles ? 0 : kStNoKeys);
      // this lane's query row's bits of keys k0 .. k0 + KT (bits past the
      // segment read as 0; the consumers mask keys outside [lo, hi) anyway)
      uint32_t mw[MW];
#pragma unroll
      for (int w = 0; w < MW; ++w) mw[w] = ~0u;
      if (masked) {
        if (lane < n_mask) {
          const int64_t n0 = int64_t(i0 + lane) * lk + k0;
#pragma unroll
          for (int w = 0; w < MW; ++w)
            mw[w] = custom_mask_word(mseg, int64_t(lq) * lk, n0 + 32 * w);
        }
        bool ones = true;
#pragma unroll
        for (int w = 0; w < MW; ++w) ones = ones && mw[w] == ~0u;
        if (__all_sync(0xffffffffu, ones)) h.flags |= kStMaskOnes;
      }
      h.k0 = k0;
      const uint32_t qbytes = t == 0 ? uint32_t(n_rows * D * 2) : 0u;
      if (!claim(st, par, h, uint32_t(n_live) * box_bytes * 2u + qbytes, t == 0, n_mask, mw)) {
        ok = false;
        break;
      }
      if (t == 0) {
        // q rows of the item, one bulk copy per packed row
        for (int r = lane; r < n_rows; r += 32) {
          const int pr = it.row0 + r;
          const T* src = static_cast<const T*>(p.q) + int64_t(tok_b + pr / G) * p.q_stride_tok +
                         int64_t(it.kv_head * G + pr % G) * p.q_stride_head;
          bulk_load(smem_u32(sQ + r * D), src, uint32_t(D * 2), FULL(st));
        }
        ++n_item;
      }
      const uint32_t dk = smem_u32(sK + st * STAGE), dv = smem_u32(sV + st * STAGE);
#pragma unroll
      for (int j = 0; j < BPL; ++j) {
        const int i = lane + 32 * j;
        if (i < n_live) {
          if constexpr (W::kSwizzled) {
            // one box per 64-column half; half x of the stage at x * KT * 128
            const uint32_t off = uint32_t(i * box_rows) * 128u;
#pragma unroll
            for (int x = 0; x < D / 64; ++x) {
              tma_load_4d(dk + x * KT * 128 + off, tkp, FULL(st), x * 64, it.kv_head, slot[j], page[j]);
              tma_load_4d(dv + x * KT * 128 + off, tvp, FULL(st), x * 64, it.kv_head, slot[j], page[j]);
            }
          } else {
            const uint32_t off = uint32_t(i) * box_bytes;
            tma_load_4d(dk + off, tkp, FULL(st), 0, it.kv_head, slot[j], page[j]);
            tma_load_4d(dv + off, tvp, FULL(st), 0, it.kv_head, slot[j], page[j]);
          }
        }
      }
    }
  }
  if (ok) {
    // end of work: a header-only stage tells the consumers to stop
    StageHdr h = {};
    h.flags = kStEnd;
    const int st = c % NS;
    if (!claim(st, uint32_t(c / NS) & 1u, h, 0u, false, 0, nullptr)) ok = false;
  }
  // Drain: the last fill of every slot has landed before the CTA exits
  // (the consumers waited for all of them unless a wait expired; this wait
  // ignores the abort flag but keeps its time bound, and an expiry is
  // reported too).
  if (lane == 0) {
    volatile WaitCtl drain = {0, 0, kWaitLimitNs};
#pragma unroll
    for (int s = 0; s < NS; ++s)
      if (armed[s] && !mbar_wait(FULL(s), last_par[s], &drain)) ctl->abort = 1;
  }
}

// MMA: the tensor-core consumer (128B-swizzled stages, 64-column boxes of
// at least 8 slots, i.e. whole 1024-byte swizzle atoms), with RH live row
// halves (RH = 4: the 32-row pair consumer); else the shuffle consumer
// (plain rows, decode only).
template <int D, int G, bool BF16, bool MMA, int RH>
__global__ void __launch_bounds__(TmaCfg<D, MMA>::THREADS, TmaCfg<D, MMA>::MINB)
    decode_tma_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, int box_rows) {
  constexpr int NCW = TmaCfg<D, MMA>::NCW, KT = TmaCfg<D, MMA>::KT;
  using WM = typename std::conditional<RH == 4, DecodeMmaPairWarp<D, G, BF16, NCW, KT>,
                                       DecodeMmaWarp<D, G, BF16, NCW, KT, (RH == 4 ? 2 : RH)>>::type;
  using W = typename std::conditional<MMA, WM, DecodeWarp<D, G, BF16, NCW, KT>>::type;
  using C = TmaCfg<D, MMA, W::ROWS>;
  constexpr int NS = C::NS, STAGE = C::STAGE;
  using T = typename W::T;

  extern __shared__ __align__(1024) uint8_t dsmem[];
  const WsHeader* hdr = static_cast<const WsHeader*>(p.ws);
  // the page table failed the index check: the whole CTA leaves before any
  // barrier or copy
  if (hdr->index_error) return;
  if (MMA && (smem_u32(dsmem) & 1023u) != 0) {
    // the swizzle pattern is anchored to 1024-byte boundaries: report and
    // skip the work rather than compute with a shifted pattern
    if (threadIdx.x == 0) atomicExch(&const_cast<WsHeader*>(hdr)->err_flag, 1);
    return;
  }
  T* sK = reinterpret_cast<T*>(dsmem);
  T* sV = sK + NS * STAGE;
  float* sm_o = reinterpret_cast<float*>(dsmem + C::O_OFF);
  float (*sm_m)[kMaxRows] = reinterpret_cast<float (*)[kMaxRows]>(dsmem + C::ML_OFF);
  float (*sm_l)[kMaxRows] = sm_m + NCW;
  T* sQ = reinterpret_cast<T*>(dsmem + C::Q_OFF);
  StageHdr* sH = reinterpret_cast<StageHdr*>(dsmem + C::HDR_OFF);
  const uint32_t* sMask = reinterpret_cast<const uint32_t*>(dsmem + C::MASK_OFF);
  const uint32_t bar0 = smem_u32(dsmem + C::BAR_OFF);
  auto FULL = [&](int s) { return bar0 + 8u * uint32_t(s); };
  auto EMPTY = [&](int s) { return bar0 + 8u * uint32_t(NS + s); };
  const uint32_t QFREE = bar0 + 8u * uint32_t(2 * NS);
  const uint32_t MERGE = bar0 + 8u * uint32_t(2 * NS + 1);
  volatile WaitCtl* ctl = reinterpret_cast<volatile WaitCtl*>(dsmem + C::BAR_OFF + C::NBAR * 8);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(FULL(s), 1);
      mbar_init(EMPTY(s), NCW);
    }
    mbar_init(QFREE, NCW);
    mbar_init(MERGE, NCW * 32);
    ctl->abort = 0;
    ctl->limit_ns = wait_limit_of(hdr);
    mbar_init_fence();
  }
  const int causal = hdr->causal;
  const int window_left = hdr->window_left;
  __syncthreads();

  if (warp == NCW) {
    decode_producer<D, G, BF16, MMA, W>(p, &tk, &tv, box_rows, dsmem, lane, causal, window_left,
                                   ctl);
  } else {
    // ------------------------------------------------------------ consumers
    float* tmp_lse = ws_ptr<float>(p.ws, hdr->off_tmp_lse);
    float* tmp_o = ws_ptr<float>(p.ws, hdr->off_tmp_o);
    W wk;
    wk.setup(warp, lane);
    uint32_t n_sync = 0;
    // barrier over the consumer threads, bounded like every other wait
    auto consumer_sync = [&] {
      mbar_arrive(MERGE);
      mbar_wait(MERGE, n_sync & 1u, ctl);
      ++n_sync;
    };
    for (int c = 0;; ++c) {
      const int st = c % NS;
      // an expired wait ends the warp's work (the abort flag then makes
      // every other wait return at once); the error is reported below
      if (!mbar_wait(FULL(st), uint32_t(c / NS) & 1u, ctl)) break;
      // the header is read in place (fields load where they are used); the
      // output fields are copied out before the slot is released
      const StageHdr& h = sH[st];
      const int flags = h.flags;
      if (flags & kStEnd) break;
      if (flags & kStFirst) {
        wk.begin(sQ, h.n_rows, p.sm_scale_log2);
        __syncwarp();
        if (lane == 0) mbar_arrive(QFREE);
      }
      if (!(flags & kStNoKeys))
        wk.stage(sK + st * STAGE, sV + st * STAGE, h, causal, window_left,
                 MMA && p.custom_mask ? sMask + st * C::ROWS * C::MASKW : nullptr);
      StageHdr out;
      if (flags & kStLast) out = h;
      __syncwarp();
      if (lane == 0) mbar_arrive(EMPTY(st));
      if (flags & kStLast) {
        wk.publish_ml(sm_m, sm_l);
        consumer_sync();
#pragma unroll
        for (int round = 0; round < W::ROUNDS; ++round) {
          if constexpr (W::kPair) {
            // the two warps of the round's M tile: key half 0 stores, half 1 adds
            const int w0 = 2 * (round >> 1);
            if (warp == w0) wk.add_o(round, out.n_rows, true, sm_o, sm_m);
            consumer_sync();
            if (warp == w0 + 1) wk.add_o(round, out.n_rows, false, sm_o, sm_m);
            consumer_sync();
          } else if (C::MB == 2) {
            // warps 0 and 2 store into buffers 0 and 1, then 1 and 3 add
            float* buf = sm_o + (warp >> 1) * 8 * D;
            if ((warp & 1) == 0) wk.add_o(round, out.n_rows, true, buf, sm_m);
            consumer_sync();
            if (warp & 1) wk.add_o(round, out.n_rows, false, buf, sm_m);
            consumer_sync();
          } else {
            for (int w = 0; w < NCW; ++w) {
              if (warp == w) wk.add_o(round, out.n_rows, w == 0, sm_o, sm_m);
              consumer_sync();
            }
          }
          write_rows<D, G, BF16, NCW, C::MB>(p, out, 8 * round, tmp_o, tmp_lse, tid, sm_o, sm_m,
                                             sm_l);
          consumer_sync();
        }
      }
    }
  }
  // the split-KV merge launched after this kernel may start its launch now
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __syncthreads();
  if (tid == 0 && ctl->abort) {
    int* err = const_cast<int*>(&hdr->err_flag);
    atomicExch(err, 1);
  }
}

// -------------------------------------------------------------- launchers

template <int D, int G, bool BF16, bool MMA, int RH>
cudaError_t launch_k(const AttnParams& p, int grid, const CUtensorMap& tk, const CUtensorMap& tv,
                     int box_rows, cudaStream_t s) {
  using C = TmaCfg<D, MMA, (MMA && RH == 4) ? 32 : 16>;
  auto k = decode_tma_kernel<D, G, BF16, MMA, RH>;
  // once per device, before any capture (no attribute call inside a captured run)
  static std::atomic<uint64_t> done{0};
  const cudaError_t attr = smem_attr_once(k, C::SMEM, done);
  if (attr != cudaSuccess) return attr;
  k<<<grid, C::THREADS, C::SMEM, s>>>(p, tk, tv, box_rows);
  return cudaGetLastError();
}

}  // namespace

// The 32-row pair consumer's launches (their own translation unit, which
// keeps each unit's compile time short).
cudaError_t launch_decode_pair(const AttnParams& p, int head_dim, int group, bool bf16, int grid,
                               const CUtensorMap& tk, const CUtensorMap& tv, int box_rows,
                               cudaStream_t s);

}  // namespace fi
