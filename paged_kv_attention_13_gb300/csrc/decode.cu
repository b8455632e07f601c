// Decode kernels: one query row per request against its paged KV, all G query
// heads of one kv head together (GQA). Bandwidth-bound: every K/V byte is
// read exactly once, scores are reduced with warp shuffles, and the online
// softmax is kept in fp32.
//
// Work item = (request, kv head, key chunk). The item's live keys stream
// through a ring of stages in shared memory, each stage a tile of KT keys of
// K and of V. Consumer warps take KT / warps keys of a stage each: a warp step
// covers 32 / (D/8) keys, each key's D/8 lanes holding 8 head-dim elements.
// At the end of an item the warps' (max, sum, o) states are merged in shared
// memory.
//
// One producer warp fills the ring: per page of a stage it issues one
// cp.async.bulk.tensor box of K and one of V (4-D maps over [pages, slot,
// kv head, dim]), and for an item's first stage q by plain bulk copy;
// mbarriers hand the stages to the consumer warps and back. The producer
// runs ahead across work items, so the ring stays full through item
// boundaries, and the consumer warps issue no load instructions at all.
// (A version in which every thread gathered 16-byte chunks with cp.async
// reached 4870 GB/s at best on the batch-64 decode, against 5750 for this
// one, and was slower at page size 1 too.)
//
// Mask for one query row (Lq = 1) [P1 "Why window_size_right stays -1"],
// [P2 "Summary"]: causal keeps every key j <= Lk - 1; the window keeps
// j >= Lk - 1 - window_left. So decode needs only a key range.
//   [P1] "Route non-causal windowed prefill to AITER's masked kernel" (#339)
//   [P2] "Support speculative-decode verify on ROCm, and stop auto routing
//         short-query prefill to AITER" (#362)
#include <type_traits>

#include "tma.cuh"

namespace fi {
namespace {

// ------------------------------------------------------------------ geometry

// Live keys [lo, hi) of one work item, visited as tiles of `kt` keys from
// `start` = lo rounded down to `align` (a power of two); keys below lo in the
// first tile are masked.
struct DecodeRange {
  int lo, hi, start, n_tiles;
};

__device__ __forceinline__ DecodeRange decode_range(const WorkItem& it, int lk, int window_left,
                                                    int align, int kt) {
  DecodeRange r;
  r.hi = min(it.kv_end, lk);
  r.lo = it.kv_begin;
  if (window_left >= 0) r.lo = max(r.lo, lk - 1 - window_left);
  r.lo = max(r.lo, 0);
  r.start = r.lo & ~(align - 1);
  r.n_tiles = r.hi > r.lo ? (r.hi - r.start + kt - 1) / kt : 0;
  return r;
}

// Merge the NWARP consumer warps' states of one work item and write o / lse:
// directly, or to the item's split-KV partial slot. sm_o holds the warps'
// unnormalised o as [NWARP][G][D] floats; sm_m / sm_l their per-head running
// max (log2 domain) and sum.
template <int D, int G, bool BF16, int NWARP>
__device__ __forceinline__ void decode_merge_write(const AttnParams& p, int token, int hk, int chunk,
                                                   int partial_base, float* tmp_o, float* tmp_lse,
                                                   int tid, const float* sm_o,
                                                   const float (*sm_m)[G],
                                                   const float (*sm_l)[G]) {
  using DT = Dt<BF16>;
  using T = typename DT::T;
  const int Hq = p.num_qo_heads;
  const bool direct = chunk < 0;
  const int slot = direct ? 0 : partial_base + chunk;
  for (int idx = tid; idx < G * (D / 4); idx += NWARP * 32) {
    const int h = idx / (D / 4);
    const int c = (idx % (D / 4)) * 4;
    float M = neg_inf();
#pragma unroll
    for (int wq = 0; wq < NWARP; ++wq) M = fmaxf(M, sm_m[wq][h]);
    const float Mu = (M == neg_inf()) ? 0.f : M;
    float den = 0.f;
    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int wq = 0; wq < NWARP; ++wq) {
      const float sc = ex2(sm_m[wq][h] - Mu);
      den += sc * sm_l[wq][h];
      const float4 ov = *reinterpret_cast<const float4*>(sm_o + (wq * G + h) * D + c);
      num.x += sc * ov.x; num.y += sc * ov.y; num.z += sc * ov.z; num.w += sc * ov.w;
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    const int head = hk * G + h;
    if (direct) {
      T* op = static_cast<T*>(p.out) + (int64_t(token) * Hq + head) * D + c;
      uint2 pk;
      pk.x = DT::pack(num.x * inv, num.y * inv);
      pk.y = DT::pack(num.z * inv, num.w * inv);
      *reinterpret_cast<uint2*>(op) = pk;
    } else {
      float* op = tmp_o + (int64_t(slot) * Hq + head) * D + c;
      *reinterpret_cast<float4*>(op) =
          make_float4(num.x * inv, num.y * inv, num.z * inv, num.w * inv);
    }
    if (c == 0) {
      const float lse = den > 0.f ? (M + __log2f(den)) * kLn2 : neg_inf();
      if (direct) {
        if (p.lse) p.lse[int64_t(token) * Hq + head] = lse;
      } else {
        tmp_lse[int64_t(slot) * Hq + head] = lse;
      }
    }
  }
}

// ------------------------------------------------------------- warp consumer

// One consumer warp's share of a work item: q of the G heads pre-scaled into
// the exp2 domain (fp32 pairs for the packed FMA), o of every head on this
// lane's 8 dims, and the running max / sum of the head whose score this lane
// holds after the reduce-scatter.
template <int D, int G, bool BF16, int NWARP, int KT>
struct DecodeWarp {
  using DT = Dt<BF16>;
  using T = typename DT::T;
  static constexpr int LPK = D / 8;          // lanes per key
  static constexpr int KPS = 32 / LPK;       // keys per warp step
  static constexpr int KPW = KT / NWARP;     // keys per warp per stage
  static constexpr int STEPS = KPW / KPS;    // warp steps per stage
  static_assert(KPW % KPS == 0, "a warp's keys of a stage are whole warp steps");
  static constexpr bool kSwizzled = false;  // reads K/V stages as plain [KT][D] rows

  int warp, lane, kg, dl;
  int myh;          // head whose score this lane holds after the reduce-scatter
  int src_of[G];    // lane (within this key's lane group) holding head h's score
  float2 q2[G][4];  // slot s holds head (myh ^ s)
  float2 o2[G][4];
  float m_me, l_me;

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

  // Load q of the item's G heads; reset o and the running max / sum. Slot s
  // holds head (myh ^ s): at each level of the reduce-scatter a lane then
  // keeps its first half of the slots and sends the second, with no per-lane
  // selection.
  __device__ __forceinline__ void begin(const AttnParams& p, int token, int hk) {
#pragma unroll
    for (int sl = 0; sl < G; ++sl) {
      const int h = myh ^ sl;
      const T* qp = static_cast<const T*>(p.q) + int64_t(token) * p.q_stride_tok +
                    int64_t(hk * G + h) * p.q_stride_head + dl * 8;
      uint4 r = ld_nc16(qp);
      const uint32_t wv[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        q2[sl][e] = make_float2(DT::lo(wv[e]) * p.sm_scale_log2, DT::hi(wv[e]) * p.sm_scale_log2);
    }
    m_me = neg_inf();
    l_me = 0.f;
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < 4; ++e) o2[h][e] = make_float2(0.f, 0.f);
  }

  // Same as begin(), with q of the G heads staged in shared memory as
  // [G][D] (head h of the group at row h).
  __device__ __forceinline__ void begin_smem(const T* qs, float sm_scale_log2) {
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

  // Consume one stage: keys k0 .. k0+KT-1 in rows 0..KT-1 of cK / cV, of
  // which [lo, hi) are live. Rows outside the live range may hold anything
  // (a neighbour's page slots): their scores are masked to -inf and their V
  // rows are read as zero, so no value there reaches o.
  __device__ __forceinline__ void stage(T* cK, T* cV, int k0, int lo, int hi) {
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

  // Merge the NWARP warps' states of the item and write o / lse (directly, or
  // to the item's split-KV partial slot). `sync` is a barrier over the
  // consumer threads (tid = 0 .. NWARP*32-1); sm_o holds NWARP x G x D
  // floats. Ends with a barrier, so the shared arrays are free on return.
  template <class Sync>
  __device__ __forceinline__ void finish(const AttnParams& p, int token, int hk, int chunk,
                                         int partial_base, float* tmp_o, float* tmp_lse, int tid,
                                         float* sm_o, float (*sm_m)[G], float (*sm_l)[G],
                                         Sync sync) {
    // sums over the warp's key groups (they share each head's max)
    float l_h[G], m_h[G];
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
    if (kg == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float4* dst = reinterpret_cast<float4*>(sm_o + (warp * G + h) * D + dl * 8);
        dst[0] = make_float4(o2[h][0].x, o2[h][0].y, o2[h][1].x, o2[h][1].y);
        dst[1] = make_float4(o2[h][2].x, o2[h][2].y, o2[h][3].x, o2[h][3].y);
      }
    }
    sync();
    decode_merge_write<D, G, BF16, NWARP>(p, token, hk, chunk, partial_base, tmp_o, tmp_lse, tid,
                                           sm_o, sm_m, sm_l);
    sync();
  }
};

// A consumer warp on the warp-level tensor cores. The GQA group is a dense
// contraction: S = Q K^T with Q the G heads' rows (padded to the 16 rows of
// mma.m16n8k16) against the warp's KPW keys, then O += P V. K and V stages
// are 128B-swizzled 64-column halves written by TMA, so ldmatrix reads them
// without bank conflicts. The fragment row of lane l is head l / 4 (rows
// G..15 are zero padding); its running max / sum live in the lane's quad.
// Per stage a warp issues about 80 instructions for its 16 keys, against
// about 900 for the shuffle-reduction consumer above.
template <int D, int G, bool BF16, int NWARP, int KT>
struct DecodeMmaWarp {
  using DT = Dt<BF16>;
  using T = typename DT::T;
  static constexpr int KPW = KT / NWARP;  // keys per warp per stage
  static constexpr int NT = KPW / 8;      // n8 score tiles per warp
  static constexpr int KD = D / 16;       // k16 steps over the head dim
  static constexpr int HALF = KT * 128;   // bytes of one 64-column half of a stage
  static_assert(KPW % 16 == 0, "a warp's keys are whole k16 steps of P V");
  static_assert(G <= 8, "the group fits the live fragment rows");
  static constexpr bool kSwizzled = true;

  int warp, lane, qr, qc;
  uint32_t qa0[KD], qa2[KD];  // A fragment, row qr: columns kd*16 + qc*2 (+8)
  float o[D / 8][4];          // rows qr (live for qr < G) and qr + 8 (padding)
  float m_me, l_me, scale;

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

  // q of the G heads staged in shared memory as [G][D]
  __device__ __forceinline__ void begin_smem(const T* qs, float sm_scale_log2) {
#pragma unroll
    for (int kd = 0; kd < KD; ++kd) {
      qa0[kd] = 0u;
      qa2[kd] = 0u;
      if (qr < G) {
        qa0[kd] = *reinterpret_cast<const uint32_t*>(qs + qr * D + kd * 16 + qc * 2);
        qa2[kd] = *reinterpret_cast<const uint32_t*>(qs + qr * D + kd * 16 + 8 + qc * 2);
      }
    }
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    m_me = neg_inf();
    l_me = 0.f;
    scale = sm_scale_log2;
  }

  // Consume one stage (keys k0 .. k0+KT-1, live [lo, hi)). In a stage that
  // is not entirely live the warp first zeroes its V rows outside the range:
  // they may hold anything (a neighbour's slots), and 0 * NaN would reach o.
  __device__ __forceinline__ void stage(T* cK, T* cV, int k0, int lo, int hi) {
    const uint32_t sk = smem_u32(cK), sv = smem_u32(cV);
    const int kb = warp * KPW;  // this warp's first key in the stage
    const bool full_tile = k0 >= lo && k0 + KT <= hi;
    if (!full_tile) {
      // lane l zeroes chunks l, l+32, ... of the warp's dead rows
      for (int idx = lane; idx < KPW * (D / 8); idx += 32) {
        const int r = kb + idx / (D / 8), c = idx % (D / 8);
        const int kk = k0 + r;
        if (kk < lo || kk >= hi)
          *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(cV) + swz(r, c)) =
              make_uint4(0u, 0u, 0u, 0u);
      }
      // these generic-proxy writes are ordered before the slot's next TMA fill
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
    }
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int kd = 0; kd < KD; ++kd) {
      const uint32_t a[4] = {qa0[kd], 0u, qa2[kd], 0u};
#pragma unroll
      for (int nt = 0; nt < NT; nt += 2) {
        const int r = kb + nt * 8 + (lane & 7) + (lane >> 4) * 8;
        const int c = kd * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sk + swz(r, c), b0, b1, b2, b3);
        mma16816<BF16>(s[nt], a, b0, b1);
        mma16816<BF16>(s[nt + 1], a, b2, b3);
      }
    }
    // row qr's scores: s[nt][e], key kb + nt*8 + qc*2 + e (e < 2)
    float mx = neg_inf();
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float x = s[nt][e] * scale;
        if (!full_tile) {
          const int kk = k0 + kb + nt * 8 + qc * 2 + e;
          if (kk < lo || kk >= hi) x = neg_inf();
        }
        s[nt][e] = x;
        mx = fmaxf(mx, x);
      }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    // lazy max, as in the shuffle consumer
    float mn = m_me;
    if (mx > m_me + 8.f || (m_me == neg_inf() && mx != neg_inf())) mn = mx;
    const float corr = (mn == m_me) ? 1.f : ex2(m_me - mn);
    const float mu = (mn == neg_inf()) ? 0.f : mn;
    m_me = mn;
    float psum = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        s[nt][e] = ex2(s[nt][e] - mu);
        psum += s[nt][e];
      }
    l_me = l_me * corr + psum;
    if (__any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        o[i][0] *= corr;
        o[i][1] *= corr;
      }
    }
#pragma unroll
    for (int kk = 0; kk < KPW / 16; ++kk) {
      const uint32_t pa[4] = {DT::pack(s[2 * kk][0], s[2 * kk][1]), 0u,
                              DT::pack(s[2 * kk + 1][0], s[2 * kk + 1][1]), 0u};
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

  template <class Sync>
  __device__ __forceinline__ void finish(const AttnParams& p, int token, int hk, int chunk,
                                         int partial_base, float* tmp_o, float* tmp_lse, int tid,
                                         float* sm_o, float (*sm_m)[G], float (*sm_l)[G],
                                         Sync sync) {
    float l = l_me;
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    if (qr < G) {
      if (qc == 0) {
        sm_m[warp][qr] = m_me;
        sm_l[warp][qr] = l;
      }
      float* dst = sm_o + (warp * G + qr) * D + qc * 2;
#pragma unroll
      for (int i = 0; i < D / 8; ++i)
        *reinterpret_cast<float2*>(dst + i * 8) = make_float2(o[i][0], o[i][1]);
    }
    sync();
    decode_merge_write<D, G, BF16, NWARP>(p, token, hk, chunk, partial_base, tmp_o, tmp_lse, tid,
                                           sm_o, sm_m, sm_l);
    sync();
  }
};

// ------------------------------------------------------------ TMA kernel

// Ring geometry of the TMA kernel: NCW consumer warps of KPW keys each per
// stage (D = 128; twice as many keys at D = 64, so a stage is always the same
// bytes), NS stages, MINB CTAs per SM. Among the shapes that fit three CTAs
// per SM, 2 stages of 64 keys measured fastest.
template <int D>
struct TmaCfg {
  static constexpr int NCW = 4;
  static constexpr int KPW = 16;
  static constexpr int KT = NCW * KPW * (128 / D);  // keys per stage (a power of two)
  static constexpr int NS = 2;
  static constexpr int MINB = 3;
  static constexpr int THREADS = (NCW + 1) * 32;
  static constexpr int STAGE = KT * D;             // elements per stage, K or V
  static constexpr int RING_BYTES = NS * STAGE * 2 * 2;
  static constexpr int NBAR = 2 * NS + 1;          // full, empty per slot; merge
  // dynamic shared memory: K/V ring | o partials | per-warp max, sum |
  // q per slot | stage header per slot | barriers, abort flag
  template <int G> static constexpr int o_off() { return RING_BYTES; }
  template <int G> static constexpr int ml_off() { return o_off<G>() + NCW * G * D * 4; }
  template <int G> static constexpr int q_off() { return ml_off<G>() + 2 * NCW * G * 4; }
  template <int G> static constexpr int hdr_off() { return q_off<G>() + NS * G * D * 2; }
  template <int G> static constexpr int bar_off() { return hdr_off<G>() + NS * 32; }
  template <int G> static constexpr int smem_bytes() { return bar_off<G>() + NBAR * 8 + 16; }
  static_assert((KT & (KT - 1)) == 0, "keys per stage is a power of two");
  static_assert(MINB * (smem_bytes<4>() + 1024) <= 233472, "MINB CTAs fit one SM's shared memory");
};

// Stage header, written by the producer before it arms the stage's barrier.
enum : int32_t { kStFirst = 1, kStLast = 2, kStEnd = 4, kStNoKeys = 8 };
struct alignas(16) StageHdr {
  int32_t flags, k0, lo, hi;                      // this stage
  int32_t token, kv_head, chunk, partial_base;    // its work item
};

// MMA selects the tensor-core consumer (stages 128B-swizzled, 64-column
// boxes; needs boxes of at least 8 slots, i.e. whole 1024-byte swizzle
// atoms), else the shuffle-reduction consumer (plain rows).
template <int D, int G, bool BF16, bool MMA>
__global__ void __launch_bounds__(TmaCfg<D>::THREADS, TmaCfg<D>::MINB)
    decode_tma_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, int box_rows) {
  using C = TmaCfg<D>;
  constexpr int NCW = C::NCW, KT = C::KT, NS = C::NS, STAGE = C::STAGE;
  using W = typename std::conditional<MMA, DecodeMmaWarp<D, G, BF16, NCW, KT>,
                                      DecodeWarp<D, G, BF16, NCW, KT>>::type;
  using T = typename W::T;

  extern __shared__ __align__(1024) uint8_t dsmem[];
  if (MMA && (smem_u32(dsmem) & 1023u) != 0) {
    // the swizzle pattern is anchored to 1024-byte boundaries: report and
    // skip the work rather than compute with a shifted pattern
    if (threadIdx.x == 0) atomicExch(&const_cast<WsHeader*>(static_cast<const WsHeader*>(p.ws))->err_flag, 1);
    return;
  }
  T* sK = reinterpret_cast<T*>(dsmem);
  T* sV = sK + NS * STAGE;
  float* sm_o = reinterpret_cast<float*>(dsmem + C::template o_off<G>());
  float (*sm_m)[G] = reinterpret_cast<float (*)[G]>(dsmem + C::template ml_off<G>());
  float (*sm_l)[G] = sm_m + NCW;
  T* sQ = reinterpret_cast<T*>(dsmem + C::template q_off<G>());  // [NS][G][D]
  StageHdr* sH = reinterpret_cast<StageHdr*>(dsmem + C::template hdr_off<G>());
  const uint32_t bar0 = smem_u32(dsmem + C::template bar_off<G>());
  auto FULL = [&](int s) { return bar0 + 8u * uint32_t(s); };
  auto EMPTY = [&](int s) { return bar0 + 8u * uint32_t(NS + s); };
  const uint32_t MERGE = bar0 + 8u * uint32_t(2 * NS);
  volatile int* abort_flag =
      reinterpret_cast<volatile int*>(dsmem + C::template bar_off<G>() + C::NBAR * 8);

  const WsHeader* hdr = static_cast<const WsHeader*>(p.ws);
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(FULL(s), 1);
      mbar_init(EMPTY(s), NCW);
    }
    mbar_init(MERGE, NCW * 32);
    *abort_flag = 0;
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == NCW) {
    // ------------------------------------------------------------ producer
    // Stage c of this CTA's sequence goes to slot c % NS; its (c / NS)-th
    // fill waits for the consumers' release of the previous one. Everything
    // a stage needs from global memory (the item's metadata, the page
    // indices) is loaded before that wait, so a full ring hides it.
    const int n_items = hdr->n_items;
    const WorkItem* items = ws_ptr<const WorkItem>(p.ws, hdr->off_items);
    const int32_t* qo_indptr = ws_ptr<const int32_t>(p.ws, hdr->off_qo_indptr);
    const int32_t* kv_indptr = ws_ptr<const int32_t>(p.ws, hdr->off_kv_indptr);
    const int32_t* kv_len = ws_ptr<const int32_t>(p.ws, hdr->off_kv_len);
    const int window_left = hdr->window_left;
    const int n_boxes = KT / box_rows;  // a stage is n_boxes boxes of box_rows slots of one page
    const uint32_t box_bytes = uint32_t(box_rows) * D * 2;
    constexpr int BPL = (KT + 31) / 32;  // boxes per lane, at most
    int c = 0;
    bool ok = true;
    uint32_t last_par[NS];
    bool armed[NS];
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      armed[s] = false;
      last_par[s] = 0;
    }
    // claim slot st for stage c: wait for its release, then write the header
    // and arm its barrier for `bytes` (lane 0); false once the CTA aborts.
    // Every armed phase is recorded (the end-of-work stage too), so the drain
    // below waits on each slot's latest phase.
    auto claim = [&](int st, uint32_t par, const StageHdr& h, uint32_t bytes) {
      bool okl = true;
      if (lane == 0) {
        if (c >= NS) okl = mbar_wait(EMPTY(st), par ^ 1u, abort_flag);
        if (okl) {
          sH[st] = h;
          mbar_expect_tx(FULL(st), bytes);
        }
      }
      okl = __shfl_sync(0xffffffffu, okl, 0) != 0;
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
      const WorkItem it = items[w];
      if (it.b < 0) continue;  // schedule padding
      const int token = qo_indptr[it.b];
      const DecodeRange R = decode_range(it, kv_len[it.b], window_left, box_rows, KT);
      const int32_t* pages = p.kv_indices + kv_indptr[it.b];
      const T* qsrc = static_cast<const T*>(p.q) + int64_t(token) * p.q_stride_tok +
                      int64_t(it.kv_head * G) * p.q_stride_head;
      const int n_st = max(R.n_tiles, 1);  // an item without keys still writes its output
      for (int t = 0; t < n_st; ++t, ++c) {
        const int st = c % NS;
        const uint32_t par = uint32_t(c / NS) & 1u;
        const int k0 = R.start + t * KT;
        const int n_live = R.n_tiles ? min(n_boxes, (R.hi - k0 + box_rows - 1) / box_rows) : 0;
        int page[BPL], slot[BPL];
#pragma unroll
        for (int j = 0; j < BPL; ++j) {
          const int i = lane + 32 * j;
          page[j] = 0;
          slot[j] = 0;
          if (i < n_live) {
            const int kb = k0 + i * box_rows;
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
        StageHdr h;
        h.flags = (t == 0 ? kStFirst : 0) | (t == n_st - 1 ? kStLast : 0) |
                  (R.n_tiles ? 0 : kStNoKeys);
        h.k0 = k0;
        h.lo = R.lo;
        h.hi = R.hi;
        h.token = token;
        h.kv_head = it.kv_head;
        h.chunk = it.chunk;
        h.partial_base = it.partial_base;
        const uint32_t qbytes = t == 0 ? uint32_t(G * D * 2) : 0u;
        if (!claim(st, par, h, uint32_t(n_live) * box_bytes * 2u + qbytes)) {
          ok = false;
          break;
        }
        if (t == 0 && lane < G)
          bulk_load(smem_u32(sQ + (st * G + lane) * D), qsrc + int64_t(lane) * p.q_stride_head,
                    uint32_t(D * 2), FULL(st));
        const uint32_t dk = smem_u32(sK + st * STAGE), dv = smem_u32(sV + st * STAGE);
#pragma unroll
        for (int j = 0; j < BPL; ++j) {
          const int i = lane + 32 * j;
          if (i < n_live) {
            if constexpr (W::kSwizzled) {
              // one box per 64-column half; half h of the stage at h * KT * 128
              const uint32_t off = uint32_t(i * box_rows) * 128u;
#pragma unroll
              for (int h = 0; h < D / 64; ++h) {
                tma_load_4d(dk + h * KT * 128 + off, &tk, FULL(st), h * 64, it.kv_head, slot[j], page[j]);
                tma_load_4d(dv + h * KT * 128 + off, &tv, FULL(st), h * 64, it.kv_head, slot[j], page[j]);
              }
            } else {
              const uint32_t off = uint32_t(i) * box_bytes;
              tma_load_4d(dk + off, &tk, FULL(st), 0, it.kv_head, slot[j], page[j]);
              tma_load_4d(dv + off, &tv, FULL(st), 0, it.kv_head, slot[j], page[j]);
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
      if (!claim(st, uint32_t(c / NS) & 1u, h, 0u)) ok = false;
    }
    // Drain: the last fill of every slot has landed before the CTA exits
    // (the consumers waited for all of them unless a wait expired; this wait
    // ignores the abort flag but keeps its time bound).
    if (lane == 0) {
      volatile int no_abort = 0;
#pragma unroll
      for (int s = 0; s < NS; ++s)
        if (armed[s] && !mbar_wait(FULL(s), last_par[s], &no_abort)) *abort_flag = 1;
    }
  } else {
    // ------------------------------------------------------------ consumers
    // Consumers read nothing from global memory: each stage's header says
    // which keys it holds and where the item's output goes, and an item's
    // first stage brings its q.
    float* tmp_lse = ws_ptr<float>(p.ws, hdr->off_tmp_lse);
    float* tmp_o = ws_ptr<float>(p.ws, hdr->off_tmp_o);
    W wk;
    wk.setup(warp, lane);
    uint32_t n_sync = 0;
    // barrier over the consumer threads, bounded like every other wait
    auto consumer_sync = [&] {
      mbar_arrive(MERGE);
      mbar_wait(MERGE, n_sync & 1u, abort_flag);
      ++n_sync;
    };
    for (int c = 0;; ++c) {
      const int st = c % NS;
      // an expired wait ends the warp's work (the abort flag then makes
      // every other wait return at once); the error is reported below
      if (!mbar_wait(FULL(st), uint32_t(c / NS) & 1u, abort_flag)) break;
      const StageHdr h = sH[st];
      if (h.flags & kStEnd) break;
      if (h.flags & kStFirst) wk.begin_smem(sQ + st * G * D, p.sm_scale_log2);
      if (!(h.flags & kStNoKeys)) wk.stage(sK + st * STAGE, sV + st * STAGE, h.k0, h.lo, h.hi);
      __syncwarp();
      if (lane == 0) mbar_arrive(EMPTY(st));
      if (h.flags & kStLast)
        wk.finish(p, h.token, h.kv_head, h.chunk, h.partial_base, tmp_o, tmp_lse, tid, sm_o,
                  sm_m, sm_l, consumer_sync);
    }
  }
  __syncthreads();
  if (tid == 0 && *abort_flag) {
    int* err = const_cast<int*>(&hdr->err_flag);
    atomicExch(err, 1);
  }
}

// -------------------------------------------------------------- launchers

template <int D, int G, bool BF16, bool MMA>
cudaError_t launch_dg(const AttnParams& p, int grid, const CUtensorMap& tk, const CUtensorMap& tv,
                      int box_rows, cudaStream_t s) {
  using C = TmaCfg<D>;
  auto k = decode_tma_kernel<D, G, BF16, MMA>;
  constexpr int smem = C::template smem_bytes<G>();
  // once per process, before any capture (no attribute call inside a captured run)
  static cudaError_t attr = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (attr != cudaSuccess) return attr;
  k<<<grid, C::THREADS, smem, s>>>(p, tk, tv, box_rows);
  return cudaGetLastError();
}

template <int D, bool BF16, bool MMA>
cudaError_t launch_d(const AttnParams& p, int group, int grid, const CUtensorMap& tk,
                     const CUtensorMap& tv, int box_rows, cudaStream_t s) {
  switch (group) {
    case 1: return launch_dg<D, 1, BF16, MMA>(p, grid, tk, tv, box_rows, s);
    case 2: return launch_dg<D, 2, BF16, MMA>(p, grid, tk, tv, box_rows, s);
    case 4: return launch_dg<D, 4, BF16, MMA>(p, grid, tk, tv, box_rows, s);
    default: return cudaErrorInvalidValue;
  }
}

template <int D, bool BF16>
cudaError_t launch_dm(const AttnParams& p, int group, int grid, const CUtensorMap& tk,
                      const CUtensorMap& tv, int box_rows, bool mma, cudaStream_t s) {
  return mma ? launch_d<D, BF16, true>(p, group, grid, tk, tv, box_rows, s)
             : launch_d<D, BF16, false>(p, group, grid, tk, tv, box_rows, s);
}

int gcd_int(int a, int b) {
  while (b) {
    const int t = a % b;
    a = b;
    b = t;
  }
  return a;
}

}  // namespace

int decode_ctas_per_sm(int head_dim) {
  return head_dim == 64 ? TmaCfg<64>::MINB : TmaCfg<128>::MINB;
}

cudaError_t launch_decode(const AttnParams& p, int head_dim, int group, bool bf16,
                          int64_t num_pages, int grid, cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  if (head_dim != 128 && head_dim != 64) return cudaErrorInvalidValue;
  // Boxes of gcd(page_size, KT) slots never cross a page: every box starts
  // at a multiple of that size (tiles start at lo rounded down to it).
  const int kt = head_dim == 128 ? TmaCfg<128>::KT : TmaCfg<64>::KT;
  const int box_rows = gcd_int(p.page_size, kt);
  // Tensor-core consumer when a box spans whole swizzle atoms (8 slots of
  // 128 bytes per 64-column half); shuffle consumer for smaller boxes.
  const bool mma = box_rows >= 8;
  const int box_cols = mma ? 64 : head_dim;
  const CUtensorMapSwizzle swz = mma ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  CUtensorMap tk, tv;
  if (num_pages <= 0 ||
      !encode_paged_kv_map(&tk, bf16, p.k, head_dim, p.num_kv_heads, p.page_size, num_pages,
                           p.k_stride_head, p.k_stride_tok, p.k_stride_page, box_cols, box_rows,
                           swz) ||
      !encode_paged_kv_map(&tv, bf16, p.v, head_dim, p.num_kv_heads, p.page_size, num_pages,
                           p.v_stride_head, p.v_stride_tok, p.v_stride_page, box_cols, box_rows,
                           swz))
    return cudaErrorInvalidValue;
  if (head_dim == 128)
    return bf16 ? launch_dm<128, true>(p, group, grid, tk, tv, box_rows, mma, stream)
                : launch_dm<128, false>(p, group, grid, tk, tv, box_rows, mma, stream);
  return bf16 ? launch_dm<64, true>(p, group, grid, tk, tv, box_rows, mma, stream)
              : launch_dm<64, false>(p, group, grid, tk, tv, box_rows, mma, stream);
}

}  // namespace fi
