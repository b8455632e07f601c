// Decode kernel: one query row per request against its paged KV, all G query
// heads of one kv head together (GQA). Bandwidth-bound: every K/V byte is
// read exactly once, with 16-byte coalesced cp.async gathers,
// scores reduced with warp shuffles, and an online softmax kept in fp32.
//
// Work item = (request, kv head, key chunk). A CTA of 4 warps streams the
// chunk's live keys through a 3-stage cp.async ring in shared memory (32 keys
// of K and V per stage, gathered page by page, zero-filled past the end), so
// two stages of loads stay in flight while one is consumed; four CTAs share
// an SM. Each warp takes
// 8 keys of a stage; a warp step covers 32 / (D/8) keys, each key's D/8 lanes
// holding 8 head-dim elements. At the end the four warps' (max, sum, o)
// states are merged in shared memory.
//
// Mask for one query row (Lq = 1) [P1 "Why window_size_right stays -1"],
// [P2 "Summary"]: causal keeps every key j <= Lk - 1; the window keeps
// j >= Lk - 1 - window_left. So decode needs only a key range.
//   [P1] "Route non-causal windowed prefill to AITER's masked kernel" (#339)
//   [P2] "Support speculative-decode verify on ROCm, and stop auto routing
//         short-query prefill to AITER" (#362)
#include "common.cuh"

namespace fi {
namespace {

constexpr int kDecodeThreads = 128;
constexpr int kDecodeStages = 3;   // cp.async ring depth
constexpr int kDecodeKT = 32;      // keys per stage

template <int D>
constexpr int decode_smem_bytes() {
  return kDecodeStages * kDecodeKT * D * 2 * 2;  // K and V rings, 16-bit elements
}

template <int D, int G, bool BF16>
__global__ void __launch_bounds__(kDecodeThreads, 4) decode_kernel(const AttnParams p) {
  using DT = Dt<BF16>;
  using T = typename DT::T;
  constexpr int LPK = D / 8;                 // lanes per key
  constexpr int KPS = 32 / LPK;              // keys per warp step
  constexpr int NWARP = kDecodeThreads / 32;
  constexpr int KPW = kDecodeKT / NWARP;     // keys per warp per stage
  constexpr int STEPS = KPW / KPS;           // warp steps per stage
  constexpr int CH = D / 8;                  // 16-byte chunks per row
  constexpr int STAGE = kDecodeKT * D;       // elements per stage

  extern __shared__ __align__(128) uint8_t dsmem[];
  T* sK = reinterpret_cast<T*>(dsmem);
  T* sV = sK + kDecodeStages * STAGE;
  __shared__ float sm_m[NWARP][G];
  __shared__ float sm_l[NWARP][G];
  // the warps' o partials reuse the ring once an item's keys are consumed
  float (*sm_o)[G][D] = reinterpret_cast<float (*)[G][D]>(dsmem);
  static_assert(NWARP * G * D * 4 <= kDecodeStages * kDecodeKT * D * 2 * 2, "o partials fit the ring");

  const WsHeader* hdr = static_cast<const WsHeader*>(p.ws);
  const int n_items = hdr->n_items;
  const WorkItem* items = ws_ptr<const WorkItem>(p.ws, hdr->off_items);
  const int32_t* qo_indptr = ws_ptr<const int32_t>(p.ws, hdr->off_qo_indptr);
  const int32_t* kv_indptr = ws_ptr<const int32_t>(p.ws, hdr->off_kv_indptr);
  const int32_t* kv_len = ws_ptr<const int32_t>(p.ws, hdr->off_kv_len);
  float* tmp_lse = ws_ptr<float>(p.ws, hdr->off_tmp_lse);
  float* tmp_o = ws_ptr<float>(p.ws, hdr->off_tmp_o);
  const int window_left = hdr->window_left;
  const int Hq = p.num_qo_heads;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int kg = lane / LPK;   // key within the warp step
  const int dl = lane % LPK;   // 8-element slice of the head dim

  for (int w = blockIdx.x; w < n_items; w += gridDim.x) {
    const WorkItem it = items[w];
    if (it.b < 0) continue;  // schedule padding
    const int b = it.b, hk = it.kv_head;
    const int lk = kv_len[b];
    const int token = qo_indptr[b];
    int lo = it.kv_begin;
    const int hi = min(it.kv_end, lk);
    if (window_left >= 0) lo = max(lo, lk - 1 - window_left);
    lo = max(lo, 0);
    const int n_tiles = hi > lo ? (hi - lo + kDecodeKT - 1) / kDecodeKT : 0;

    const int32_t* pages = p.kv_indices + kv_indptr[b];
    const T* kbase = static_cast<const T*>(p.k) + int64_t(hk) * p.k_stride_head;
    const T* vbase = static_cast<const T*>(p.v) + int64_t(hk) * p.v_stride_head;
    // gather one stage of K and V rows (16-byte cp.async, zero-fill past hi)
    // Thread t copies 16-byte chunk (t % CH) of rows t / CH + i * (128 / CH) of
    // every stage: K and V share the page lookup, and everything that does not
    // depend on the stage is computed once per item.
    constexpr int ROWS_PER_PASS = kDecodeThreads / CH;
    constexpr int PASSES = kDecodeKT / ROWS_PER_PASS;
    const int my_c = tid % CH, my_row = tid / CH;
    const T* kcol = kbase + my_c * 8;
    const T* vcol = vbase + my_c * 8;
    const uint32_t sk0 = smem_u32(sK + my_row * D + my_c * 8);
    const uint32_t sv0 = smem_u32(sV + my_row * D + my_c * 8);
    auto issue = [&](int tile, int stage) {
      const int kt = lo + tile * kDecodeKT + my_row;
#pragma unroll
      for (int i = 0; i < PASSES; ++i) {
        const int j = kt + i * ROWS_PER_PASS;
        const T* ks = static_cast<const T*>(p.k);
        const T* vs = static_cast<const T*>(p.v);
        int bytes = 0;
        if (j < hi) {
          int32_t pi, slot;
          if (p.page_shift >= 0) {
            pi = j >> p.page_shift;
            slot = j & ((1 << p.page_shift) - 1);
          } else {
            pi = j / p.page_size;
            slot = j - pi * p.page_size;
          }
          const int64_t page = __ldg(pages + pi);
          ks = kcol + page * p.k_stride_page + int64_t(slot) * p.k_stride_tok;
          vs = vcol + page * p.v_stride_page + int64_t(slot) * p.v_stride_tok;
          bytes = 16;
        }
        const uint32_t off = uint32_t((stage * STAGE + i * ROWS_PER_PASS * D) * 2);
        cp_async16(sk0 + off, ks, bytes);
        cp_async16(sv0 + off, vs, bytes);
      }
    };
#pragma unroll
    for (int s = 0; s < kDecodeStages - 1; ++s) {
      if (s < n_tiles) issue(s, s);
      cp_async_commit();
    }

    // After the reduce-scatter below, this lane holds the score of head
    // `myh` of its key; the running max / sum of that head live on the lanes
    // that own it, o (all heads, this lane's 8 dims) lives on every lane.
    int myh = 0;
    {
      int cnt = G;
#pragma unroll
      for (int off = LPK / 2; off >= 1; off >>= 1) {
        if (cnt > 1) {
          cnt >>= 1;
          if (lane & off) myh += cnt;
        }
      }
    }
    // q of every head in the group, pre-scaled into the log2 domain, as pairs
    // for the packed fp32x2 FMA. Slot s holds head (myh ^ s): at each level of
    // the reduce-scatter a lane then keeps its first half of the slots and
    // sends the second, with no per-lane selection.
    float2 q2[G][4];
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
    float m_me = neg_inf(), l_me = 0.f;
    float2 o2[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < 4; ++e) o2[h][e] = make_float2(0.f, 0.f);
    // lane (within this key's lane group) that holds head h's score
    int src_of[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      int l_in = 0, cnt = G, rem = h;
#pragma unroll
      for (int off = LPK / 2; off >= 1; off >>= 1) {
        if (cnt > 1) {
          cnt >>= 1;
          if (rem >= cnt) { l_in |= off; rem -= cnt; }
        }
      }
      src_of[h] = (lane & ~(LPK - 1)) | l_in;
    }

    for (int tile = 0; tile < n_tiles; ++tile) {
      cp_async_wait<kDecodeStages - 2>();
      __syncthreads();
      {
        const int nt = tile + kDecodeStages - 1;
        if (nt < n_tiles) issue(nt, nt % kDecodeStages);
        cp_async_commit();
      }
      const int st = tile % kDecodeStages;
      const int kt = lo + tile * kDecodeKT;
      const bool full_tile = kt + kDecodeKT <= hi;
      const T* cK = sK + st * STAGE;
      const T* cV = sV + st * STAGE;
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
        s[u] = (full_tile || kt + key < hi) ? part[0] : neg_inf();
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
        const uint4 vr = *reinterpret_cast<const uint4*>(cV + key * D + dl * 8);
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
    cp_async_wait<0>();
    __syncthreads();  // every warp is done with the ring before it holds o partials

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
        float4* dst = reinterpret_cast<float4*>(&sm_o[warp][h][dl * 8]);
        dst[0] = make_float4(o2[h][0].x, o2[h][0].y, o2[h][1].x, o2[h][1].y);
        dst[1] = make_float4(o2[h][2].x, o2[h][2].y, o2[h][3].x, o2[h][3].y);
      }
    }
    __syncthreads();

    // merge the warps and write: direct to out/lse, or to a partial slot
    const bool direct = it.chunk < 0;
    const int slot = direct ? 0 : it.partial_base + it.chunk;
    for (int idx = tid; idx < G * (D / 4); idx += kDecodeThreads) {
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
        const float4 ov = *reinterpret_cast<const float4*>(&sm_o[wq][h][c]);
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
    __syncthreads();
  }
}

template <int D, int G, bool BF16>
cudaError_t launch_dg(const AttnParams& p, int grid, cudaStream_t s) {
  auto k = decode_kernel<D, G, BF16>;
  // once per process, before any capture (no attribute call inside a captured run)
  static cudaError_t attr =
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, decode_smem_bytes<D>());
  if (attr != cudaSuccess) return attr;
  k<<<grid, kDecodeThreads, decode_smem_bytes<D>(), s>>>(p);
  return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_d(const AttnParams& p, int group, int grid, cudaStream_t s) {
  switch (group) {
    case 1: return launch_dg<D, 1, BF16>(p, grid, s);
    case 2: return launch_dg<D, 2, BF16>(p, grid, s);
    case 4: return launch_dg<D, 4, BF16>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode(const AttnParams& p, int head_dim, int group, bool bf16, int grid,
                          cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  if (head_dim == 128) return bf16 ? launch_d<128, true>(p, group, grid, stream)
                                   : launch_d<128, false>(p, group, grid, stream);
  if (head_dim == 64) return bf16 ? launch_d<64, true>(p, group, grid, stream)
                                  : launch_d<64, false>(p, group, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fi
