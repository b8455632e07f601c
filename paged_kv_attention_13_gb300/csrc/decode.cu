// Decode kernel: one query row per request against its paged KV, all G query
// heads of one kv head together (GQA). Bandwidth-bound: every K/V byte is
// read exactly once, with 16-byte coalesced cp.async gathers,
// scores reduced with warp shuffles, and an online softmax kept in fp32.
//
// Work item = (request, kv head, key chunk). A CTA of 4 warps streams the
// chunk's live keys through a 4-stage cp.async ring in shared memory (32 keys
// of K and V per stage, gathered page by page, zero-filled past the end), so
// three stages of loads stay in flight while one is consumed. Each warp takes
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
constexpr int kDecodeStages = 4;   // cp.async ring depth
constexpr int kDecodeKT = 32;      // keys per stage

template <int D>
constexpr int decode_smem_bytes() {
  return kDecodeStages * kDecodeKT * D * 2 * 2;  // K and V rings, 16-bit elements
}

template <int D, int G, bool BF16>
__global__ void __launch_bounds__(kDecodeThreads, 3) decode_kernel(const AttnParams p) {
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
  __shared__ __align__(16) float sm_o[NWARP][G][D];

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
    auto issue = [&](int tile, int stage) {
      const int kt = lo + tile * kDecodeKT;
      for (int idx = tid; idx < kDecodeKT * CH; idx += kDecodeThreads) {
        const int key = idx / CH, c = idx % CH;
        const int j = kt + key;
        const T* ks = static_cast<const T*>(p.k);
        const T* vs = static_cast<const T*>(p.v);
        int bytes = 0;
        if (j < hi) {
          ks = kbase + kv_row_offset(pages, j, p.page_size, p.page_shift, p.k_stride_page,
                                     p.k_stride_tok) + c * 8;
          vs = vbase + kv_row_offset(pages, j, p.page_size, p.page_shift, p.v_stride_page,
                                     p.v_stride_tok) + c * 8;
          bytes = 16;
        }
        cp_async16(smem_u32(sK + stage * STAGE + key * D + c * 8), ks, bytes);
        cp_async16(smem_u32(sV + stage * STAGE + key * D + c * 8), vs, bytes);
      }
    };
#pragma unroll
    for (int s = 0; s < kDecodeStages - 1; ++s) {
      if (s < n_tiles) issue(s, s);
      cp_async_commit();
    }

    // q slice of every head in the group, pre-scaled into the log2 domain
    float qf[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const T* qp = static_cast<const T*>(p.q) + int64_t(token) * p.q_stride_tok +
                    int64_t(hk * G + h) * p.q_stride_head + dl * 8;
      uint4 r = ld_nc16(qp);
      const uint32_t wv[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        qf[h][2 * e] = DT::lo(wv[e]) * p.sm_scale_log2;
        qf[h][2 * e + 1] = DT::hi(wv[e]) * p.sm_scale_log2;
      }
    }
    float m[G], l[G], o[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = neg_inf();
      l[h] = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) o[h][e] = 0.f;
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
      const T* cK = sK + st * STAGE;
      const T* cV = sV + st * STAGE;
      float s[STEPS][G];
#pragma unroll
      for (int u = 0; u < STEPS; ++u) {
        const int key = warp * KPW + u * KPS + kg;
        const uint4 kr = *reinterpret_cast<const uint4*>(cK + key * D + dl * 8);
        const uint32_t wv[4] = {kr.x, kr.y, kr.z, kr.w};
        float kf[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          kf[2 * e] = DT::lo(wv[e]);
          kf[2 * e + 1] = DT::hi(wv[e]);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float acc = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) acc = fmaf(qf[h][e], kf[e], acc);
          s[u][h] = acc;
        }
      }
#pragma unroll
      for (int off = LPK / 2; off >= 1; off >>= 1)
#pragma unroll
        for (int u = 0; u < STEPS; ++u)
#pragma unroll
          for (int h = 0; h < G; ++h) s[u][h] += __shfl_xor_sync(0xffffffffu, s[u][h], off);
      float mx[G];
#pragma unroll
      for (int h = 0; h < G; ++h) mx[h] = neg_inf();
#pragma unroll
      for (int u = 0; u < STEPS; ++u) {
        const bool in = (kt + warp * KPW + u * KPS + kg) < hi;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          if (!in) s[u][h] = neg_inf();
          mx[h] = fmaxf(mx[h], s[u][h]);
        }
      }
#pragma unroll
      for (int off = LPK; off < 32; off <<= 1)
#pragma unroll
        for (int h = 0; h < G; ++h) mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], off));
      float pm[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float mn = fmaxf(m[h], mx[h]);
        const float mu = (mn == neg_inf()) ? 0.f : mn;
        const float corr = ex2(m[h] - mu);
        m[h] = mn;
        pm[h] = mu;
        l[h] *= corr;
#pragma unroll
        for (int e = 0; e < 8; ++e) o[h][e] *= corr;
      }
#pragma unroll
      for (int u = 0; u < STEPS; ++u) {
        const int key = warp * KPW + u * KPS + kg;
        const uint4 vr = *reinterpret_cast<const uint4*>(cV + key * D + dl * 8);
        const uint32_t wv[4] = {vr.x, vr.y, vr.z, vr.w};
        float vf[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          vf[2 * e] = DT::lo(wv[e]);
          vf[2 * e + 1] = DT::hi(wv[e]);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float pr = ex2(s[u][h] - pm[h]);
          l[h] += pr;
#pragma unroll
          for (int e = 0; e < 8; ++e) o[h][e] = fmaf(pr, vf[e], o[h][e]);
        }
      }
    }
    cp_async_wait<0>();

    // the warp's key groups share m; sum their l and o
#pragma unroll
    for (int off = LPK; off < 32; off <<= 1) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], off);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[h][e] += __shfl_xor_sync(0xffffffffu, o[h][e], off);
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        sm_m[warp][h] = m[h];
        sm_l[warp][h] = l[h];
      }
    }
    if (kg == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float4* dst = reinterpret_cast<float4*>(&sm_o[warp][h][dl * 8]);
        dst[0] = make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
        dst[1] = make_float4(o[h][4], o[h][5], o[h][6], o[h][7]);
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
