// Prefill / verify kernel on the warp-level tensor-core path (mma.sync
// m16n8k16, fp32 accumulate): the general kernel for any query length, used
// for speculative verify and short queries (M = 16 packed rows) and as the
// M = 64 prefill tile.
//
// A tile packs query rows and the GQA group: packed row r = query row * g +
// head in group, all heads of one kv head, so every K/V tile staged in shared
// memory serves g query heads. K/V rows are gathered page by page straight
// from the cache with cp.async (16-byte, XOR-swizzled
// shared memory, a 2-stage ring) - no contiguous copy of the cache is ever
// made.
//
// Mask [P1 "Why window_size_right stays -1"], [P2 "Summary"] for query row i
// and key j: (!causal || j <= i + Lk - Lq) && (wl < 0 || j + Lq + wl >= Lk + i).
// Tiles fully outside [window lower bound, causal upper bound] are never
// visited (the loop runs over the tile's live range only); the per-element
// test runs only on tiles that straddle a bound.
//   [P1] "Route non-causal windowed prefill to AITER's masked kernel" (#339)
//   [P2] "Support speculative-decode verify on ROCm, and stop auto routing
//         short-query prefill to AITER" (#362)
#include "common.cuh"

namespace fi {
namespace {

constexpr int kThreads = 128;
constexpr int kN = 64;  // keys per KV tile

template <int D, int WM>
struct MmaCfg {
  static constexpr int M = 16 * WM;        // packed rows per tile
  static constexpr int WN = 4 / WM;        // warps along keys
  static constexpr int NW = kN / WN;       // keys per warp per tile
  static constexpr int NT = NW / 8;        // n8 score tiles per warp
  static constexpr int KD = D / 16;        // k16 steps over the head dim
  static constexpr int CH = D / 8;         // 16-byte chunks per row
  static constexpr int Q_ELEMS = M * D;
  static constexpr int KV_ELEMS = kN * D;
  static constexpr int STAGES = 2;  // cp.async ring depth
  static constexpr int SMEM_BYTES = (Q_ELEMS + 2 * STAGES * KV_ELEMS) * 2;
};

// XOR swizzle of 16-byte chunks inside a row (conflict-free ldmatrix)
__device__ __forceinline__ int swz(int row, int chunk) { return chunk ^ (row & 7); }

template <int D, int WM, bool BF16>
__global__ void __launch_bounds__(kThreads) prefill_mma_kernel(const AttnParams p) {
  using C = MmaCfg<D, WM>;
  using DT = Dt<BF16>;
  using T = typename DT::T;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  T* sQ = reinterpret_cast<T*>(smem_raw);
  T* sK = sQ + C::Q_ELEMS;                 // [STAGES][kN][D]
  T* sV = sK + C::STAGES * C::KV_ELEMS;    // [STAGES][kN][D]

  const WsHeader* hdr = static_cast<const WsHeader*>(p.ws);
  if (hdr->index_error) return;  // the page table failed the index check: no work
  const int n_items = hdr->n_items;
  const WorkItem* items = ws_ptr<const WorkItem>(p.ws, hdr->off_items);
  const int32_t* qo_indptr = ws_ptr<const int32_t>(p.ws, hdr->off_qo_indptr);
  const int32_t* kv_indptr = ws_ptr<const int32_t>(p.ws, hdr->off_kv_indptr);
  const int32_t* kv_len = ws_ptr<const int32_t>(p.ws, hdr->off_kv_len);
  float* tmp_lse = ws_ptr<float>(p.ws, hdr->off_tmp_lse);
  float* tmp_o = ws_ptr<float>(p.ws, hdr->off_tmp_o);
  const int g = hdr->group;
  const int causal = hdr->causal;
  const int wl = hdr->window_left;
  const int tile_rows = hdr->tile_rows;
  const int Hq = p.num_qo_heads;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int wm = warp % WM;   // row group of this warp
  const int wn = warp / WM;   // key group of this warp
  const int qr = lane >> 2;   // fragment row (and +8)
  const int qc = lane & 3;    // fragment column pair

  for (int w = blockIdx.x; w < n_items; w += gridDim.x) {
    const WorkItem it = items[w];
    if (it.b < 0) continue;  // schedule padding
    const int b = it.b, hk = it.kv_head;
    const int token0 = qo_indptr[b];
    const int lq = qo_indptr[b + 1] - token0;
    const int lk = kv_len[b];
    const int n_rows = min(tile_rows, lq * g - it.row0);
    const int i0 = it.row0 / g;
    const int i1 = (it.row0 + n_rows) / g - 1;
    int hi_t = causal ? min(lk, i1 + lk - lq + 1) : lk;
    int lo_t = wl >= 0 ? max(0, lk - lq + i0 - wl) : 0;
    const int kv_lo = max(it.kv_begin, lo_t);
    const int kv_hi = min(it.kv_end, hi_t);
    const bool ragged = p.ragged != 0;
    const bool custom = p.custom_mask != nullptr;
    const int mask_base = custom ? ws_ptr<const int32_t>(p.ws, hdr->off_mask_indptr)[b] : 0;
    const int kv_start = kv_indptr[b];  // ragged: first row; paged: first page-table entry
    const int32_t* pages = ragged ? nullptr : p.kv_indices + kv_start;

    // ---- stage Q (packed rows) and the first K/V tile
    for (int idx = tid; idx < C::M * C::CH; idx += kThreads) {
      const int r = idx / C::CH, c = idx % C::CH;
      const T* src = static_cast<const T*>(p.q);
      int bytes = 0;
      if (r < n_rows) {
        const int pr = it.row0 + r;
        src += int64_t(token0 + pr / g) * p.q_stride_tok + int64_t(hk * g + pr % g) * p.q_stride_head + c * 8;
        bytes = 16;
      }
      cp_async16(smem_u32(sQ + r * D + swz(r, c) * 8), src, bytes);
    }
    auto load_kv = [&](int stage, int kt) {
      T* dk = sK + stage * C::KV_ELEMS;
      T* dv = sV + stage * C::KV_ELEMS;
      for (int idx = tid; idx < kN * C::CH; idx += kThreads) {
        const int r = idx / C::CH, c = idx % C::CH;
        const int j = kt + r;
        const T* ks = static_cast<const T*>(p.k);
        const T* vs = static_cast<const T*>(p.v);
        int bytes = 0;
        if (j < kv_hi) {
          ks += kv_row_offset(pages, j, p.page_size, p.page_shift, p.k_stride_page, p.k_stride_tok,
                              ragged, kv_start) +
                int64_t(hk) * p.k_stride_head + c * 8;
          vs += kv_row_offset(pages, j, p.page_size, p.page_shift, p.v_stride_page, p.v_stride_tok,
                              ragged, kv_start) +
                int64_t(hk) * p.v_stride_head + c * 8;
          bytes = 16;
        }
        cp_async16(smem_u32(dk + r * D + swz(r, c) * 8), ks, bytes);
        cp_async16(smem_u32(dv + r * D + swz(r, c) * 8), vs, bytes);
      }
    };
    const int n_kt = kv_lo < kv_hi ? (kv_hi - kv_lo + kN - 1) / kN : 0;
#pragma unroll
    for (int s = 0; s < C::STAGES - 1; ++s) {
      if (s < n_kt) load_kv(s, kv_lo + s * kN);
      cp_async_commit();  // group s (group 0 also carries Q)
    }
    cp_async_wait<C::STAGES - 2>();
    __syncthreads();

    uint32_t qa[C::KD][4];
#pragma unroll
    for (int kd = 0; kd < C::KD; ++kd) {
      const int r = wm * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
      const int c = kd * 2 + (lane >> 4);
      ldsm_x4(smem_u32(sQ + r * D + swz(r, c) * 8), qa[kd][0], qa[kd][1], qa[kd][2], qa[kd][3]);
    }

    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m[2] = {neg_inf(), neg_inf()};
    float l[2] = {0.f, 0.f};
    // query row of this thread's two fragment rows
    int qi[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) qi[hr] = (it.row0 + wm * 16 + qr + hr * 8) / g;

    for (int t = 0; t < n_kt; ++t) {
      const int kt = kv_lo + t * kN;
      cp_async_wait<C::STAGES - 2>();  // tile t has landed
      __syncthreads();                 // and every warp is done with tile t - 1
      {
        const int nt = t + C::STAGES - 1;
        if (nt < n_kt) load_kv(nt % C::STAGES, kv_lo + nt * kN);
        cp_async_commit();
      }
      const int stage = t % C::STAGES;
      const T* cK = sK + stage * C::KV_ELEMS;
      const T* cV = sV + stage * C::KV_ELEMS;

      // S = Q K^T over this warp's NW keys
      float s[C::NT][4];
#pragma unroll
      for (int nt = 0; nt < C::NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int kd = 0; kd < C::KD; ++kd) {
#pragma unroll
        for (int nt = 0; nt < C::NT; nt += 2) {
          const int r = wn * C::NW + nt * 8 + (lane & 7) + (lane >> 4) * 8;
          const int c = kd * 2 + ((lane >> 3) & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(smem_u32(cK + r * D + swz(r, c) * 8), b0, b1, b2, b3);
          mma16816<BF16>(s[nt], qa[kd], b0, b1);
          mma16816<BF16>(s[nt + 1], qa[kd], b2, b3);
        }
      }
      // scale into the log2 domain, mask boundary tiles
      const bool need_mask = (kt + kN > kv_hi) || custom ||
                             (causal && kt + kN - 1 > i0 + lk - lq) ||
                             (wl >= 0 && kt < lk - lq + i1 - wl);
#pragma unroll
      for (int nt = 0; nt < C::NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float x = s[nt][e] * p.sm_scale_log2;
          if (need_mask) {
            const int j = kt + wn * C::NW + nt * 8 + qc * 2 + (e & 1);
            const int i = qi[e >> 1];
            bool ok = j < kv_hi;
            if (causal && j > i + lk - lq) ok = false;
            if (wl >= 0 && j + lq + wl < lk + i) ok = false;
            // custom mask: read only for the tile's real rows (i < lq), whose
            // bits lie inside the request's segment
            if (custom && ok && (i >= lq || !custom_mask_bit(p.custom_mask, mask_base, i, j, lk)))
              ok = false;
            if (!ok) x = neg_inf();
          }
          s[nt][e] = x;
        }
      }
      // online softmax over the two fragment rows
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        float mx = neg_inf();
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt) mx = fmaxf(mx, fmaxf(s[nt][2 * hr], s[nt][2 * hr + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mn = fmaxf(m[hr], mx);
        const float mu = (mn == neg_inf()) ? 0.f : mn;
        const float corr = ex2(m[hr] - mu);
        m[hr] = mn;
        l[hr] *= corr;
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
          o[i][2 * hr] *= corr;
          o[i][2 * hr + 1] *= corr;
        }
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt) {
          const float p0 = ex2(s[nt][2 * hr] - mu);
          const float p1 = ex2(s[nt][2 * hr + 1] - mu);
          s[nt][2 * hr] = p0;
          s[nt][2 * hr + 1] = p1;
          l[hr] += p0 + p1;
        }
      }
      // O += P V
#pragma unroll
      for (int kk = 0; kk < C::NW / 16; ++kk) {
        uint32_t pa[4];
        pa[0] = DT::pack(s[2 * kk][0], s[2 * kk][1]);
        pa[1] = DT::pack(s[2 * kk][2], s[2 * kk][3]);
        pa[2] = DT::pack(s[2 * kk + 1][0], s[2 * kk + 1][1]);
        pa[3] = DT::pack(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
        for (int dn = 0; dn < D / 16; ++dn) {
          const int r = wn * C::NW + kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
          const int c = dn * 2 + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(smem_u32(cV + r * D + swz(r, c) * 8), b0, b1, b2, b3);
          mma16816<BF16>(o[2 * dn], pa, b0, b1);
          mma16816<BF16>(o[2 * dn + 1], pa, b2, b3);
        }
      }
    }
    cp_async_wait<0>();
    __syncthreads();

    // row sums across the quad
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      l[hr] += __shfl_xor_sync(0xffffffffu, l[hr], 1);
      l[hr] += __shfl_xor_sync(0xffffffffu, l[hr], 2);
    }

    if constexpr (C::WN > 1) {
      // warps hold the same rows over different keys: merge them in smem
      float* sm_o = reinterpret_cast<float*>(sK);            // [WN][16][D]
      float* sm_ml = sm_o + C::WN * 16 * D;                   // [WN][16][2]
#pragma unroll
      for (int i = 0; i < D / 8; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = qr + (e >> 1) * 8;
          const int c = i * 8 + qc * 2 + (e & 1);
          sm_o[(wn * 16 + r) * D + c] = o[i][e];
        }
      if (qc == 0) {
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          sm_ml[(wn * 16 + qr + hr * 8) * 2 + 0] = m[hr];
          sm_ml[(wn * 16 + qr + hr * 8) * 2 + 1] = l[hr];
        }
      }
      __syncthreads();
      // thread -> (row, 4-column group)
      for (int idx = tid; idx < 16 * (D / 4); idx += kThreads) {
        const int r = idx / (D / 4);
        const int c = (idx % (D / 4)) * 4;
        float M = neg_inf();
#pragma unroll
        for (int q = 0; q < C::WN; ++q) M = fmaxf(M, sm_ml[(q * 16 + r) * 2]);
        const float Mu = (M == neg_inf()) ? 0.f : M;
        float den = 0.f, a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int q = 0; q < C::WN; ++q) {
          const float sc = ex2(sm_ml[(q * 16 + r) * 2] - Mu);
          den += sc * sm_ml[(q * 16 + r) * 2 + 1];
          const float* src = sm_o + (q * 16 + r) * D + c;
          a0 += sc * src[0]; a1 += sc * src[1]; a2 += sc * src[2]; a3 += sc * src[3];
        }
        if (r >= n_rows) continue;
        const int pr = it.row0 + r;
        const int t = token0 + pr / g;
        const int head = hk * g + pr % g;
        const float inv = den > 0.f ? 1.f / den : 0.f;
        if (it.chunk < 0) {
          uint2 pk;
          pk.x = DT::pack(a0 * inv, a1 * inv);
          pk.y = DT::pack(a2 * inv, a3 * inv);
          *reinterpret_cast<uint2*>(static_cast<T*>(p.out) + (int64_t(t) * Hq + head) * D + c) = pk;
          if (c == 0 && p.lse) p.lse[int64_t(t) * Hq + head] = den > 0.f ? (M + __log2f(den)) * kLn2 : neg_inf();
        } else {
          const int slot = it.partial_base + (pr / g - i0) * it.num_chunks + it.chunk;
          *reinterpret_cast<float4*>(tmp_o + (int64_t(slot) * Hq + head) * D + c) =
              make_float4(a0 * inv, a1 * inv, a2 * inv, a3 * inv);
          if (c == 0) tmp_lse[int64_t(slot) * Hq + head] = den > 0.f ? (M + __log2f(den)) * kLn2 : neg_inf();
        }
      }
      __syncthreads();
    } else {
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int r = wm * 16 + qr + hr * 8;
        if (r >= n_rows) continue;
        const int pr = it.row0 + r;
        const int t = token0 + pr / g;
        const int head = hk * g + pr % g;
        const float inv = l[hr] > 0.f ? 1.f / l[hr] : 0.f;
        const float lse = l[hr] > 0.f ? (m[hr] + __log2f(l[hr])) * kLn2 : neg_inf();
        if (it.chunk < 0) {
          T* op = static_cast<T*>(p.out) + (int64_t(t) * Hq + head) * D + qc * 2;
#pragma unroll
          for (int i = 0; i < D / 8; ++i)
            *reinterpret_cast<uint32_t*>(op + i * 8) = DT::pack(o[i][2 * hr] * inv, o[i][2 * hr + 1] * inv);
          if (qc == 0 && p.lse) p.lse[int64_t(t) * Hq + head] = lse;
        } else {
          const int slot = it.partial_base + (pr / g - i0) * it.num_chunks + it.chunk;
          float* op = tmp_o + (int64_t(slot) * Hq + head) * D + qc * 2;
#pragma unroll
          for (int i = 0; i < D / 8; ++i)
            *reinterpret_cast<float2*>(op + i * 8) = make_float2(o[i][2 * hr] * inv, o[i][2 * hr + 1] * inv);
          if (qc == 0) tmp_lse[int64_t(slot) * Hq + head] = lse;
        }
      }
      __syncthreads();
    }
  }
}

template <int D, int WM, bool BF16>
cudaError_t launch_t(const AttnParams& p, int grid, cudaStream_t s) {
  using C = MmaCfg<D, WM>;
  auto k = prefill_mma_kernel<D, WM, BF16>;
  // once per device (not per launch, so a run() inside stream capture makes
  // no attribute call); the first run() on a device must precede any capture
  static std::atomic<uint64_t> done{0};
  const cudaError_t attr = smem_attr_once(k, C::SMEM_BYTES, done);
  if (attr != cudaSuccess) return attr;
  k<<<grid, kThreads, C::SMEM_BYTES, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_mma(const AttnParams& p, int head_dim, int kernel, bool bf16, int grid,
                               cudaStream_t s) {
  if (grid <= 0) return cudaSuccess;
  const bool m16 = kernel == kPrefillM16;
#define FI_DISPATCH(D)                                                              \
  if (head_dim == D) {                                                              \
    if (m16) return bf16 ? launch_t<D, 1, true>(p, grid, s) : launch_t<D, 1, false>(p, grid, s); \
    return bf16 ? launch_t<D, 4, true>(p, grid, s) : launch_t<D, 4, false>(p, grid, s); \
  }
  FI_DISPATCH(128)
  FI_DISPATCH(64)
#undef FI_DISPATCH
  return cudaErrorInvalidValue;
}

int kernel_ctas_per_sm(int kernel, int head_dim, int group, bool bf16, int page_size) {
  (void)bf16;
  switch (kernel) {
    case kDecode: return decode_ctas_per_sm(head_dim, page_size, group);
    case kPrefillM16: return head_dim == 128 ? 3 : 6;
    case kPrefillM64: return head_dim == 128 ? 2 : 4;
    case kPrefillM128: return 1;
  }
  return 1;
}


}  // namespace fi
