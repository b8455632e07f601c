// Merging attention states by their log-sum-exp ("Refuse attention inputs the
// ROCm kernels would compute wrongly" (#399), "Graph-mode partial_state
// merge"; split-KV in "Support speculative-decode verify on ROCm ..." (#362)):
//   m = max_i s_i,  s = m + ln sum_i exp(s_i - m),  o = sum_i exp(s_i - s) o_i,
// with every state at -inf giving o = 0, s = -inf. One warp per (row, head),
// the head dim spread over the lanes with 16-byte accesses. A device-side row
// count bounds the rows touched, so a graph replayed after a smaller re-plan
// writes nothing past its outputs.
#include "common.cuh"

namespace fi {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

template <int OUT>  // 0 f16, 1 bf16, 2 f32
__device__ __forceinline__ void store4(void* base, int64_t idx, float a, float b, float c,
                                       float d) {
  if constexpr (OUT == 2) {
    *reinterpret_cast<float4*>(static_cast<float*>(base) + idx) = make_float4(a, b, c, d);
  } else {
    using DT = Dt<OUT == 1>;
    uint2 pk;
    pk.x = DT::pack(a, b);
    pk.y = DT::pack(c, d);
    *reinterpret_cast<uint2*>(static_cast<typename DT::T*>(base) + idx) = pk;
  }
}

template <int OUT>
__device__ __forceinline__ float4 load4(const void* base, int64_t idx) {
  if constexpr (OUT == 2) {
    return *reinterpret_cast<const float4*>(static_cast<const float*>(base) + idx);
  } else {
    using DT = Dt<OUT == 1>;
    const uint2 w = *reinterpret_cast<const uint2*>(static_cast<const typename DT::T*>(base) + idx);
    return make_float4(DT::lo(w.x), DT::hi(w.x), DT::lo(w.y), DT::hi(w.y));
  }
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Merge states [beg, end) of v [n, H, D] / s [n, H] for one (row, head) into
// (v_out + out_off, s_out). D is a multiple of 4; lane handles 4-wide columns.
// The scores and value columns of the first kMB states are loaded together
// before any arithmetic, and later states kMB at a time, so a row costs about
// one memory round trip per kMB states rather than one per state and pass.
constexpr int kMB = 6;

template <int OUT>
__device__ void merge_one(const float* __restrict__ v, const float* __restrict__ s, int beg,
                          int end, int H, int D, int h, void* v_out, int64_t out_off,
                          float* s_out, int64_t s_off, int lane) {
  const int n = end - beg;
  const int c0 = lane * 4;
  float s0[kMB];
  float4 x0[kMB];
#pragma unroll
  for (int k = 0; k < kMB; ++k) {
    const bool live = k < n;
    s0[k] = live ? __ldg(s + int64_t(beg + k) * H + h) : neg_inf();
    x0[k] = (live && c0 < D)
                ? *reinterpret_cast<const float4*>(v + (int64_t(beg + k) * H + h) * D + c0)
                : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float m = s0[0];
#pragma unroll
  for (int k = 1; k < kMB; ++k) m = fmaxf(m, s0[k]);
  if (n > kMB) {  // warp-uniform: the remaining scores, spread over the lanes
    float mr = neg_inf();
    for (int i = beg + kMB + lane; i < end; i += 32) mr = fmaxf(mr, __ldg(s + int64_t(i) * H + h));
    m = fmaxf(m, warp_max(mr));
  }
  const float mu = (m == neg_inf()) ? 0.f : m;
  float w0[kMB];
  float den = 0.f;
#pragma unroll
  for (int k = 0; k < kMB; ++k) {
    w0[k] = ex2((s0[k] - mu) * kLog2e);
    den += w0[k];
  }
  if (n > kMB) {
    float dr = 0.f;
    for (int i = beg + kMB + lane; i < end; i += 32)
      dr += ex2((__ldg(s + int64_t(i) * H + h) - mu) * kLog2e);
    den += warp_sum(dr);
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  for (int c = c0; c < D; c += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int i = beg;
    if (c == c0) {  // the first states' columns are already in registers
#pragma unroll
      for (int k = 0; k < kMB; ++k) {
        const float w = w0[k] * inv;
        acc.x += w * x0[k].x; acc.y += w * x0[k].y; acc.z += w * x0[k].z; acc.w += w * x0[k].w;
      }
      i = beg + kMB;
    }
    for (; i < end; i += kMB) {
      float sk[kMB];
      float4 xk[kMB];
#pragma unroll
      for (int k = 0; k < kMB; ++k) {
        const bool live = i + k < end;
        sk[k] = live ? __ldg(s + int64_t(i + k) * H + h) : neg_inf();
        xk[k] = live ? *reinterpret_cast<const float4*>(v + (int64_t(i + k) * H + h) * D + c)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < kMB; ++k) {
        const float w = ex2((sk[k] - mu) * kLog2e) * inv;
        acc.x += w * xk[k].x; acc.y += w * xk[k].y; acc.z += w * xk[k].z; acc.w += w * xk[k].w;
      }
    }
    store4<OUT>(v_out, out_off + c, acc.x, acc.y, acc.z, acc.w);
  }
  if (lane == 0 && s_out) s_out[s_off] = den > 0.f ? m + logf(den) : neg_inf();
}

// Workspace partials of a plan -> out / lse (rows listed in merge_rows).
template <int OUT>
__global__ void __launch_bounds__(256, 4) merge_workspace_kernel(const void* ws, void* out,
                                                                 float* lse, int H, int D) {
  // The plan's metadata (header, merge rows, merge_indptr) was copied in
  // before the attention kernel started, so the first task's bounds are read
  // while that kernel is still running.
  const WsHeader* hdr = static_cast<const WsHeader*>(ws);
  if (hdr->index_error) return;  // the page table failed the index check: no work
  const int n_rows = hdr->n_merge_rows;
  const int32_t* merge_indptr = ws_ptr<const int32_t>(ws, hdr->off_merge_indptr);
  const int32_t* merge_rows = ws_ptr<const int32_t>(ws, hdr->off_merge_rows);
  const float* tmp_lse = ws_ptr<const float>(ws, hdr->off_tmp_lse);
  const float* tmp_o = ws_ptr<const float>(ws, hdr->off_tmp_o);
  const int lane = threadIdx.x & 31;
  const int64_t total = int64_t(n_rows) * H;
  const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
  int64_t wi = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int t = 0, beg = 0, end = 0;
  if (wi < total) {
    t = merge_rows[wi / H];
    beg = merge_indptr[t];
    end = merge_indptr[t + 1];
  }
  // launched as a programmatic dependent of the attention kernel: its launch
  // overlaps that kernel's tail, and this wait makes the partials visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (; wi < total; wi += warps) {
    const int h = int(wi % H);
    merge_one<OUT>(tmp_o, tmp_lse, beg, end, H, D, h, out, (int64_t(t) * H + h) * D, lse,
                   int64_t(t) * H + h, lane);
    const int64_t nx = wi + warps;
    if (nx < total) {
      t = merge_rows[nx / H];
      beg = merge_indptr[t];
      end = merge_indptr[t + 1];
    }
  }
}

// Caller tensors: row r merges states merge_indptr[r] .. merge_indptr[r+1]-1.
template <int OUT>
__global__ void __launch_bounds__(256) merge_states_kernel(const float* v, const float* s,
                                                           const int32_t* merge_indptr, int rows,
                                                           const int32_t* rows_dev, int H, int D,
                                                           void* v_out, float* s_out) {
  int n = rows;
  if (rows_dev) n = min(n, *rows_dev);
  const int lane = threadIdx.x & 31;
  const int64_t total = int64_t(max(n, 0)) * H;
  const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
  for (int64_t wi = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); wi < total;
       wi += warps) {
    const int r = int(wi / H), h = int(wi % H);
    merge_one<OUT>(v, s, merge_indptr[r], merge_indptr[r + 1], H, D, h, v_out,
                   (int64_t(r) * H + h) * D, s_out, int64_t(r) * H + h, lane);
  }
}

// Two states, strided inputs, packed outputs (may alias input a).
template <int DT_>
__global__ void __launch_bounds__(256) merge_two_kernel(const MergeTwoParams p) {
  int n = p.rows;
  if (p.num_rows_dev) n = min(n, *p.num_rows_dev);
  const int lane = threadIdx.x & 31;
  const int H = p.heads, D = p.head_dim;
  const int64_t total = int64_t(max(n, 0)) * H;
  const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
  for (int64_t wi = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); wi < total;
       wi += warps) {
    const int r = int(wi / H), h = int(wi % H);
    const float sa = p.sa[int64_t(r) * p.sa_sr + h];
    const float sb = p.sb[int64_t(r) * p.sb_sr + h];
    const float m = fmaxf(sa, sb);
    const float mu = (m == neg_inf()) ? 0.f : m;
    const float ea = ex2((sa - mu) * kLog2e), eb = ex2((sb - mu) * kLog2e);
    const float den = ea + eb;
    const float wa = den > 0.f ? ea / den : 0.f, wb = den > 0.f ? eb / den : 0.f;
    const int64_t oa = int64_t(r) * p.va_sr + int64_t(h) * p.va_sh;
    const int64_t ob = int64_t(r) * p.vb_sr + int64_t(h) * p.vb_sh;
    const int64_t oo = (int64_t(r) * H + h) * D;
    for (int c = lane; c < D; c += 32) {
      float xa, xb;
      if constexpr (DT_ == 2) {
        xa = static_cast<const float*>(p.va)[oa + c];
        xb = static_cast<const float*>(p.vb)[ob + c];
        static_cast<float*>(p.vo)[oo + c] = wa * xa + wb * xb;
      } else {
        using DT = Dt<DT_ == 1>;
        using T = typename DT::T;
        const uint32_t ra = static_cast<const unsigned short*>(p.va)[oa + c];
        const uint32_t rb = static_cast<const unsigned short*>(p.vb)[ob + c];
        xa = DT::lo(ra);
        xb = DT::lo(rb);
        static_cast<T*>(p.vo)[oo + c] = DT::from_float(wa * xa + wb * xb);
      }
    }
    __syncwarp();
    if (lane == 0) p.so[int64_t(r) * H + h] = den > 0.f ? m + logf(den) : neg_inf();
  }
}

int merge_grid(int64_t warps_needed) {
  int64_t blocks = (warps_needed + 7) / 8;
  if (blocks > 152 * 8) blocks = 152 * 8;
  return blocks < 1 ? 1 : int(blocks);
}

}  // namespace

cudaError_t launch_merge_workspace(const void* ws, void* out, float* lse, int H, int D,
                                   bool bf16, int grid, cudaStream_t s) {
  // programmatic dependent launch on the attention kernel before it in the
  // stream (also inside a captured graph)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = bf16 ? cudaLaunchKernelEx(&cfg, merge_workspace_kernel<1>, ws, out, lse, H, D)
                       : cudaLaunchKernelEx(&cfg, merge_workspace_kernel<0>, ws, out, lse, H, D);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_merge_states(const float* v, const float* s, const int32_t* merge_indptr,
                                int32_t rows, int H, int D, void* v_out, int out_dtype,
                                float* s_out, const int32_t* rows_dev, cudaStream_t st) {
  const int grid = merge_grid(int64_t(rows) * H);
  switch (out_dtype) {
    case 0: merge_states_kernel<0><<<grid, 256, 0, st>>>(v, s, merge_indptr, rows, rows_dev, H, D, v_out, s_out); break;
    case 1: merge_states_kernel<1><<<grid, 256, 0, st>>>(v, s, merge_indptr, rows, rows_dev, H, D, v_out, s_out); break;
    case 2: merge_states_kernel<2><<<grid, 256, 0, st>>>(v, s, merge_indptr, rows, rows_dev, H, D, v_out, s_out); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_merge_two(const MergeTwoParams& p, cudaStream_t st) {
  const int grid = merge_grid(int64_t(p.rows) * p.heads);
  switch (p.dtype) {
    case 0: merge_two_kernel<0><<<grid, 256, 0, st>>>(p); break;
    case 1: merge_two_kernel<1><<<grid, 256, 0, st>>>(p); break;
    case 2: merge_two_kernel<2><<<grid, 256, 0, st>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace fi
