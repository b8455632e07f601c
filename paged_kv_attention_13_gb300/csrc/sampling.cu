// Chain speculative-sampling acceptance step: the sampler the multi-token
// verify pass feeds ("Support speculative-decode verify on ROCm, and stop
// auto routing short-query prefill to AITER" (#362), "Summary";
// "Architecture / design notes": chain_speculative_sampling takes
// (batch_size, num_speculate_tokens), a chain). The pages give no formula;
// the steps are the published speculative sampling (Leviathan, Kalman and
// Matias 2023; Chen et al. 2023):
//   draft i (token x_i) is accepted while u_i * q_i(x_i) <= p_i(x_i)
//   (product and compare in fp32); at the first rejection i one token is
//   drawn from max(0, p_i - q_i) (fp32 differences; p_i itself when that is
//   all zero), or from p_n when every draft is accepted; a draw with uniform
//   u takes the smallest token whose cumulative weight exceeds u * total,
//   the weights summed in fp64.
//
// Four CTAs per request, one thread-block cluster: each runs the n acceptance
// tests (warp 0, a ballot finds the first rejection), then streams its quarter
// of the drawn row in blocks of 128 tokens, dealt round-robin to its warps
// (one coalesced 16-byte load per lane per block, eight blocks in flight per
// warp), summing each block's weight in fp32 into shared memory, and its
// quarter's total in fp64 (after a rejection, p's own block sums come from the
// same pass, for the all-zero-residual fallback). After a cluster barrier
// every CTA reads the four totals through distributed shared memory and finds
// the quarter that holds u * total; the CTA that owns it scans its block sums
// (fp64), re-reads the one block that holds the target and writes the
// outputs. The kernel is bound by the one or two rows of V floats it reads
// per request. (Weights are
// summed in fp32 inside a 128-token block and in fp64 across blocks, so a
// draw within about 1e-6 of a cumulative boundary may land on the
// neighbouring token of an all-fp64 sum.)
#include <cooperative_groups.h>

#include "common.cuh"

namespace fi {
namespace {

namespace cg = cooperative_groups;

constexpr int kSlices = 4;  // CTAs (one cluster) per request
constexpr int kSampThreads = 512;
constexpr int kSampWarps = kSampThreads / 32;
constexpr int kBlk = 128;  // tokens per block sum

// This lane's four weights of block blk: tokens blk * 128 + lane * 4 + k,
// p or max(0, p - q) (fp32), 0 past the end.
__device__ __forceinline__ float4 lane_weights(const float* p, const float* q, int blk, int lane,
                                               int V, bool vec) {
  const int t = blk * kBlk + lane * 4;
  float4 a, c = make_float4(0.f, 0.f, 0.f, 0.f);
  if (vec && t + 4 <= V) {
    a = __ldg(reinterpret_cast<const float4*>(p + t));
    if (q) c = __ldg(reinterpret_cast<const float4*>(q + t));
  } else {
    a.x = t < V ? __ldg(p + t) : 0.f;
    a.y = t + 1 < V ? __ldg(p + t + 1) : 0.f;
    a.z = t + 2 < V ? __ldg(p + t + 2) : 0.f;
    a.w = t + 3 < V ? __ldg(p + t + 3) : 0.f;
    if (q) {
      c.x = t < V ? __ldg(q + t) : 0.f;
      c.y = t + 1 < V ? __ldg(q + t + 1) : 0.f;
      c.z = t + 2 < V ? __ldg(q + t + 2) : 0.f;
      c.w = t + 3 < V ? __ldg(q + t + 3) : 0.f;
    }
  }
  if (q) {
    a.x = fmaxf(0.f, __fsub_rn(a.x, c.x));
    a.y = fmaxf(0.f, __fsub_rn(a.y, c.y));
    a.z = fmaxf(0.f, __fsub_rn(a.z, c.z));
    a.w = fmaxf(0.f, __fsub_rn(a.w, c.w));
  }
  return a;
}

__device__ __forceinline__ float lane_sum(const float4 w) {
  return __fadd_rn(__fadd_rn(__fadd_rn(w.x, w.y), w.z), w.w);
}

// Block sums of the row into bsum[0 .. nb) (all warps; the caller
// synchronises). Warp w owns blocks w, w + 16, w + 32, ...; it loads kUnroll
// of them before reducing any, so that many 16-byte loads per lane are in
// flight (one at a time left the kernel waiting on memory latency).
constexpr int kUnroll = 8;

// Sums of blocks [b0, b1) into bsum[blk - b0] (all warps; the caller
// synchronises). Warp w owns blocks b0 + w, b0 + w + 16, ...; it loads
// kUnroll of them before reducing any, so that many 16-byte loads per lane
// are in flight.
__device__ void block_sums(const float* p, const float* q, int V, bool vec, int b0, int b1,
                           float* bsum, int warp, int lane) {
  for (int blk0 = b0 + warp; blk0 < b1; blk0 += kSampWarps * kUnroll) {
    float4 w[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int blk = blk0 + u * kSampWarps;
      w[u] = blk < b1 ? lane_weights(p, q, blk, lane, V, vec) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float s = lane_sum(w[u]);
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, off));
      const int blk = blk0 + u * kSampWarps;
      if (lane == 0 && blk < b1) bsum[blk - b0] = s;
    }
  }
}

// The residual's block sums into bsum and p's into bsum_p, in one pass over
// p and q (same arithmetic, in the same order, as block_sums of each); half
// the unroll, since each block brings two rows' loads.
constexpr int kUnroll2 = kUnroll / 2;
__device__ void block_sums_both(const float* p, const float* q, int V, bool vec, int b0, int b1,
                                float* bsum, float* bsum_p, int warp, int lane) {
  for (int blk0 = b0 + warp; blk0 < b1; blk0 += kSampWarps * kUnroll2) {
    float4 a[kUnroll2], c[kUnroll2];
#pragma unroll
    for (int u = 0; u < kUnroll2; ++u) {
      const int blk = blk0 + u * kSampWarps;
      a[u] = blk < b1 ? lane_weights(p, nullptr, blk, lane, V, vec) : make_float4(0.f, 0.f, 0.f, 0.f);
      c[u] = blk < b1 ? lane_weights(q, nullptr, blk, lane, V, vec) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kUnroll2; ++u) {
      const float4 r = make_float4(fmaxf(0.f, __fsub_rn(a[u].x, c[u].x)), fmaxf(0.f, __fsub_rn(a[u].y, c[u].y)),
                                   fmaxf(0.f, __fsub_rn(a[u].z, c[u].z)), fmaxf(0.f, __fsub_rn(a[u].w, c[u].w)));
      float s = lane_sum(r), sp = lane_sum(a[u]);
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, off));
        sp = __fadd_rn(sp, __shfl_xor_sync(0xffffffffu, sp, off));
      }
      const int blk = blk0 + u * kSampWarps;
      if (lane == 0 && blk < b1) {
        bsum[blk - b0] = s;
        bsum_p[blk - b0] = sp;
      }
    }
  }
}

// fp64 total of n fp32 values (one warp).
__device__ double warp_total(const float* v, int n, int lane) {
  double t = 0.0;
  for (int k = lane; k < n; k += 32) t += double(v[k]);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
  return t;
}

__global__ void __cluster_dims__(kSlices, 1, 1) __launch_bounds__(kSampThreads, 2)
    chain_spec_kernel(const SpecParams sp) {
  extern __shared__ float bsum[];  // this CTA's block sums (drawn row, then p alone)
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = int(cluster.block_rank());
  const int b = blockIdx.x / kSlices;  // the request
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = sp.n, V = sp.vocab;
  const int nb = (V + kBlk - 1) / kBlk;
  // this CTA's quarter of the blocks
  const int b0 = int(int64_t(nb) * rank / kSlices), b1 = int(int64_t(nb) * (rank + 1) / kSlices);
  const int mb = b1 - b0;
  float* bsum_p = bsum + mb;  // p alone, for the all-zero-residual fallback
  __shared__ int s_acc, s_token;
  __shared__ double s_tot[2];  // this quarter's totals: drawn row, p alone

  // 1. acceptance tests, 32 drafts per ballot (every CTA of the cluster)
  if (warp == 0) {
    int acc = n;
    for (int i0 = 0; i0 < n; i0 += 32) {
      const int i = i0 + lane;
      bool ok = true;
      if (i < n) {
        const int x = sp.draft_ids[int64_t(b) * sp.ids_sb + i];
        const float q = __ldg(sp.draft_probs + int64_t(b) * sp.dp_sb + int64_t(i) * sp.dp_si + x);
        const float p = __ldg(sp.target_probs + int64_t(b) * sp.tp_sb + int64_t(i) * sp.tp_si + x);
        const float u = __ldg(sp.u_accept + int64_t(b) * sp.ua_sb + i);
        ok = __fmul_rn(u, q) <= p;
      }
      const unsigned rej = __ballot_sync(0xffffffffu, !ok);
      if (rej) {
        acc = i0 + __ffs(rej) - 1;
        break;
      }
    }
    if (lane == 0) s_acc = acc;
  }
  __syncthreads();
  const int acc = s_acc;

  // 2. block sums of this quarter: the residual at the first rejection (and
  // p alone), or p_n
  const float* p = sp.target_probs + int64_t(b) * sp.tp_sb + int64_t(acc) * sp.tp_si;
  const float* q = acc < n ? sp.draft_probs + int64_t(b) * sp.dp_sb + int64_t(acc) * sp.dp_si
                           : nullptr;
  const bool vec = (reinterpret_cast<uintptr_t>(p) % 16 == 0) &&
                   (!q || reinterpret_cast<uintptr_t>(q) % 16 == 0);
  if (q) block_sums_both(p, q, V, vec, b0, b1, bsum, bsum_p, warp, lane);
  else block_sums(p, nullptr, V, vec, b0, b1, bsum, warp, lane);
  __syncthreads();
  if (warp == 0) {
    const double t0 = warp_total(bsum, mb, lane);
    const double t1 = q ? warp_total(bsum_p, mb, lane) : t0;
    if (lane == 0) {
      s_tot[0] = t0;
      s_tot[1] = t1;
      s_token = -1;
    }
  }
  cluster.sync();  // every quarter's totals are in its shared memory

  // 3. the quarter that holds u * total (same answer in every CTA)
  double tot[kSlices][2];
#pragma unroll
  for (int r = 0; r < kSlices; ++r) {
    const double* rt = cluster.map_shared_rank(s_tot, r);
    tot[r][0] = rt[0];
    tot[r][1] = rt[1];
  }
  cluster.sync();  // no CTA leaves while another still reads its totals
  double all0 = 0.0, all1 = 0.0;
#pragma unroll
  for (int r = 0; r < kSlices; ++r) {
    all0 += tot[r][0];
    all1 += tot[r][1];
  }
  const bool use_p = q && !(all0 > 0.0);  // an all-zero residual: draw from p itself
  const int which = use_p ? 1 : 0;
  const double total = use_p ? all1 : all0;
  const double target = double(__ldg(sp.u_sample + b)) * total;
  int owner = -1, last = -1;
  double run = 0.0, owner_start = 0.0, last_start = 0.0;
#pragma unroll
  for (int r = 0; r < kSlices; ++r) {
    if (tot[r][which] > 0.0) {
      last = r;
      last_start = run;
    }
    if (owner < 0 && run + tot[r][which] > target) {
      owner = r;
      owner_start = run;
    }
    run += tot[r][which];
  }
  if (owner < 0) {  // rounding put the target past the end: the last positive quarter
    owner = last;
    owner_start = last_start;
  }
  const int writer = owner >= 0 ? owner : 0;  // with no weight at all, rank 0 writes -1
  if (rank != writer) return;

  // 4. the owner: the block (fp64 scan of its block sums), then the token
  if (warp == 0 && owner >= 0) {
    const float* bs = use_p ? bsum_p : bsum;
    const float* qq = use_p ? nullptr : q;
    double run_b = owner_start;  // cumulative weight before block k0
    int blk = -1, last_blk = -1;
    double blk_start = 0.0, lb_start = 0.0;
    for (int k0 = 0; k0 < mb && blk < 0; k0 += 32) {
      const double v = k0 + lane < mb ? double(bs[k0 + lane]) : 0.0;
      double c = v;  // inclusive scan over the lanes
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, c, off);
        if (lane >= off) c += y;
      }
      const unsigned pos = __ballot_sync(0xffffffffu, v > 0.0);
      if (pos) {
        const int l = 31 - __clz(pos);
        last_blk = b0 + k0 + l;
        lb_start = run_b + __shfl_sync(0xffffffffu, c - v, l);
      }
      const unsigned hit = __ballot_sync(0xffffffffu, k0 + lane < mb && run_b + c > target);
      if (hit) {
        const int l = __ffs(hit) - 1;
        blk = b0 + k0 + l;
        blk_start = run_b + __shfl_sync(0xffffffffu, c - v, l);
      }
      run_b += __shfl_sync(0xffffffffu, c, 31);
    }
    if (blk < 0) {
      blk = last_blk;
      blk_start = lb_start;
    }
    int token = -1;
    if (blk >= 0) {
      const float4 w = lane_weights(p, qq, blk, lane, V, vec);
      const double ls = double(lane_sum(w));
      double c = ls;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, c, off);
        if (lane >= off) c += y;
      }
      // this lane's tokens: the first whose cumulative weight exceeds the target
      double cum = blk_start + (c - ls);
      const float wk[4] = {w.x, w.y, w.z, w.w};
      int mine = -1, mine_last = -1;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        cum += double(wk[k]);
        if (wk[k] > 0.f) mine_last = blk * kBlk + lane * 4 + k;
        if (mine < 0 && cum > target) mine = blk * kBlk + lane * 4 + k;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, mine >= 0);
      const unsigned pos = __ballot_sync(0xffffffffu, mine_last >= 0);
      if (hit) token = __shfl_sync(0xffffffffu, mine, __ffs(hit) - 1);
      else if (pos) token = __shfl_sync(0xffffffffu, mine_last, 31 - __clz(pos));
    }
    if (lane == 0) s_token = token;
  }
  __syncthreads();

  // 5. outputs: accepted drafts, the drawn token, then -1
  int32_t* out = sp.out_tokens + int64_t(b) * (n + 1);
  for (int i = tid; i <= n; i += kSampThreads) {
    int32_t v = -1;
    if (i < acc) v = sp.draft_ids[int64_t(b) * sp.ids_sb + i];
    else if (i == acc) v = s_token;
    out[i] = v;
  }
  if (tid == 0) {
    sp.out_accepted[b] = acc;
    if (sp.out_emitted) sp.out_emitted[b] = acc + 1;
  }
}

}  // namespace

// two arrays of block sums for a quarter of the blocks in 48 KB
int chain_spec_max_vocab() { return (48 * 1024 / 8 - 1) * kSlices * kBlk; }

cudaError_t launch_chain_spec_sampling(const SpecParams& sp, int batch, cudaStream_t stream) {
  if (batch <= 0) return cudaSuccess;
  const int nb = (sp.vocab + kBlk - 1) / kBlk;
  const int mb = (nb + kSlices - 1) / kSlices + 1;
  chain_spec_kernel<<<batch * kSlices, kSampThreads, size_t(2 * mb) * sizeof(float), stream>>>(sp);
  return cudaGetLastError();
}

}  // namespace fi
