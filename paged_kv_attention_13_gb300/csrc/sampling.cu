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
// One CTA per request. Warp 0 runs the n acceptance tests at once (a ballot
// finds the first rejection). The drawn row is then streamed once, in blocks
// of 128 tokens dealt round-robin to the warps (one coalesced 16-byte load per
// lane per block): each block's weight is summed in fp32 (four tokens per lane,
// then a butterfly over the lanes) into shared memory. Warp 0 scans the block
// sums in fp64 to find the block holding u * total, re-reads that one block and
// picks the token. The kernel is bound by the one or two rows of V floats it
// reads per request. (Weights are summed in fp32 inside a 128-token block and
// in fp64 across blocks, so a draw within about 1e-6 of a cumulative boundary
// may land on the neighbouring token of an all-fp64 sum.)
#include "common.cuh"

namespace fi {
namespace {

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

// Block sums of the row into bsum[0 .. nb) (all warps); returns nothing, the
// caller synchronises.
__device__ void block_sums(const float* p, const float* q, int V, bool vec, int nb, float* bsum,
                           int warp, int lane) {
  for (int blk = warp; blk < nb; blk += kSampWarps) {
    float s = lane_sum(lane_weights(p, q, blk, lane, V, vec));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, off));
    if (lane == 0) bsum[blk] = s;
  }
}

__global__ void __launch_bounds__(kSampThreads) chain_spec_kernel(const SpecParams sp) {
  extern __shared__ float bsum[];  // [ceil(V / 128)] block sums
  const int b = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = sp.n, V = sp.vocab;
  const int nb = (V + kBlk - 1) / kBlk;
  __shared__ int s_acc, s_zero, s_token;

  // 1. acceptance tests, 32 drafts per ballot
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

  // 2. the row to draw from: the residual at the first rejection, or p_n
  const float* p = sp.target_probs + int64_t(b) * sp.tp_sb + int64_t(acc) * sp.tp_si;
  const float* q = acc < n ? sp.draft_probs + int64_t(b) * sp.dp_sb + int64_t(acc) * sp.dp_si
                           : nullptr;
  const bool vec = (reinterpret_cast<uintptr_t>(p) % 16 == 0) &&
                   (!q || reinterpret_cast<uintptr_t>(q) % 16 == 0);
  block_sums(p, q, V, vec, nb, bsum, warp, lane);
  __syncthreads();
  if (q) {  // an all-zero residual (p == q): draw from p itself
    if (warp == 0) {
      bool any = false;
      for (int k = lane; k < nb; k += 32) any = any || bsum[k] > 0.f;
      any = __any_sync(0xffffffffu, any);
      if (lane == 0) s_zero = !any;
    }
    __syncthreads();
    if (s_zero) {
      q = nullptr;
      block_sums(p, q, V, vec, nb, bsum, warp, lane);
    }
    __syncthreads();
  }

  // 3. warp 0: the block holding u * total (fp64 scan of the block sums),
  // then the token inside it
  if (warp == 0) {
    double tot = 0.0;
    for (int k = lane; k < nb; k += 32) tot += double(bsum[k]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
    const double target = double(__ldg(sp.u_sample + b)) * tot;
    double run = 0.0;  // cumulative weight before block k0
    int blk = -1, last_blk = -1;
    double blk_start = 0.0, last_start = 0.0;
    for (int k0 = 0; k0 < nb && blk < 0; k0 += 32) {
      const double v = k0 + lane < nb ? double(bsum[k0 + lane]) : 0.0;
      double c = v;  // inclusive scan over the lanes
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, c, off);
        if (lane >= off) c += y;
      }
      const unsigned pos = __ballot_sync(0xffffffffu, v > 0.0);
      if (pos) {
        const int l = 31 - __clz(pos);
        last_blk = k0 + l;
        last_start = run + __shfl_sync(0xffffffffu, c - v, l);
      }
      const unsigned hit = __ballot_sync(0xffffffffu, k0 + lane < nb && run + c > target);
      if (hit) {
        const int l = __ffs(hit) - 1;
        blk = k0 + l;
        blk_start = run + __shfl_sync(0xffffffffu, c - v, l);
      }
      run += __shfl_sync(0xffffffffu, c, 31);
    }
    if (blk < 0) {  // rounding put the target past the end: the last positive block
      blk = last_blk;
      blk_start = last_start;
    }
    int token = -1;
    if (blk >= 0) {
      const float4 w = lane_weights(p, q, blk, lane, V, vec);
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

  // 4. outputs: accepted drafts, the drawn token, then -1
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

int chain_spec_max_vocab() { return 48 * 1024 / 4 * kBlk; }

cudaError_t launch_chain_spec_sampling(const SpecParams& sp, int batch, cudaStream_t stream) {
  if (batch <= 0) return cudaSuccess;
  const int nb = (sp.vocab + kBlk - 1) / kBlk;
  chain_spec_kernel<<<batch, kSampThreads, size_t(nb) * sizeof(float), stream>>>(sp);
  return cudaGetLastError();
}

}  // namespace fi
