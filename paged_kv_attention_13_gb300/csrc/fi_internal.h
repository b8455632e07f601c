// Shared host/device definitions of libfi: the workspace layout written by
// the planner and read by the kernels, and the kernel launch parameters.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace fi {

// One unit of work: a tile of packed query rows (query row x head in the GQA
// group) of one request and one kv head, against one chunk of its keys. The
// second half repeats the request's metadata, so a kernel that starts an item
// needs no further load before it reads the page table.
struct alignas(64) WorkItem {
  int32_t b;             // request
  int32_t kv_head;
  int32_t row0;          // first packed row (query row * group + head in group)
  int32_t kv_begin;      // this chunk's key range [kv_begin, kv_end) before masking
  int32_t kv_end;
  int32_t chunk;         // -1: the tile has one chunk and writes out/lse directly
  int32_t num_chunks;    // chunks of this tile
  int32_t partial_base;  // partial slot of the tile's first token, chunk 0
  int32_t tok0;          // qo_indptr[b]: global index of the request's first query row
  int32_t lq;            // query rows of the request
  int32_t lk;            // keys of the request
  int32_t kv_start;      // kv_indptr[b]: first page-table entry (ragged: first K/V row)
  int32_t mask_base;     // mask_indptr[b]: first byte of the request's custom mask
  int32_t pad[3];
};
static_assert(sizeof(WorkItem) == 64, "work item is sixteen int32");
// the first eight fields of every item are reported by fi_plan_get_info
constexpr int kItemPublicInts = 8;

// Device workspace header (the first bytes of the caller's workspace). The
// kernels read every offset from here, so a re-plan that moves arrays is seen
// by a captured graph on its next replay.
struct alignas(128) WsHeader {
  int32_t n_items;
  int32_t n_merge_rows;  // tokens whose partial states get merged
  int32_t total_rows;    // T
  int32_t batch;
  int32_t group;         // Hq / Hk
  int32_t causal;
  int32_t window_left;
  int32_t tile_rows;     // packed rows per tile
  int32_t num_qo_heads;
  int32_t head_dim;
  int32_t err_flag;      // set by a kernel whose bounded wait expired
  int32_t index_error;   // kv_indices entries out of range, counted by the index check;
                         // the attention kernels do no work while it is non-zero
  int64_t off_qo_indptr;     // int32 [batch+1]
  int64_t off_kv_indptr;     // int32 [batch+1]
  int64_t off_kv_len;        // int32 [batch]
  int64_t off_merge_indptr;  // int32 [T+1]
  int64_t off_merge_rows;    // int32 [n_merge_rows]
  int64_t off_items;         // WorkItem [n_items], always kItemsOffset
  int64_t off_tmp_lse;       // float [partials, Hq]
  int64_t off_tmp_o;         // float [partials, Hq, d]
  int64_t off_mask_indptr;   // int32 [batch+1]: byte offset of each request's custom mask
  uint64_t wait_limit_ns;    // limit of every bounded wait on an mbarrier (0: 2 s)
};
static_assert(sizeof(WsHeader) == 128, "header is 128 bytes");
// The work items follow the header directly: a CTA loads its first item in
// the same round trip as the header.
constexpr int64_t kItemsOffset = sizeof(WsHeader);

template <typename T>
__host__ __device__ inline T* ws_ptr(const void* ws, int64_t off) {
  return reinterpret_cast<T*>(reinterpret_cast<uintptr_t>(ws) + static_cast<uintptr_t>(off));
}

// Everything a run() kernel needs besides the workspace.
struct AttnParams {
  const void* q;
  int64_t q_stride_tok, q_stride_head;
  const void* k;
  int64_t k_stride_page, k_stride_tok, k_stride_head;
  const void* v;
  int64_t v_stride_page, v_stride_tok, v_stride_head;
  const int32_t* kv_indices;
  void* out;        // packed [T, Hq, d]
  float* lse;       // packed [T, Hq] or null
  const void* ws;   // workspace base (WsHeader first)
  float sm_scale_log2;  // sm_scale * log2(e)
  int32_t num_qo_heads;
  int32_t num_kv_heads;
  int32_t page_size;
  int32_t page_shift;   // log2(page_size) when it is a power of two, else -1
  // Ragged (contiguous) K/V: key j of request b is row kv_indptr[b] + j of
  // k / v ([rows, Hk, d]); kv_indices is unused, and page_size / page_shift
  // are 1 << 30 / 30 (one logical page per request).
  int32_t ragged;
  int64_t kv_rows;      // ragged: rows of k / v (the TMA maps' extent)
  // Custom (tree) mask or null: request b's bits (query row i, key j at bit
  // i * Lk + j, least significant bit first) start at byte
  // mask_indptr[b] (workspace array); ANDed into the causal / window mask.
  const uint8_t* custom_mask;
};

enum KernelId : int32_t {
  kDecode = 0,
  kPrefillM16 = 1,
  kPrefillM64 = 2,
  kPrefillM128 = 3,
};

// Launchers (defined in the .cu files). Each returns cudaGetLastError().
// The short-query kernel (kDecode): items of at most 16 packed rows.
// num_pages: pages in the K/V cache tensors (the TMA maps' outer extent);
// tile_rows: the plan's packed rows per item (at most 16).
cudaError_t launch_decode(const AttnParams& p, int head_dim, int group, bool bf16,
                          int64_t num_pages, int tile_rows, int grid, cudaStream_t stream);
// Its tensor-core consumer: any query length with q_len * group <= 16, for
// groups 1, 2, 4, 8, 16 and page sizes whose boxes span whole swizzle atoms.
bool decode_mma_supports(int head_dim, int page_size, int group);
// Its CUDA-core consumer: decode (one query row per request), groups 1, 2, 4.
bool decode_shuffle_supports(int head_dim, int group);
// CTAs per SM the short-query kernel is built for (depends on its consumer).
int decode_ctas_per_sm(int head_dim, int page_size, int group);
cudaError_t launch_prefill_mma(const AttnParams& p, int head_dim, int kernel, bool bf16,
                               int grid, cudaStream_t stream);
cudaError_t launch_prefill_tc(const AttnParams& p, int head_dim, int group, int tile_rows,
                              int64_t q_rows, int64_t num_pages, bool bf16, int grid,
                              cudaStream_t stream);
// Whether the tensor-memory prefill kernel handles this shape.
bool prefill_tc_supports(int head_dim, int page_size, int group);
// Merge the workspace partials of a plan into out / lse.
cudaError_t launch_merge_workspace(const void* ws, void* out, float* lse, int num_heads,
                                   int head_dim, bool bf16, int grid, cudaStream_t stream);
// Variable-length merge over caller tensors.
cudaError_t launch_merge_states(const float* v, const float* s, const int32_t* merge_indptr,
                                int32_t rows, int num_heads, int head_dim, void* v_out,
                                int out_dtype, float* s_out, const int32_t* num_rows_dev,
                                cudaStream_t stream);
// Two-state merge over caller tensors (all packed except the inputs' strides
// which are [rows, H, d] / [rows, H] element strides).
struct MergeTwoParams {
  const void* va; const void* vb; void* vo;
  const float* sa; const float* sb; float* so;
  int64_t va_sr, va_sh, vb_sr, vb_sh;  // row / head strides of v_a, v_b
  int64_t sa_sr, sb_sr;                // row strides of s_a, s_b (head stride 1)
  int32_t rows, heads, head_dim, dtype;
  const int32_t* num_rows_dev;
};
cudaError_t launch_merge_two(const MergeTwoParams& p, cudaStream_t stream);

// Chain speculative-sampling acceptance step (element strides; the vocabulary
// dim is contiguous): draft_probs [B, n, V], draft_ids [B, n], target_probs
// [B, n+1, V], u_accept [B, n], u_sample [B] -> out_tokens [B, n+1] (packed),
// out_accepted [B], out_emitted [B] (or null).
struct SpecParams {
  const float* draft_probs;
  int64_t dp_sb, dp_si;
  const int32_t* draft_ids;
  int64_t ids_sb;
  const float* target_probs;
  int64_t tp_sb, tp_si;
  const float* u_accept;
  int64_t ua_sb;
  const float* u_sample;
  int32_t n, vocab;
  int32_t* out_tokens;
  int32_t* out_accepted;
  int32_t* out_emitted;
};
cudaError_t launch_chain_spec_sampling(const SpecParams& sp, int batch, cudaStream_t stream);
// Largest vocabulary it takes (its block sums live in 48 KB of shared memory).
int chain_spec_max_vocab();

// Count page-table entries of the plan in `ws` outside [0, num_pages) into
// the header's index_error (which the caller zeroes first).
cudaError_t launch_check_indices(void* ws, const int32_t* kv_indices, int64_t num_pages,
                                 int num_sms, cudaStream_t stream);

// Raise a kernel's dynamic shared-memory limit on the current device, once
// per device: the attribute belongs to each device's context, so the first
// launch on every device sets it (before any capture on that device). `done`
// is the kernel's own bit set of devices already configured.
template <class K>
cudaError_t smem_attr_once(K kernel, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Occupancy of each run kernel (CTAs per SM), for persistent grid sizing.
int kernel_ctas_per_sm(int kernel, int head_dim, int group, bool bf16, int page_size);

}  // namespace fi
