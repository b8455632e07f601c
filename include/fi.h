/*
 * fi.h - C ABI of the GB300 paged-KV attention library (libfi.so).
 *
 * Batched attention over a paged KV cache for LLM serving: prefill,
 * single-row decode and multi-token speculative verify, computing
 * softmax(Q K^T * sm_scale + mask) V with fp32 accumulation and a per-row
 * log-sum-exp, plus split-KV partial states merged by their log-sum-exp.
 *
 * The operation is the one described by three pull requests of the
 * AMD-Ecosystem FlashInfer fork, cited below by key:
 *   [P1] "Route non-causal windowed prefill to AITER's masked kernel" (#339)
 *   [P2] "Support speculative-decode verify on ROCm, and stop auto routing
 *         short-query prefill to AITER" (#362)
 *   [P3] "Refuse attention inputs the ROCm kernels would compute wrongly" (#399)
 *
 * Definition (per request b, query row i in [0, Lq_b), query head h,
 * g = num_qo_heads / num_kv_heads, kv head h / g):
 *   Lk_b  = (kv_indptr[b+1] - kv_indptr[b] - 1) * page_size + last_page_len[b]
 *           (0 when the request has no page) - from the page metadata, never
 *           from a caller-supplied length [P2 "Review notes"];
 *   key j lives in page kv_indices[kv_indptr[b] + j / page_size], slot
 *           j % page_size;
 *   valid(i, j) = (!causal || j <= i + Lk - Lq)                [P2 "Summary"]
 *              && (window_left < 0 || j + Lq + window_left >= Lk + i)
 *              - a left-only window anchored bottom-right and applied with
 *                or without causal [P1 "Why window_size_right stays -1"];
 *                all compares are signed [P1 "What changed"];
 *   s_j = sm_scale * <q[i,h,:], k[j,h/g,:]>;
 *   lse = ln sum_{valid j} exp(s_j)      (natural log; -inf when no key is valid)
 *   o   = sum_{valid j} exp(s_j - lse) v[j,h/g,:]   (0 when no key is valid).
 *
 * Conventions for every entry point:
 *   - All tensor data pointers are DEVICE pointers owned by the caller; the
 *     library never frees them. Host arrays are read during the call only.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Launches are asynchronous on it; run calls never synchronise
 *     the host and never allocate, so they can be captured in a CUDA graph.
 *   - Strides are in elements. The last dimension of every tensor must have
 *     stride 1; a strided last dim is refused, never copied [P3 "Strided
 *     layouts", "Architecture / design notes"].
 *   - Errors are return codes; nothing aborts or traps. fi_last_error() gives
 *     a thread-local message naming the field, the expected value and the
 *     value given [P3 "Plan-vs-run shapes"].
 *   - Stream order between a plan and its runs (outside stream capture) is
 *     kept by the library: a run() on another stream than the one fi_plan()
 *     uploaded on waits for that upload, a run() on another stream than the
 *     plan's previous run() waits for that run (the runs of one plan share its
 *     split-KV scratch), and fi_plan() waits for the plan's latest run() before
 *     it overwrites the workspace. A run() captured in a CUDA graph reads the
 *     plan that the workspace holds when the graph is launched: launch the
 *     graph on the stream that re-plans, or order the two yourself, and do not
 *     re-plan on another stream while a launch of the graph is in flight
 *     [P2 "Architecture / design notes"]. fi_plan() itself refuses a stream
 *     that is capturing.
 *   - Kernel configuration (the dynamic shared-memory limit) is applied once
 *     per device at the first run() there; make that first run() before any
 *     capture on that device.
 *   - Environment, read once per process: FI_LOG=1 prints every refusal and
 *     CUDA failure on stderr, 2 also each committed plan (kernel, tile rows,
 *     items, chunks, grid), 3 also each run() launch; unset or 0 prints
 *     nothing. FI_CHECK_INDICES=1 makes every paged run() check the plan's
 *     page-table entries on the device first (see fi_check_kv_indices); a run
 *     whose table fails does no attention work and fi_plan_device_error
 *     reports it.
 */
#ifndef FI_H_
#define FI_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fi_status {
  FI_OK = 0,
  FI_ERR_INVALID_ARG = 1,          /* null pointer, bad rank, negative size, ... */
  FI_ERR_STRIDED_LAST_DIM = 2,     /* an input whose last dim has stride != 1 */
  FI_ERR_NONCONTIGUOUS_OUTPUT = 3, /* out / lse / merge outputs not packed */
  FI_ERR_GQA_INDIVISIBLE = 4,      /* num_kv_heads == 0 or Hq % Hk != 0 */
  FI_ERR_PLAN_MISMATCH = 5,        /* run() tensors disagree with plan() */
  FI_ERR_NOT_PLANNED = 6,          /* run() before a successful plan() */
  FI_ERR_KV_SHORTER_THAN_Q = 7,    /* causal with Lk_b < Lq_b (from metadata) */
  FI_ERR_CAPACITY = 8,             /* workspace too small / graph-frozen shape */
  FI_ERR_UNSUPPORTED = 9,          /* head_dim, dtype or group size not built */
  FI_ERR_CUDA = 10                 /* a CUDA runtime call failed */
} fi_status;

typedef enum fi_dtype { FI_F16 = 0, FI_BF16 = 1, FI_F32 = 2, FI_I32 = 3, FI_U8 = 4 } fi_dtype;

/* A strided view of caller-owned device memory. Unused trailing entries of
 * shape/stride are ignored. */
typedef struct fi_tensor {
  void* data;
  fi_dtype dtype;
  int32_t ndim; /* 1..4 */
  int64_t shape[4];
  int64_t stride[4]; /* elements */
} fi_tensor;

typedef struct fi_plan_s* fi_plan_t;

/* Read-back of a plan's host-side metadata (for tests and diagnostics). */
typedef struct fi_plan_info {
  int32_t batch;
  int32_t total_rows;     /* T = qo_indptr[batch] */
  int32_t kernel;         /* 0 decode, 1 prefill M=16, 2 prefill M=64, 3 prefill M=128 */
  int32_t tile_rows;      /* packed (query row x head-in-group) rows per tile */
  int32_t num_items;      /* work items (request, kv head, q tile, kv chunk) */
  int32_t num_partials;   /* partial (o, lse) slots used for split-KV */
  int32_t num_merge_rows; /* query tokens whose partials are merged */
  int32_t max_chunks;     /* most KV chunks any tile was split into */
  int32_t grid;           /* CTAs launched by run() */
  int32_t graph_mode;
} fi_plan_info;

/*
 * Bytes of device workspace a plan needs for the given capacities.
 * max_kv_chunks bounds how many split-KV chunks one query tile may be cut
 * into (the planner never exceeds what the workspace holds).
 */
size_t fi_workspace_bytes(int32_t max_batch, int32_t max_total_rows, int32_t num_qo_heads,
                          int32_t head_dim, int32_t max_kv_chunks);

/*
 * Create a plan object bound to a caller-owned device workspace.
 *   workspace       device buffer, 256-byte aligned, or NULL for a host-only
 *                   plan (validation and planning without a GPU; run()
 *                   refuses it).
 *   enable_graph_capture  non-zero: run() launches a grid that does not depend
 *                   on the batch, the kernel choice is frozen by the first
 *                   plan, and later plans may not exceed max_batch or
 *                   max_total_rows [P2 "Architecture / design notes"].
 * The library allocates only the host plan object and a pinned host staging
 * buffer here. Returns FI_ERR_CAPACITY if workspace_bytes cannot hold the
 * metadata for max_batch / max_total_rows.
 */
fi_status fi_plan_create(fi_plan_t* plan, void* workspace, size_t workspace_bytes,
                         int32_t enable_graph_capture, int32_t max_batch,
                         int32_t max_total_rows);

/*
 * Plan one batch ([P2 "What changed"], [P3 "Plan-vs-run shapes"]).
 *   qo_indptr      host int32 [batch+1], non-decreasing from 0. Must be NULL
 *                  when q_len_per_req >= 1: the planner then uses
 *                  qo_indptr[b] = q_len_per_req * b (the verify adapter of
 *                  [P2 "What changed"]).
 *   kv_indptr      host int32 [batch+1], page offsets into kv_indices.
 *   last_page_len  host int32 [batch]; in [1, page_size] for a request with
 *                  pages (ignored for a request with none).
 *   page_size      tokens per page, >= 1.
 *   num_qo_heads, num_kv_heads  Hq % Hk must be 0 and Hk > 0 [P3 "GQA head
 *                  divisibility"].
 *   head_dim       64 or 128.
 *   causal         bottom-right causal mask when non-zero.
 *   window_left    -1 (no window) or >= 0; values >= Lk act as -1.
 *   dtype          FI_F16 or FI_BF16 (q, K, V and out share it).
 *   q_len_per_req  0 plans a prefill (fi_batch_prefill_paged); 1 plans a
 *                  decode and > 1 a speculative verify with that many draft
 *                  rows per request (fi_batch_decode_paged; verify forces the
 *                  causal mask) [P2 "What changed"].
 *   force_kv_chunks 0 lets the planner split KV; > 0 cuts every query tile's
 *                  full key range [0, Lk) into exactly that many chunks.
 *   stream         the metadata upload is enqueued on it.
 * Validates everything before changing any state: a refused plan leaves the
 * previous plan usable [P2 "Review notes"], [P3 "Plan-vs-run shapes"]. Host
 * arrays are deep-copied [P3 "AITER decode LSE fallback"]. Refusals:
 * FI_ERR_GQA_INDIVISIBLE, FI_ERR_KV_SHORTER_THAN_Q (causal and Lk_b < Lq_b,
 * including Lk_b < q_len_per_req), FI_ERR_CAPACITY (workspace, or a graph-mode
 * plan beyond its capacities or changing a frozen shape), FI_ERR_UNSUPPORTED,
 * FI_ERR_INVALID_ARG.
 */
fi_status fi_plan(fi_plan_t plan, const int32_t* qo_indptr, const int32_t* kv_indptr,
                  const int32_t* last_page_len, int32_t batch, int32_t page_size,
                  int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                  int32_t causal, int32_t window_left, fi_dtype dtype,
                  int32_t q_len_per_req, int32_t force_kv_chunks, void* stream);

/*
 * Batched prefill over the paged cache, for a plan made with q_len_per_req 0.
 *   q           [T', Hq, d], T' >= planned T (graph callers may pad; rows past T
 *               are neither read nor written), any token/head strides.
 *   k_cache, v_cache  [num_pages, page_size, Hk, d] (NHD), any page/token/head
 *               strides; 16-byte aligned rows.
 *   kv_indices  int32 [>= kv_indptr[batch]], contiguous.
 *   sm_scale    score scale (usually 1/sqrt(d)).
 *   out         [T', Hq, d] packed, dtype of q. Rows < T are written.
 *   lse         [T', Hq] fp32 packed, or NULL.
 * Shape, head, head_dim, page_size and dtype must match the plan
 * (FI_ERR_PLAN_MISMATCH names the field); FI_ERR_NOT_PLANNED before a plan.
 */
fi_status fi_batch_prefill_paged(fi_plan_t plan, const fi_tensor* q, const fi_tensor* k_cache,
                                 const fi_tensor* v_cache, const fi_tensor* kv_indices,
                                 float sm_scale, fi_tensor* out, fi_tensor* lse, void* stream);

/*
 * Batched decode (q_len_per_req == 1) or speculative verify
 * (q_len_per_req > 1, causal) for a plan made with that q_len_per_req.
 * q is [batch * q_len_per_req (or more), Hq, d]; the other arguments are as
 * for fi_batch_prefill_paged.
 */
fi_status fi_batch_decode_paged(fi_plan_t plan, const fi_tensor* q, const fi_tensor* k_cache,
                                const fi_tensor* v_cache, const fi_tensor* kv_indices,
                                float sm_scale, fi_tensor* out, fi_tensor* lse, void* stream);

/*
 * Ragged prefill over contiguous K/V: the third prefill entry point beside
 * single and paged prefill ("Route non-causal windowed prefill to AITER's
 * masked kernel" (#339), "Pull request overview", whose regression tests
 * cover all three), which runs on K/V that is already contiguous, so there
 * is no page gather ("Support speculative-decode verify on ROCm, and stop
 * auto routing short-query prefill to AITER" (#362), "Architecture / design
 * notes"). The keys of request b are rows kv_indptr[b] .. kv_indptr[b+1]-1 of
 * one [rows, Hk, d] tensor, so no page table is read; masks, GQA grouping,
 * lse and the split-KV merge are those of fi_batch_prefill_paged.
 *
 * fi_plan_ragged: as fi_plan for a prefill, with
 *   kv_indptr  host int32 [batch+1]: each request's first K/V row (kv_len_b =
 *              kv_indptr[b+1] - kv_indptr[b]); nondecreasing, kv_indptr[0] = 0.
 * There is no page size or last_page_len. Refusals as for fi_plan
 * (FI_ERR_KV_SHORTER_THAN_Q under the causal mask, ...).
 *
 * fi_batch_prefill_ragged: run a plan from fi_plan_ragged.
 *   q     [T, Hq, d]  as for fi_batch_prefill_paged;
 *   k, v  [rows, Hk, d], rows >= kv_indptr[batch], same dtype as q, last dim
 *         contiguous, other strides multiples of 8 elements, 16-byte aligned;
 *   out / lse as for fi_batch_prefill_paged.
 * A paged plan given to this call, or a ragged plan to the paged calls, is
 * refused with FI_ERR_PLAN_MISMATCH. Nothing is allocated or synchronised.
 */
/*
 * Paged prefill with a custom (tree) mask. Tree drafts (EAGLE-2, Medusa,
 * SpecInfer) need a topology mask: the causal verify mask lets a draft attend
 * to a sibling on another branch ("Support speculative-decode verify on ROCm,
 * and stop auto routing short-query prefill to AITER" (#362), "Architecture /
 * design notes"). The mask is ANDed into the mask that causal / window_left
 * define; plan with causal = 0 to apply it alone.
 *
 * fi_plan_masked: as fi_plan for a prefill, plus
 *   mask_indptr  host int32 [batch+1]: request b's mask bits start at byte
 *                mask_indptr[b] of the custom_mask tensor; its segment holds
 *                Lq_b * Lk_b bits (query row i, key j at bit i * Lk_b + j,
 *                least significant bit of each byte first), so
 *                mask_indptr[b+1] - mask_indptr[b] >= ceil(Lq_b * Lk_b / 8).
 * Masked plans run on the same kernels as unmasked ones: the short-query
 * kernel (at most 32 packed rows per request), the tcgen05 kernel (more rows,
 * page sizes that are multiples of 8) or the mma.sync kernels (other page
 * sizes). FI_ERR_INVALID_ARG for a segment shorter than its request's bits or
 * a decreasing mask_indptr.
 *
 * fi_batch_prefill_paged_masked: as fi_batch_prefill_paged, plus
 *   custom_mask  device FI_U8 [>= mask_indptr[batch]] bytes, contiguous.
 * A masked plan refuses the unmasked run calls and an unmasked plan this one
 * (FI_ERR_PLAN_MISMATCH).
 */
fi_status fi_plan_masked(fi_plan_t plan, const int32_t* qo_indptr, const int32_t* kv_indptr,
                         const int32_t* last_page_len, int32_t batch, int32_t page_size,
                         int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                         int32_t causal, int32_t window_left, fi_dtype dtype,
                         const int32_t* mask_indptr, int32_t force_kv_chunks, void* stream);
fi_status fi_batch_prefill_paged_masked(fi_plan_t plan, const fi_tensor* q,
                                        const fi_tensor* k_cache, const fi_tensor* v_cache,
                                        const fi_tensor* kv_indices, const fi_tensor* custom_mask,
                                        float sm_scale, fi_tensor* out, fi_tensor* lse,
                                        void* stream);

fi_status fi_plan_ragged(fi_plan_t plan, const int32_t* qo_indptr, const int32_t* kv_indptr,
                         int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads,
                         int32_t head_dim, int32_t causal, int32_t window_left, fi_dtype dtype,
                         int32_t force_kv_chunks, void* stream);
fi_status fi_batch_prefill_ragged(fi_plan_t plan, const fi_tensor* q, const fi_tensor* k,
                                  const fi_tensor* v, float sm_scale, fi_tensor* out,
                                  fi_tensor* lse, void* stream);

/*
 * Merge two attention states by their log-sum-exp [P3 "Graph-mode
 * partial_state merge"]:
 *   m = max(s_a, s_b), s = m + ln(exp(s_a - m) + exp(s_b - m)),
 *   v = exp(s_a - s) v_a + exp(s_b - s) v_b;  both -inf gives v = 0, s = -inf.
 *   v_a, v_b, v_out  [rows, H, d], one dtype of FI_F16 / FI_BF16 / FI_F32;
 *                    v_out packed; v_out may be v_a (in place, element-wise).
 *   s_a, s_b, s_out  [rows, H] fp32 natural-log LSE; s_out packed, may be s_a.
 *   num_rows_dev     optional device int32: only rows < *num_rows_dev are
 *                    touched, so a captured graph re-planned to fewer rows
 *                    does not write past its output. NULL = all rows.
 */
fi_status fi_merge_state(const fi_tensor* v_a, const fi_tensor* s_a, const fi_tensor* v_b,
                         const fi_tensor* s_b, fi_tensor* v_out, fi_tensor* s_out,
                         const int32_t* num_rows_dev, void* stream);

/*
 * Variable-length merge: row r merges states merge_indptr[r] ..
 * merge_indptr[r+1]-1 of v [n, H, d] (fp32) / s [n, H] (fp32) into
 * v_out [rows, H, d] (F16/BF16/F32, packed) and s_out [rows, H] (fp32,
 * packed, or NULL). merge_indptr_dev is a device int32 [rows+1]; a row with
 * no state gets v = 0, s = -inf. num_rows_dev as for fi_merge_state.
 */
fi_status fi_merge_states(const fi_tensor* v, const fi_tensor* s, const int32_t* merge_indptr_dev,
                          int32_t rows, fi_tensor* v_out, fi_tensor* s_out,
                          const int32_t* num_rows_dev, void* stream);

/*
 * Chain speculative-sampling acceptance step: the sampler the multi-token
 * verify feeds ("Support speculative-decode verify on ROCm, and stop auto
 * routing short-query prefill to AITER" (#362), "Summary"; it takes a chain
 * of num_speculate_tokens drafts per request, not a tree, "Architecture /
 * design notes"). The steps are the published speculative sampling
 * (Leviathan, Kalman and Matias 2023; Chen et al. 2023):
 *   draft i (token x_i) is accepted while u_i * q_i(x_i) <= p_i(x_i), the
 *   product and compare in fp32; at the first rejection i one token is drawn
 *   from max(0, p_i - q_i) (p_i when that is all zero), or from p_n if all n
 *   drafts are accepted. A draw with uniform u picks the smallest token t
 *   whose cumulative weight (fp64) exceeds u * total weight.
 *
 *   draft_probs       F32 [B, n, V]   q; vocabulary dim contiguous
 *   draft_token_ids   I32 [B, n]      x
 *   target_probs      F32 [B, n+1, V] p (row n: the bonus distribution)
 *   uniform_accept    F32 [B, n]      the acceptance tests' uniforms
 *   uniform_sample    F32 [B]         the final draw's uniform, in [0, 1)
 *   output_token_ids  I32 [B, n+1]    out: accepted drafts, the drawn token,
 *                                     then -1 (packed)
 *   accepted_num      I32 [B]         out: drafts accepted before the first
 *                                     rejection
 *   emitted_num       I32 [B] or NULL out: accepted_num + 1
 * All device memory, caller-owned; one CTA per request on `stream`; nothing
 * is allocated. The draft arguments may be NULL when n = 0. Errors:
 * FI_ERR_INVALID_ARG (shapes, dtypes), FI_ERR_STRIDED_LAST_DIM,
 * FI_ERR_NONCONTIGUOUS_OUTPUT, FI_ERR_CUDA.
 */
fi_status fi_chain_speculative_sampling(const fi_tensor* draft_probs,
                                        const fi_tensor* draft_token_ids,
                                        const fi_tensor* target_probs,
                                        const fi_tensor* uniform_accept,
                                        const fi_tensor* uniform_sample,
                                        fi_tensor* output_token_ids, fi_tensor* accepted_num,
                                        fi_tensor* emitted_num, void* stream);

/* Copy a plan's host metadata out (any pointer may be NULL):
 *   items [num_items * 8] int32: per work item {request (-1 = schedule
 *         padding), kv_head, first packed row, kv_begin, kv_end, chunk (-1 =
 *         written directly), chunks of the item's row tile, partial base};
 *         the items sit in per-CTA order: CTA c runs positions c, c + grid, ...;
 *   merge_indptr [total_rows + 1]: partial slots of each query token. */
fi_status fi_plan_get_info(fi_plan_t plan, fi_plan_info* info, int32_t* items,
                           int32_t items_capacity, int32_t* merge_indptr,
                           int32_t merge_capacity);

/* Copy the plan's device-side metadata back to the host (synchronises the
 * stream): the same layout as fi_plan_get_info's arrays. For tests. */
fi_status fi_plan_read_device(fi_plan_t plan, int32_t* items, int32_t items_capacity,
                              int32_t* merge_indptr, int32_t merge_capacity, void* stream);

/* Read the device error flags of the plan's workspace (ordered after the
 * plan's latest upload and run(); synchronises the stream). *err_flag is a bit
 * set, 0 when nothing went wrong since the last fi_plan or clear:
 *   1  a kernel's bounded wait on an mbarrier expired (2 s, or the limit of
 *      fi_plan_set_wait_limit): the kernel gave up the rest of its work,
 *      waited (bounded) for its own copies and tensor-core work in flight and
 *      exited, so the context stays usable but that launch's output is not
 *      valid;
 *   2  the page-table check (fi_check_kv_indices, or FI_CHECK_INDICES) found
 *      entries outside the cache; the attention work of the run it guarded
 *      was not done.
 * clear != 0 resets both afterwards. Errors: FI_ERR_INVALID_ARG (NULL plan or
 * pointer, host-only plan), FI_ERR_NOT_PLANNED, FI_ERR_CUDA. */
fi_status fi_plan_device_error(fi_plan_t plan, int32_t* err_flag, int clear, void* stream);

/* Limit, in nanoseconds, of every bounded wait on an mbarrier in the plan's
 * kernels, from the next fi_plan on; 0 restores the default of 2 s. A small
 * limit makes waits expire on purpose, which is how the failure path (abort,
 * drain, error flag, usable context) is tested; the waits that drain a CTA's
 * own copies and tensor-core work before it exits always keep the 2 s limit.
 * Errors: FI_ERR_INVALID_ARG (NULL plan). */
fi_status fi_plan_set_wait_limit(fi_plan_t plan, uint64_t limit_ns);

/* Range check of the plan's page table on the device ([P2 "Review notes"]: a
 * wrong page table or indptr becomes a memory fault; [P3 "What changed"]).
 * Counts the entries kv_indices[0 .. kv_indptr[batch]) outside
 * [0, num_pages) into the plan's workspace, where fi_plan_device_error reads
 * them as bit 2 and where the attention kernels of a run read them and then
 * do no work. Launches one small kernel on `stream`, never traps; the count
 * stays until the next check, fi_plan or clear. kv_indices: device int32,
 * contiguous, at least kv_indptr[batch] entries; num_pages: pages in the K/V
 * cache. Errors: FI_ERR_INVALID_ARG, FI_ERR_NOT_PLANNED, FI_ERR_PLAN_MISMATCH
 * (a ragged plan, or a table shorter than planned), FI_ERR_CUDA. */
fi_status fi_check_kv_indices(fi_plan_t plan, const fi_tensor* kv_indices, int64_t num_pages,
                              void* stream);

/*
 * Batch decode that allocates nothing (the pages have no counterpart; this is
 * an addition of this library).
 *
 * For callers that cannot allocate device memory when they run attention: a
 * serving loop that handed all GPU memory to its own pool up front, code that
 * runs inside another framework's allocator, or a host path where a
 * cudaMalloc/cudaFree (or a caching allocator's growth) would stall the device.
 * Instead of a caller workspace it uses one fixed scratch array compiled into
 * libfi: fi_noalloc_scratch_bytes() bytes (32 MiB) that every GPU which loads
 * the library holds until the process exits. The call makes no cudaMalloc,
 * cudaFree or other allocating call; out and lse are the caller's.
 *
 *   q            [>= batch, Hq, d] bf16/fp16, one query row per request.
 *   k_cache, v_cache  [pages, page_size, Hk, d], as for fi_batch_decode_paged.
 *   kv_indices   int32 device page table; kv_indptr_dev [batch+1] and
 *                last_page_len_dev [batch] are device int32 arrays, read on the
 *                device (their values are trusted: they are not checked on the
 *                host).
 *   window_left  -1 or >= 0; kv_chunks in [1, 64]: each request's keys are cut
 *                into that many even chunks whose partial states are merged.
 *   out, lse     packed [>= batch, Hq, d] / [>= batch, Hq] fp32.
 * Group size 1, 2 or 4 and head_dim 64 or 128. A batch whose plan and partial
 * states do not fit the scratch returns FI_ERR_CAPACITY (message from
 * fi_noalloc_last_error()). The first call on a device looks up the array's
 * device address once with that device current; make that first call before
 * any stream capture. Every call rewrites the scratch from scratch, and calls
 * share it: two calls that overlap on the GPU (different streams, no ordering)
 * race.
 */
fi_status fi_batch_decode_paged_noalloc(const fi_tensor* q, const fi_tensor* k_cache,
                                        const fi_tensor* v_cache, const fi_tensor* kv_indices,
                                        const int32_t* kv_indptr_dev,
                                        const int32_t* last_page_len_dev, int32_t batch,
                                        int32_t window_left, int32_t kv_chunks, float sm_scale,
                                        fi_tensor* out, fi_tensor* lse, void* stream);
/* Size of the fixed scratch array behind fi_batch_decode_paged_noalloc. */
size_t fi_noalloc_scratch_bytes(void);
/* Error flag of the latest fi_batch_decode_paged_noalloc on the current device
 * (the flag belongs to that call; the next call clears it): 1 when one of its
 * bounded waits expired and its out / lse are not valid, else 0 (also before
 * the first call). clear != 0 resets it. Synchronises `stream`; allocates
 * nothing. Errors: FI_ERR_INVALID_ARG (NULL err_flag), FI_ERR_CUDA. */
fi_status fi_noalloc_device_error(int32_t* err_flag, int clear, void* stream);
/* Thread-local message of the last refusal of fi_batch_decode_paged_noalloc. */
const char* fi_noalloc_last_error(void);

void fi_plan_destroy(fi_plan_t plan);
const char* fi_last_error(void);
const char* fi_status_str(fi_status status);

#ifdef __cplusplus
}
#endif

#endif /* FI_H_ */
