// C ABI of libfi: argument validation, the host planner, the metadata upload
// and the run() launches. Page citations use the keys of include/fi.h:
//   [P1] "Route non-causal windowed prefill to AITER's masked kernel" (#339)
//   [P2] "Support speculative-decode verify on ROCm, and stop auto routing
//         short-query prefill to AITER" (#362)
//   [P3] "Refuse attention inputs the ROCm kernels would compute wrongly" (#399)
#include "../../include/fi.h"

#include <algorithm>
#include <numeric>
#include <functional>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstddef>
#include <cstring>
#include <string>
#include <vector>

#include "fi_internal.h"

using fi::WorkItem;
using fi::WsHeader;
using fi::kItemPublicInts;
using fi::kItemsOffset;

namespace {

thread_local std::string g_last_error;

// FI_LOG (read once per process): 0 or unset = silent; 1 = every refusal or
// CUDA failure on stderr; 2 = also each committed plan (kernel, tile, items,
// chunks, grid); 3 = also each run() launch. Costs one branch at level 0.
int log_level() {
  static const int lvl = [] {
    const char* e = std::getenv("FI_LOG");
    return e ? std::atoi(e) : 0;
  }();
  return lvl;
}

// FI_CHECK_INDICES=1 (read once per process): every paged run() first checks
// the plan's page-table entries against the cache's page count on the device;
// a bad entry is counted in the workspace header and the attention kernels of
// that run do no work (fi_plan_device_error then reports it).
bool check_indices_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("FI_CHECK_INDICES");
    return e && std::atoi(e) != 0;
  }();
  return on;
}

fi_status fail(fi_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  if (log_level() >= 1) std::fprintf(stderr, "[fi] %s: %s\n", st == FI_ERR_CUDA ? "error" : "refused", buf);
  return st;
}

fi_status ok() {
  g_last_error.clear();
  return FI_OK;
}

constexpr int64_t kAlign = 256;
int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Everything a committed plan knows (host copy; the device copy is uploaded).
struct PlanState {
  int32_t batch = 0, total_rows = 0, page_size = 0, hq = 0, hk = 0, d = 0;
  int32_t causal = 0, window_left = -1, dtype = 0, q_len_per_req = 0, group = 1;
  int32_t kernel = 0, tile_rows = 0, grid = 0, max_chunks = 1, n_partials = 0;
  int32_t kv_indices_len = 0;  // page-table entries (ragged: K/V rows) the plan reads
  int32_t ragged = 0;          // contiguous K/V rows instead of a page table
  int32_t masked = 0;          // a custom mask is ANDed in
  int32_t mask_bytes = 0;      // custom mask bytes the plan reads (mask_indptr[batch])
  std::vector<int32_t> qo_indptr, kv_indptr, kv_len, merge_indptr, merge_rows, mask_indptr;
  std::vector<WorkItem> items;
  WsHeader hdr{};
  int64_t meta_bytes = 0;   // header + metadata arrays (uploaded)
  int64_t total_bytes = 0;  // + partial buffers
};

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace

struct fi_plan_s {
  void* ws = nullptr;
  size_t ws_bytes = 0;
  bool host_only = true;
  bool graph = false;
  int32_t max_batch = 0, max_total_rows = 0;
  int num_sms = 152;
  // Two pinned host buffers for the metadata upload, used in turn: a plan
  // waits (on the host) only for the upload made two plans earlier, so a
  // serving loop can plan step n+1 while step n's upload is still queued.
  void* staging[2] = {nullptr, nullptr};
  size_t staging_bytes[2] = {0, 0};
  cudaEvent_t staged[2] = {nullptr, nullptr};  // each buffer's upload has completed
  bool staged_pending[2] = {false, false};
  int stage_next = 0;
  cudaEvent_t upload_done = nullptr;  // the latest upload (the one run() must follow)
  bool upload_pending = false;
  cudaStream_t upload_stream = nullptr;  // the stream of the last metadata upload
  // Stream order between plan() and run(): every run() outside a capture
  // records run_done on its stream; a run on another stream than the upload's
  // waits for upload_done, a run on another stream than the previous run's
  // waits for run_done, and plan() waits for run_done before it overwrites
  // the workspace.
  cudaEvent_t run_done = nullptr;
  bool run_recorded = false;
  cudaStream_t last_run_stream = nullptr;
  uint64_t wait_limit_ns = 0;  // written into each plan's header (0: the kernels' 2 s)
  bool planned = false;
  PlanState st;
  // shape frozen by the first plan of a graph-mode plan object
  bool frozen = false;
  int32_t fz_kernel = 0, fz_qlpr = 0, fz_hq = 0, fz_hk = 0, fz_d = 0, fz_dtype = 0, fz_page = 0;
  int32_t fz_ragged = 0, fz_masked = 0;
};

extern "C" const char* fi_last_error(void) { return g_last_error.c_str(); }

extern "C" const char* fi_status_str(fi_status s) {
  switch (s) {
    case FI_OK: return "FI_OK";
    case FI_ERR_INVALID_ARG: return "FI_ERR_INVALID_ARG";
    case FI_ERR_STRIDED_LAST_DIM: return "FI_ERR_STRIDED_LAST_DIM";
    case FI_ERR_NONCONTIGUOUS_OUTPUT: return "FI_ERR_NONCONTIGUOUS_OUTPUT";
    case FI_ERR_GQA_INDIVISIBLE: return "FI_ERR_GQA_INDIVISIBLE";
    case FI_ERR_PLAN_MISMATCH: return "FI_ERR_PLAN_MISMATCH";
    case FI_ERR_NOT_PLANNED: return "FI_ERR_NOT_PLANNED";
    case FI_ERR_KV_SHORTER_THAN_Q: return "FI_ERR_KV_SHORTER_THAN_Q";
    case FI_ERR_CAPACITY: return "FI_ERR_CAPACITY";
    case FI_ERR_UNSUPPORTED: return "FI_ERR_UNSUPPORTED";
    case FI_ERR_CUDA: return "FI_ERR_CUDA";
  }
  return "FI_ERR_UNKNOWN";
}

namespace {

// Metadata bytes for a batch (header + int arrays + items), 256-aligned.
int64_t meta_bytes_for(int64_t batch, int64_t rows, int64_t n_merge, int64_t n_items) {
  int64_t off = kItemsOffset;
  off += int64_t(sizeof(WorkItem)) * n_items;  // items
  off = align_up(off + 4 * (batch + 1), 16);  // qo_indptr
  off = align_up(off + 4 * (batch + 1), 16);  // kv_indptr
  off = align_up(off + 4 * batch, 16);        // kv_len
  off = align_up(off + 4 * (rows + 1), 16);   // merge_indptr
  off = align_up(off + 4 * n_merge, 32);      // merge_rows
  off = align_up(off + 4 * (batch + 1), 16);  // mask_indptr
  return align_up(off, kAlign);
}

int64_t partial_bytes_for(int64_t n_partials, int64_t hq, int64_t d) {
  return align_up(4 * n_partials * hq, kAlign) + align_up(4 * n_partials * hq * d, kAlign);
}

}  // namespace

extern "C" size_t fi_workspace_bytes(int32_t max_batch, int32_t max_total_rows,
                                     int32_t num_qo_heads, int32_t head_dim,
                                     int32_t max_kv_chunks) {
  if (max_batch < 0 || max_total_rows < 0 || num_qo_heads <= 0 || head_dim <= 0) return 0;
  int64_t chunks = std::max<int32_t>(max_kv_chunks, 1);
  int64_t rows = max_total_rows;
  // every tile holds >= 1 token, so tiles <= rows; items <= tiles * chunks * heads
  int64_t items = std::max<int64_t>(rows, 1) * chunks * num_qo_heads;
  int64_t partials = chunks > 1 ? rows * chunks : 0;
  return static_cast<size_t>(meta_bytes_for(max_batch, rows, rows, items) +
                             partial_bytes_for(partials, num_qo_heads, head_dim));
}

extern "C" fi_status fi_plan_create(fi_plan_t* out, void* workspace, size_t workspace_bytes,
                                    int32_t enable_graph_capture, int32_t max_batch,
                                    int32_t max_total_rows) {
  if (!out) return fail(FI_ERR_INVALID_ARG, "plan: output pointer is NULL");
  *out = nullptr;
  if (max_batch < 0 || max_total_rows < 0)
    return fail(FI_ERR_INVALID_ARG, "plan_create: max_batch=%d max_total_rows=%d must be >= 0",
                max_batch, max_total_rows);
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0)
    return fail(FI_ERR_INVALID_ARG, "plan_create: workspace must be 256-byte aligned");
  if (workspace && enable_graph_capture &&
      static_cast<int64_t>(workspace_bytes) < meta_bytes_for(max_batch, max_total_rows, 0, 0))
    return fail(FI_ERR_CAPACITY, "plan_create: workspace_bytes=%zu cannot hold the metadata of "
                "max_batch=%d max_total_rows=%d", workspace_bytes, max_batch, max_total_rows);
  fi_plan_s* p = new (std::nothrow) fi_plan_s();
  if (!p) return fail(FI_ERR_INVALID_ARG, "plan_create: out of host memory");
  p->ws = workspace;
  p->ws_bytes = workspace_bytes;
  p->host_only = (workspace == nullptr);
  p->graph = enable_graph_capture != 0;
  p->max_batch = max_batch;
  p->max_total_rows = max_total_rows;
  if (!p->host_only) {
    int n = device_sm_count();
    if (n <= 0) {
      delete p;
      return fail(FI_ERR_CUDA, "plan_create: no CUDA device (%s)",
                  cudaGetErrorString(cudaGetLastError()));
    }
    p->num_sms = n;
    cudaEvent_t* evs[4] = {&p->upload_done, &p->run_done, &p->staged[0], &p->staged[1]};
    for (cudaEvent_t* e : evs) {
      if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) {
        for (cudaEvent_t* f : evs)
          if (*f) cudaEventDestroy(*f);
        delete p;
        return fail(FI_ERR_CUDA, "plan_create: cudaEventCreate failed");
      }
    }
  }
  *out = p;
  return ok();
}

extern "C" void fi_plan_destroy(fi_plan_t p) {
  if (!p) return;
  for (int i = 0; i < 2; ++i) {
    if (p->staged_pending[i]) cudaEventSynchronize(p->staged[i]);
    if (p->staged[i]) cudaEventDestroy(p->staged[i]);
    if (p->staging[i]) cudaFreeHost(p->staging[i]);
  }
  if (p->upload_done) cudaEventDestroy(p->upload_done);
  if (p->run_done) cudaEventDestroy(p->run_done);
  delete p;
}

namespace {

// The short-query kernel (kDecode) takes every request of at most 16 packed
// rows (one tile) on its tensor-core consumer when the group and page size allow, and
// decode on its CUDA-core consumer otherwise (groups 1, 2, 4).
// Requests of up to kShortRowsMax packed rows go to the short-query kernel
// too: 17 to 32 rows in one 32-row tile of its pair consumer (two M tiles,
// one read of the keys).
constexpr int64_t kShortRowsMax = 32;

int choose_kernel(int32_t q_len_per_req, int32_t g, int64_t max_rows_per_req, int32_t d,
                  int32_t page_size, bool masked) {
  if (max_rows_per_req <= kShortRowsMax && fi::decode_mma_supports(d, page_size, g))
    return fi::kDecode;
  if (masked) {  // the custom mask is read by every kernel
    if (max_rows_per_req > kShortRowsMax && fi::prefill_tc_supports(d, page_size, g))
      return fi::kPrefillM128;
    if (max_rows_per_req <= 16 && g <= 16) return fi::kPrefillM16;
    return g <= 64 ? fi::kPrefillM64 : -1;
  }
  if (q_len_per_req == 1 && fi::decode_shuffle_supports(d, g)) return fi::kDecode;
  // above the short-query kernel's rows: the tcgen05 kernel wherever its TMA
  // boxes fit (head_dim 64 or 128, page sizes that are multiples of 8); the
  // mma.sync kernels keep page sizes 1..7 and other odd sizes
  if (max_rows_per_req > kShortRowsMax && fi::prefill_tc_supports(d, page_size, g))
    return fi::kPrefillM128;
  if (max_rows_per_req <= 16 && g <= 16) return fi::kPrefillM16;
  if (g <= 64) return fi::kPrefillM64;
  if (fi::prefill_tc_supports(d, page_size, g)) return fi::kPrefillM128;
  return -1;
}

int tile_rows_of(int kernel, int g, int64_t max_rows_per_req, int32_t d, int32_t page_size) {
  switch (kernel) {
    case fi::kDecode:
      // tensor-core consumer: one row half (8 rows) when every request fits,
      // else two; CUDA-core consumer: the G heads of one token
      if (!fi::decode_mma_supports(d, page_size, g)) return g;
      if (max_rows_per_req <= 8 && g <= 8) return (8 / g) * g;
      return max_rows_per_req <= 16 ? (16 / g) * g : (32 / g) * g;
    case fi::kPrefillM16: return (16 / g) * g;
    case fi::kPrefillM64: return (64 / g) * g;
    case fi::kPrefillM128: return 2 * ((128 / g) * g);  // two 128-row Q tiles
  }
  return 0;
}

struct Tile {
  int32_t b, row0, rows, lo, hi, lk;
  int32_t first_token;  // global token index of the tile's first query row
  int32_t n_tokens;
};

// Build a complete plan into `ns` without touching the plan object.
// ragged: kv_indptr_h holds each request's first K/V row (contiguous K/V),
// last_page_len_h is unused, and page_size is kRaggedPage (one logical page).
constexpr int32_t kRaggedPage = 1 << 30;
// A short-query item's fixed cost (its q rows, the consumer warps' merge, the
// output writes) in keys of the same item: the schedule weighs such an item
// as (live keys + kItemKeys) x rows. Measured on the batch-32 verify kernel
// against a weight of live x rows + 64: 128 took it from 66.7 to 64.7 us (no
// CTA with five items; decode and tree verify unchanged), 384 gave 65.7. The
// prefill kernels keep live x rows + 64.
constexpr int64_t kItemKeys = 128;

fi_status build_plan(const fi_plan_s& P, const int32_t* qo_indptr_h, const int32_t* kv_indptr_h,
                     const int32_t* last_page_len_h, int32_t batch, int32_t page_size,
                     int32_t hq, int32_t hk, int32_t d, int32_t causal, int32_t window_left,
                     fi_dtype dtype, int32_t q_len_per_req, int32_t force_kv_chunks,
                     bool ragged, const int32_t* mask_indptr_h, PlanState& ns) {
  // ---- argument validation, before anything is written [P2 "Review notes"]
  if (batch < 0) return fail(FI_ERR_INVALID_ARG, "plan: batch=%d must be >= 0", batch);
  if (batch > 0 && (!kv_indptr_h || (!ragged && !last_page_len_h)))
    return fail(FI_ERR_INVALID_ARG, "plan: kv_indptr and last_page_len must be non-NULL");
  if (page_size < 1) return fail(FI_ERR_INVALID_ARG, "plan: page_size=%d must be >= 1", page_size);
  // [P3 "GQA head divisibility"]: refuse zero kv heads and a group that does not divide
  if (hk <= 0 || hq <= 0 || hq % hk != 0)
    return fail(FI_ERR_GQA_INDIVISIBLE,
                "plan: num_qo_heads=%d is not a multiple of num_kv_heads=%d", hq, hk);
  if (d != 64 && d != 128)
    return fail(FI_ERR_UNSUPPORTED, "plan: head_dim=%d (built: 64, 128)", d);
  if (dtype != FI_F16 && dtype != FI_BF16)
    return fail(FI_ERR_UNSUPPORTED, "plan: dtype=%d (built: FI_F16, FI_BF16)", (int)dtype);
  if (window_left < -1)
    return fail(FI_ERR_INVALID_ARG, "plan: window_left=%d must be -1 or >= 0", window_left);
  if (q_len_per_req < 0)
    return fail(FI_ERR_INVALID_ARG, "plan: q_len_per_req=%d must be >= 0", q_len_per_req);
  if (force_kv_chunks < 0 || force_kv_chunks > 4096)
    return fail(FI_ERR_INVALID_ARG, "plan: force_kv_chunks=%d must be in [0, 4096]",
                force_kv_chunks);
  if (q_len_per_req >= 1 && qo_indptr_h)
    return fail(FI_ERR_INVALID_ARG, "plan: qo_indptr must be NULL when q_len_per_req=%d >= 1 "
                "(it is q_len_per_req * b)", q_len_per_req);
  if (q_len_per_req == 0 && batch > 0 && !qo_indptr_h)
    return fail(FI_ERR_INVALID_ARG, "plan: qo_indptr is NULL for a prefill plan");
  // the verify adapter makes the mask causal [P2 "What changed"]
  const int32_t eff_causal = (q_len_per_req > 1) ? 1 : (causal ? 1 : 0);
  const int32_t g = hq / hk;

  ns = PlanState();
  ns.batch = batch; ns.page_size = page_size; ns.hq = hq; ns.hk = hk; ns.d = d;
  ns.causal = eff_causal; ns.window_left = window_left; ns.dtype = dtype;
  ns.ragged = ragged ? 1 : 0;
  ns.q_len_per_req = q_len_per_req; ns.group = g;
  ns.qo_indptr.resize(batch + 1);
  ns.kv_indptr.resize(batch + 1);
  ns.kv_len.resize(batch);
  int64_t qacc = 0;
  ns.qo_indptr[0] = 0;
  for (int32_t b = 0; b <= batch; ++b) {
    int64_t v = (q_len_per_req >= 1) ? int64_t(q_len_per_req) * b
                                      : (qo_indptr_h ? int64_t(qo_indptr_h[b]) : 0);
    if (b == 0 && v != 0) return fail(FI_ERR_INVALID_ARG, "plan: qo_indptr[0]=%lld must be 0", (long long)v);
    if (v < qacc) return fail(FI_ERR_INVALID_ARG, "plan: qo_indptr decreases at b=%d", b);
    if (v > INT32_MAX) return fail(FI_ERR_INVALID_ARG, "plan: total query rows overflow int32");
    qacc = v;
    ns.qo_indptr[b] = static_cast<int32_t>(v);
  }
  ns.total_rows = ns.qo_indptr[batch];
  int64_t max_rows_per_req = 0;
  for (int32_t b = 0; b <= batch; ++b) {
    int32_t v = kv_indptr_h ? kv_indptr_h[b] : 0;
    if (b == 0 && v != 0) return fail(FI_ERR_INVALID_ARG, "plan: kv_indptr[0]=%d must be 0", v);
    if (b > 0 && v < ns.kv_indptr[b - 1])
      return fail(FI_ERR_INVALID_ARG, "plan: kv_indptr decreases at b=%d", b);
    ns.kv_indptr[b] = v;
  }
  ns.kv_indices_len = ns.kv_indptr[batch];
  for (int32_t b = 0; b < batch; ++b) {
    // [P2 "Review notes"]: kv_len from the page metadata (paged_kv_t::get_length)
    int64_t pages = int64_t(ns.kv_indptr[b + 1]) - ns.kv_indptr[b];
    int64_t lk = 0;
    if (ragged) {
      lk = pages;  // rows of the contiguous K/V
    } else if (pages > 0) {
      int32_t last = last_page_len_h[b];
      if (last < 1 || last > page_size)
        return fail(FI_ERR_INVALID_ARG, "plan: last_page_len[%d]=%d outside [1, page_size=%d]",
                    b, last, page_size);
      lk = (pages - 1) * page_size + last;
    }
    if (lk > INT32_MAX / 2) return fail(FI_ERR_INVALID_ARG, "plan: kv_len of request %d too long", b);
    int64_t lq = int64_t(ns.qo_indptr[b + 1]) - ns.qo_indptr[b];
    // [P2 "Review notes"]: a causal request whose KV is shorter than its query
    // rows would be masked against a range shorter than the query; refuse it.
    if (eff_causal && lk < lq)
      return fail(FI_ERR_KV_SHORTER_THAN_Q,
                  "plan: request %d has kv_len=%lld (from kv_indptr/last_page_len) < qo_len=%lld "
                  "under the causal mask", b, (long long)lk, (long long)lq);
    ns.kv_len[b] = static_cast<int32_t>(lk);
    max_rows_per_req = std::max<int64_t>(max_rows_per_req, lq * g);
  }
  // custom mask segments: byte offsets, each long enough for its Lq x Lk bits
  ns.masked = mask_indptr_h ? 1 : 0;
  ns.mask_indptr.assign(batch + 1, 0);
  if (mask_indptr_h) {
    if (mask_indptr_h[0] < 0) return fail(FI_ERR_INVALID_ARG, "plan: mask_indptr[0] < 0");
    for (int32_t b = 0; b < batch; ++b) {
      const int64_t lq = int64_t(ns.qo_indptr[b + 1]) - ns.qo_indptr[b];
      const int64_t need = (lq * ns.kv_len[b] + 7) / 8;
      const int64_t have = int64_t(mask_indptr_h[b + 1]) - mask_indptr_h[b];
      if (have < need)
        return fail(FI_ERR_INVALID_ARG, "plan: mask_indptr gives request %d %lld bytes, its %lld x "
                    "%d mask needs %lld", b, (long long)have, (long long)lq, ns.kv_len[b],
                    (long long)need);
    }
    for (int32_t b = 0; b <= batch; ++b) ns.mask_indptr[b] = mask_indptr_h[b];
    ns.mask_bytes = mask_indptr_h[batch];
  }

  // ---- graph-mode capacities and frozen shape [P2 "Architecture / design notes"]
  if (P.graph) {
    if (batch > P.max_batch)
      return fail(FI_ERR_CAPACITY, "plan: batch=%d exceeds the graph capacity max_batch=%d",
                  batch, P.max_batch);
    if (ns.total_rows > P.max_total_rows)
      return fail(FI_ERR_CAPACITY, "plan: total rows=%d exceed the graph capacity "
                  "max_total_rows=%d", ns.total_rows, P.max_total_rows);
    // the kernel cannot follow per-batch lengths once captured: bound them
    max_rows_per_req = (q_len_per_req >= 1) ? int64_t(q_len_per_req) * g
                                             : int64_t(P.max_total_rows) * g;
  }
  ns.kernel = choose_kernel(q_len_per_req, g, max_rows_per_req, d, page_size, mask_indptr_h != nullptr);
  if (ns.kernel < 0)
    return fail(FI_ERR_UNSUPPORTED, "plan: GQA group %d is larger than the widest tile", g);
  if (P.graph && P.frozen) {
    const char* field = nullptr;
    int32_t want = 0, got = 0;
    if (q_len_per_req != P.fz_qlpr) { field = "q_len_per_req"; want = P.fz_qlpr; got = q_len_per_req; }
    else if (hq != P.fz_hq) { field = "num_qo_heads"; want = P.fz_hq; got = hq; }
    else if (hk != P.fz_hk) { field = "num_kv_heads"; want = P.fz_hk; got = hk; }
    else if (d != P.fz_d) { field = "head_dim"; want = P.fz_d; got = d; }
    else if (dtype != P.fz_dtype) { field = "dtype"; want = P.fz_dtype; got = dtype; }
    else if (page_size != P.fz_page) { field = "page_size"; want = P.fz_page; got = page_size; }
    else if (int32_t(ragged) != P.fz_ragged) { field = "ragged"; want = P.fz_ragged; got = ragged; }
    else if (ns.masked != P.fz_masked) { field = "masked"; want = P.fz_masked; got = ns.masked; }
    else if (ns.kernel != P.fz_kernel) { field = "kernel"; want = P.fz_kernel; got = ns.kernel; }
    if (field)
      return fail(FI_ERR_CAPACITY, "plan: %s is frozen at %d by the first graph-mode plan, got %d",
                  field, want, got);
  }
  ns.tile_rows = tile_rows_of(ns.kernel, g, max_rows_per_req, d, page_size);

  // ---- tiles and their live key ranges
  std::vector<Tile> tiles;
  int64_t total_len = 0, max_len = 0;
  for (int32_t b = 0; b < batch; ++b) {
    const int64_t lq = int64_t(ns.qo_indptr[b + 1]) - ns.qo_indptr[b];
    const int64_t lk = ns.kv_len[b];
    for (int64_t row0 = 0; row0 < lq * g; row0 += ns.tile_rows) {
      const int64_t rows = std::min<int64_t>(ns.tile_rows, lq * g - row0);
      const int64_t i0 = row0 / g, i1 = (row0 + rows) / g - 1;
      int64_t hi = eff_causal ? std::min<int64_t>(lk, i1 + lk - lq + 1) : lk;
      int64_t lo = window_left >= 0 ? std::max<int64_t>(0, lk - lq + i0 - window_left) : 0;
      hi = std::max<int64_t>(hi, 0);
      if (lo > hi) lo = hi;
      Tile t{b, int32_t(row0), int32_t(rows), int32_t(lo), int32_t(hi), int32_t(lk),
             int32_t(ns.qo_indptr[b] + i0), int32_t(i1 - i0 + 1)};
      tiles.push_back(t);
      total_len += hi - lo;
      max_len = std::max<int64_t>(max_len, hi - lo);
    }
  }

  // ---- KV split
  const int ctas_per_sm =
      std::max(1, fi::kernel_ctas_per_sm(ns.kernel, d, g, dtype == FI_BF16, page_size));
  const int64_t grid_cap = int64_t(P.num_sms) * ctas_per_sm;
  const int64_t avail = P.host_only ? INT64_MAX / 4 : int64_t(P.ws_bytes);
  auto item_cost = [&](int64_t live, int64_t rows) {
    return ns.kernel == fi::kDecode ? (live + kItemKeys) * rows : live * rows + 64;
  };
  auto count_for = [&](int64_t chunk_len, int64_t* n_items, int64_t* n_partials) {
    int64_t items = 0, partials = 0;
    for (const Tile& t : tiles) {
      int64_t n = 1;
      if (force_kv_chunks > 0) n = force_kv_chunks;
      else if (chunk_len > 0 && t.hi - t.lo > chunk_len) n = (t.hi - t.lo + chunk_len - 1) / chunk_len;
      items += n * hk;
      if (n > 1) partials += n * t.n_tokens;
    }
    *n_items = items;
    *n_partials = partials;
  };
  auto fits = [&](int64_t n_items, int64_t n_partials, int64_t n_merge) {
    return meta_bytes_for(batch, ns.total_rows, n_merge, n_items) +
               partial_bytes_for(n_partials, hq, d) <= avail;
  };
  int64_t chunk_len = 0;  // 0 = no split
  if (force_kv_chunks == 0 && !tiles.empty()) {
    const int64_t min_chunk = 256;
    const int64_t units = int64_t(tiles.size()) * hk;
    // split when the tiles alone cannot keep every SM busy and balanced:
    // aim at ~2 items per resident CTA (measured against 4 and 8: fewer,
    // longer items win on decode and verify once the longest-first schedule
    // balances them), no chunk shorter than min_chunk keys
    int64_t want = (total_len * hk + 2 * grid_cap - 1) / (2 * grid_cap);
    want = std::max<int64_t>(min_chunk, (want + 63) / 64 * 64);
    if (max_len > want && units < 4 * grid_cap * 4) {
      chunk_len = want;
      // A few long units over many CTAs balance badly when their chunk count
      // does not fit the grid (8 units of 5 chunks on 19 bundles: 2 bundles
      // in 19 carry a third). When the units number at most half the bins,
      // try the chunk lengths that cut the longest unit into k0 - 3 .. k0 + 4
      // pieces and keep the one whose static schedule ends first, counting
      // each split item's partial state (written, then read by the merge:
      // about 2 x rows keys' worth of traffic). With more units the longest-
      // first schedule balances them already, and the search (about 3 us per
      // candidate on 200 groups) is skipped.
      auto makespan = [&](int64_t cl) {
        std::vector<int64_t> costs;
        for (const Tile& t : tiles) {
          const int64_t len = t.hi - t.lo;
          const int64_t n = (cl > 0 && len > cl) ? (len + cl - 1) / cl : 1;
          for (int64_t c = 0; c < n; ++c) {
            const int64_t live = n > 1 ? std::min<int64_t>(cl, len - c * cl) : len;
            costs.push_back(item_cost(live, t.rows) + (n > 1 ? 2 * int64_t(t.rows) * t.rows : 0));
          }
        }
        std::sort(costs.begin(), costs.end(), std::greater<int64_t>());
        const int64_t n_all = int64_t(costs.size()) * hk;
        const int64_t Gs = std::max<int64_t>(1, P.graph ? grid_cap : std::min<int64_t>(n_all, grid_cap));
        const int64_t per = (Gs % hk == 0) ? hk : 1;  // CTAs that take one group together
        const int64_t reps = hk / per;                 // takes per group
        std::vector<int64_t> heap(size_t(Gs / per), 0);  // min-heap of bin loads
        int64_t worst = 0;
        for (int64_t c : costs)
          for (int64_t r = 0; r < reps; ++r) {
            std::pop_heap(heap.begin(), heap.end(), std::greater<int64_t>());
            heap.back() += c;
            worst = std::max(worst, heap.back());
            std::push_heap(heap.begin(), heap.end(), std::greater<int64_t>());
          }
        return worst;
      };
      const bool bundled = grid_cap % hk == 0;
      const int64_t bins = bundled ? grid_cap / hk : grid_cap;
      const int64_t units_b = int64_t(tiles.size()) * (bundled ? 1 : hk);
      const bool few = 2 * units_b <= bins;
      int64_t best = few ? makespan(want) : 0;
      const int64_t k0 = (max_len + want - 1) / want;
      for (int64_t k = std::max<int64_t>(2, k0 - 3); few && k <= k0 + 4; ++k) {
        const int64_t cl = ((max_len + k - 1) / k + 63) / 64 * 64;
        if (cl < min_chunk || cl >= max_len || cl == chunk_len) continue;
        const int64_t m = makespan(cl);
        if (m < best) {
          best = m;
          chunk_len = cl;
        }
      }
    }
    // grow the chunks until the partial states fit the workspace
    while (chunk_len > 0) {
      int64_t ni, np;
      count_for(chunk_len, &ni, &np);
      if (fits(ni, np, ns.total_rows)) break;
      chunk_len *= 2;
      if (chunk_len >= max_len) chunk_len = 0;
    }
  }
  {
    int64_t ni, np;
    count_for(chunk_len, &ni, &np);
    if (ni > INT32_MAX / 2 || np > INT32_MAX / 2)
      return fail(FI_ERR_CAPACITY, "plan: %lld work items exceed the planner's range", (long long)ni);
    if (!fits(ni, np, ns.total_rows))
      return fail(FI_ERR_CAPACITY, "plan: workspace_bytes=%zu < %lld needed for %lld items and "
                  "%lld partial states", P.ws_bytes,
                  (long long)(meta_bytes_for(batch, ns.total_rows, ns.total_rows, ni) +
                              partial_bytes_for(np, hq, d)),
                  (long long)ni, (long long)np);
  }

  // ---- work items, partial slots and the merge index
  ns.merge_indptr.assign(ns.total_rows + 1, 0);
  std::vector<int32_t> merge_count(ns.total_rows, 0);
  int32_t partial_cursor = 0;
  int32_t max_chunks = 1;
  int64_t G = 0;  // the grid

  // Balanced spans (when the plan splits keys): the live keys of all tiles,
  // laid end to end, are cut into one contiguous span per bundle of Hk CTAs
  // (one CTA per kv head), every span of about the same cost,
  // (keys + kSpanItemKeys) x rows per piece. A bundle takes the rest of the
  // tile it starts in and as much of the next ones as its share allows, so
  // the CTAs end at about the same time: a longest-first schedule of
  // fixed-length chunks left 5% of the CTA time idle on the batch-32 verify
  // (and fewer, longer items cost fewer item ends and fewer partial states).
  // Cuts fall on multiples of kCut keys and no piece is shorter than
  // kMinPiece keys.
  auto schedule_spans = [&]() -> bool {
    // Cut granularity (a stage of the short-query kernel, a key tile of the
    // tcgen05 kernel), the shortest piece, and an item's fixed cost in keys.
    // Short-query kernel: a per-item timeline of the batch-32 verify and
    // batch-64 decode runs (item end times against their keys) put the fixed
    // cost near zero once the producer runs ahead across items; 32 keys keep
    // pieces from being cut for nothing. tcgen05 kernel: an item reloads its
    // Q tile and writes a 64 KB partial state, about 128 keys' worth.
    const bool tc = ns.kernel == fi::kPrefillM128;
    const int64_t kCut = tc ? 128 : 64;
    const int64_t kMinPiece = tc ? 256 : 64;
    const int64_t kSpanItemKeys = tc ? 128 : 32;
    // A piece's rows as the kernel pays them: the tcgen05 kernel computes a
    // whole 128-row Q tile whatever its live rows (a request's last tile of 46
    // rows costs half a two-tile piece, not a fifth); the short-query kernel
    // pays by rows.
    auto wrows = [&](const Tile& t) -> double {
      return tc ? (t.rows > 128 ? 256.0 : 128.0) : double(t.rows);
    };
    if (grid_cap % hk != 0) return false;
    const int64_t B = grid_cap / hk;
    if (B < 2) return false;
    double total = 0;
    for (const Tile& t : tiles) total += double(t.hi - t.lo + kSpanItemKeys) * wrows(t);
    struct Piece { int32_t bundle, tile, kb, ke; };
    std::vector<Piece> pieces, trial;
    pieces.reserve(tiles.size() + size_t(B));
    trial.reserve(tiles.size() + size_t(B));
    // One walk: every bundle takes up to `share` of cost from its own start
    // (a piece that starts costs kSpanItemKeys x rows on top of its keys); cuts
    // round to multiples of kCut keys, a remainder shorter than kMinPiece keys
    // stays with its piece, and a bundle with room for less than kMinPiece
    // keys ends there. Returns the bundles used, or B + 1 once it needs more.
    // share >= (kSpanItemKeys + 2 kMinPiece) x the largest rows, so a fresh
    // bundle always takes a piece and every step advances.
    auto walk = [&](double share, std::vector<Piece>& out) {
      out.clear();
      int64_t bundle = 0;
      double room = share;
      for (size_t ti = 0; ti < tiles.size() && bundle < B; ++ti) {
        const Tile& t = tiles[ti];
        const double rows = wrows(t);
        int64_t pos = t.lo;
        for (;;) {
          const double fit = room / rows - double(kSpanItemKeys);  // keys a piece here may take
          const int64_t rest = t.hi - pos;
          if (fit >= double(rest - kMinPiece)) {
            out.push_back({int32_t(bundle), int32_t(ti), int32_t(pos), int32_t(t.hi)});
            room -= double(rest + kSpanItemKeys) * rows;
            break;
          }
          if (fit < double(kMinPiece)) {  // too little room: the next bundle starts here
            if (++bundle >= B) break;
            room = share;
            continue;
          }
          int64_t cut = (pos + int64_t(fit) + kCut / 2) / kCut * kCut;
          cut = std::max<int64_t>(cut, pos + kMinPiece);
          out.push_back({int32_t(bundle), int32_t(ti), int32_t(pos), int32_t(cut)});
          pos = cut;
          if (++bundle >= B) break;
          room = share;
        }
      }
      if (bundle >= B) return B + 1;
      return out.empty() ? int64_t(1) : int64_t(out.back().bundle) + 1;
    };
    // the smallest share whose walk fits the B bundles (bisection; each walk
    // is tiles + bundles steps)
    double max_rows = 1;
    for (const Tile& t : tiles) max_rows = std::max(max_rows, wrows(t));
    double lo_s = std::max(total / double(B), double(kSpanItemKeys + 2 * kMinPiece) * max_rows);
    double hi_s = 2.0 * lo_s;
    for (int iter = 0; iter < 24; ++iter) {
      const double mid = 0.5 * (lo_s + hi_s);
      if (walk(mid, trial) <= B) hi_s = mid;
      else lo_s = mid;
    }
    if (walk(hi_s, pieces) > B) return false;
    // pieces per tile -> chunk counts, partial slots; refuse (fall back to the
    // chunked schedule) when the partial states do not fit the workspace
    std::vector<int32_t> n_of(tiles.size(), 0), base_of(tiles.size(), -1), next(tiles.size(), 0);
    for (const Piece& pc : pieces) n_of[size_t(pc.tile)]++;
    int64_t np = 0;
    for (size_t ti = 0; ti < tiles.size(); ++ti)
      if (n_of[ti] > 1) np += int64_t(n_of[ti]) * tiles[ti].n_tokens;
    const int64_t used = pieces.empty() ? 1 : int64_t(pieces.back().bundle) + 1;
    const int64_t g_spans = P.graph ? grid_cap : used * hk;
    std::vector<int32_t> per_bundle(size_t(used), 0);
    for (const Piece& pc : pieces) per_bundle[size_t(pc.bundle)]++;
    int32_t rounds = 0;
    for (int32_t c : per_bundle) rounds = std::max(rounds, c);
    const int64_t ni = int64_t(rounds) * g_spans;
    if (np > INT32_MAX / 2 || ni > INT32_MAX / 2 || !fits(ni, np, ns.total_rows)) return false;
    for (size_t ti = 0; ti < tiles.size(); ++ti) {
      const Tile& t = tiles[ti];
      max_chunks = std::max(max_chunks, n_of[ti]);
      if (n_of[ti] > 1) {
        base_of[ti] = partial_cursor;
        partial_cursor += n_of[ti] * t.n_tokens;
        for (int32_t k = 0; k < t.n_tokens; ++k) merge_count[size_t(t.first_token + k)] = n_of[ti];
      }
    }
    WorkItem pad{};
    pad.b = -1;
    ns.items.assign(size_t(ni), pad);
    std::fill(per_bundle.begin(), per_bundle.end(), 0);
    for (const Piece& pc : pieces) {
      const Tile& t = tiles[size_t(pc.tile)];
      const int32_t n = n_of[size_t(pc.tile)];
      WorkItem it{};
      it.b = t.b;
      it.row0 = t.row0;
      it.kv_begin = pc.kb;
      it.kv_end = pc.ke;
      it.chunk = n > 1 ? next[size_t(pc.tile)]++ : -1;
      it.num_chunks = n;
      it.partial_base = base_of[size_t(pc.tile)];
      const int64_t slot = per_bundle[size_t(pc.bundle)]++;
      for (int32_t h = 0; h < hk; ++h) {
        it.kv_head = h;
        ns.items[size_t(slot * g_spans + int64_t(pc.bundle) * hk + h)] = it;
      }
    }
    G = g_spans;
    return true;
  };
  const bool spans = (ns.kernel == fi::kDecode || ns.kernel == fi::kPrefillM128) &&
                     force_kv_chunks == 0 && chunk_len > 0 && schedule_spans();
  if (!spans) {
    // Items are made per (tile, chunk) group - one per kv head, all of the same
    // cost - and the groups are sorted by cost, longest first.
    struct Group { int64_t cost; WorkItem it; };
    std::vector<Group> groups;
    {
      size_t n_est = 0;
      for (const Tile& t : tiles) {
        int64_t n = 1;
        if (force_kv_chunks > 0) n = force_kv_chunks;
        else if (chunk_len > 0 && t.hi - t.lo > chunk_len) n = (t.hi - t.lo + chunk_len - 1) / chunk_len;
        n_est += size_t(n);
      }
      groups.reserve(n_est);
    }
    for (const Tile& t : tiles) {
      int64_t n = 1;
      if (force_kv_chunks > 0) n = force_kv_chunks;
      else if (chunk_len > 0 && t.hi - t.lo > chunk_len) n = (t.hi - t.lo + chunk_len - 1) / chunk_len;
      max_chunks = std::max<int32_t>(max_chunks, int32_t(n));
      const int32_t base = (n > 1) ? partial_cursor : -1;
      if (n > 1) {
        partial_cursor += int32_t(n) * t.n_tokens;
        for (int32_t k = 0; k < t.n_tokens; ++k) merge_count[t.first_token + k] = int32_t(n);
      }
      for (int64_t c = 0; c < n; ++c) {
        int64_t kb, ke;
        if (force_kv_chunks > 0) {  // even cut of the full key range [0, Lk)
          kb = int64_t(t.lk) * c / n;
          ke = int64_t(t.lk) * (c + 1) / n;
        } else if (n > 1) {         // chunk_len cut of the live range
          kb = t.lo + c * chunk_len;
          ke = std::min<int64_t>(t.hi, kb + chunk_len);
        } else {
          kb = t.lo;
          ke = t.hi;
        }
        const int64_t live = std::max<int64_t>(0, std::min<int64_t>(ke, t.hi) - std::max<int64_t>(kb, t.lo));
        Group gr;
        gr.cost = item_cost(live, t.rows);
        if (ns.kernel == fi::kPrefillM128) {
          // The tcgen05 kernel pays per 128-key tile, counted from the K/V box
          // boundary at or below the first live key, at a fixed 128 rows per
          // Q tile: a tile costs twice as much with two Q tiles (more than 128
          // rows) as with one (a one-tile item spreads its key tiles over both
          // softmax warpgroups); an item's start and epilogue cost about two
          // such steps. Weighing live keys by rows instead left the longest
          // CTA of the batch-16 prefill about 4% above the mean.
          const int64_t klo = std::max<int64_t>(kb, t.lo), khi = std::min<int64_t>(ke, t.hi);
          const int64_t box = std::gcd<int64_t>(page_size, 128);
          const int64_t n_kt = khi > klo ? (khi - klo / box * box + 127) / 128 : 0;
          gr.cost = (n_kt * (t.rows > 128 ? 2 : 1) + 2) * 1024;
        }
        gr.it.b = t.b; gr.it.kv_head = 0; gr.it.row0 = t.row0;
        gr.it.kv_begin = int32_t(kb); gr.it.kv_end = int32_t(ke);
        gr.it.chunk = (n > 1) ? int32_t(c) : -1;
        gr.it.num_chunks = int32_t(n);
        gr.it.partial_base = base;
        groups.push_back(gr);
      }
    }
    std::stable_sort(groups.begin(), groups.end(),
                     [](const Group& a, const Group& b) { return a.cost > b.cost; });
    // Static longest-processing-time schedule for the persistent grid: groups,
    // longest first, go to the least-loaded bundle of Hk CTAs (one item per CTA
    // of the bundle; a bundle is one CTA when Hk does not divide the grid),
    // found with a binary min-heap of bundle loads; CTA c then finds its list at
    // positions c, c + grid, ... (padded with items whose request is -1, which
    // every kernel skips).
    const int64_t n_all = int64_t(groups.size()) * hk;
    G = std::max<int64_t>(1, P.graph ? grid_cap : std::min<int64_t>(n_all, grid_cap));
    const int32_t bundle = (G % hk == 0) ? hk : 1;
    const int32_t n_bundles = int32_t(G / bundle);
    {
      std::vector<int64_t> load(static_cast<size_t>(n_bundles), 0);
      std::vector<int32_t> heap(static_cast<size_t>(n_bundles));  // heap-ordered by (load, id)
      for (int32_t c = 0; c < n_bundles; ++c) heap[size_t(c)] = c;
      auto less = [&](int32_t a, int32_t b) {
        return load[size_t(a)] != load[size_t(b)] ? load[size_t(a)] < load[size_t(b)] : a < b;
      };
      auto take = [&](int64_t cost) {  // least-loaded bundle gets `cost`
        const int32_t c = heap[0];
        load[size_t(c)] += cost;
        size_t k = 0;
        const size_t n = size_t(n_bundles);
        for (;;) {
          size_t l = 2 * k + 1, r = l + 1, m = k;
          if (l < n && less(heap[l], heap[m])) m = l;
          if (r < n && less(heap[r], heap[m])) m = r;
          if (m == k) break;
          std::swap(heap[k], heap[m]);
          k = m;
        }
        return c;
      };
      std::vector<int32_t> cta_of(static_cast<size_t>(n_all));
      std::vector<int32_t> count(static_cast<size_t>(G), 0);
      int64_t i = 0;
      for (const Group& gr : groups) {
        if (bundle == hk) {
          const int32_t c0 = take(gr.cost) * hk;
          for (int32_t h = 0; h < hk; ++h, ++i) {
            cta_of[size_t(i)] = c0 + h;
            count[size_t(c0 + h)]++;
          }
        } else {
          for (int32_t h = 0; h < hk; ++h, ++i) {
            const int32_t c = take(gr.cost);
            cta_of[size_t(i)] = c;
            count[size_t(c)]++;
          }
        }
      }
      int32_t rounds = 0;
      for (int32_t c : count) rounds = std::max(rounds, c);
      WorkItem pad{};
      pad.b = -1;
      ns.items.assign(size_t(rounds) * size_t(G), pad);
      std::vector<int32_t> next(static_cast<size_t>(G), 0);
      i = 0;
      for (const Group& gr : groups) {
        for (int32_t h = 0; h < hk; ++h, ++i) {
          const int32_t c = cta_of[size_t(i)];
          WorkItem it = gr.it;
          it.kv_head = h;
          ns.items[size_t(next[size_t(c)]++) * size_t(G) + size_t(c)] = it;
        }
      }
    }
  }
  // A captured kernel keeps its grid: an empty graph-mode plan still holds a
  // grid's worth of (padding) items, which the short-query kernel's CTAs load
  // before they read the item count.
  if (P.graph && ns.items.empty()) {
    WorkItem pad{};
    pad.b = -1;
    ns.items.assign(size_t(std::max<int64_t>(G, 1)), pad);
  }
  // every item repeats its request's metadata
  for (WorkItem& it : ns.items) {
    if (it.b < 0) continue;
    it.tok0 = ns.qo_indptr[size_t(it.b)];
    it.lq = ns.qo_indptr[size_t(it.b) + 1] - it.tok0;
    it.lk = ns.kv_len[size_t(it.b)];
    it.kv_start = ns.kv_indptr[size_t(it.b)];
    it.mask_base = ns.mask_indptr[size_t(it.b)];
  }
  if (partial_cursor > 0) {  // else merge_indptr stays all zero (no row is split)
    int32_t acc = 0;  // running sum in a register: no store-to-load chain
    for (int32_t t = 0; t < ns.total_rows; ++t) {
      acc += merge_count[t];
      ns.merge_indptr[t + 1] = acc;
      if (merge_count[t] > 1) ns.merge_rows.push_back(t);
    }
  }
  ns.n_partials = partial_cursor;
  ns.max_chunks = max_chunks;
  const int64_t n_items = int64_t(ns.items.size());
  ns.grid = int32_t(n_items == 0 ? 0 : G);

  // ---- device layout
  WsHeader& h = ns.hdr;
  std::memset(&h, 0, sizeof h);
  h.n_items = int32_t(n_items);
  h.n_merge_rows = int32_t(ns.merge_rows.size());
  h.total_rows = ns.total_rows;
  h.batch = batch;
  h.group = g;
  h.causal = eff_causal;
  h.window_left = window_left;
  h.tile_rows = ns.tile_rows;
  h.num_qo_heads = hq;
  h.head_dim = d;
  int64_t off = kItemsOffset;
  h.off_items = off; off += int64_t(sizeof(WorkItem)) * n_items;
  h.off_qo_indptr = off; off = align_up(off + 4 * (batch + 1), 16);
  h.off_kv_indptr = off; off = align_up(off + 4 * (batch + 1), 16);
  h.off_kv_len = off; off = align_up(off + 4 * batch, 16);
  h.off_merge_indptr = off; off = align_up(off + 4 * (ns.total_rows + 1), 16);
  h.off_merge_rows = off; off = align_up(off + 4 * int64_t(ns.merge_rows.size()), 32);
  h.off_mask_indptr = off; off = align_up(off + 4 * (batch + 1), 16);
  ns.meta_bytes = align_up(off, kAlign);
  h.off_tmp_lse = ns.meta_bytes;
  h.off_tmp_o = ns.meta_bytes + align_up(4 * int64_t(ns.n_partials) * hq, kAlign);
  ns.total_bytes = ns.meta_bytes + partial_bytes_for(ns.n_partials, hq, d);
  if (!P.host_only && ns.total_bytes > int64_t(P.ws_bytes))
    return fail(FI_ERR_CAPACITY, "plan: workspace_bytes=%zu < %lld needed for %lld scheduled items "
                "and %d partial states", P.ws_bytes, (long long)ns.total_bytes,
                (long long)n_items, ns.n_partials);
  return FI_OK;
}

void write_staging(const PlanState& s, uint8_t* dst) {
  std::memset(dst, 0, s.meta_bytes);
  std::memcpy(dst, &s.hdr, sizeof(WsHeader));
  auto put = [&](int64_t off, const void* src, size_t n) {
    if (n) std::memcpy(dst + off, src, n);
  };
  put(s.hdr.off_qo_indptr, s.qo_indptr.data(), 4 * s.qo_indptr.size());
  put(s.hdr.off_kv_indptr, s.kv_indptr.data(), 4 * s.kv_indptr.size());
  put(s.hdr.off_kv_len, s.kv_len.data(), 4 * s.kv_len.size());
  put(s.hdr.off_merge_indptr, s.merge_indptr.data(), 4 * s.merge_indptr.size());
  put(s.hdr.off_merge_rows, s.merge_rows.data(), 4 * s.merge_rows.size());
  put(s.hdr.off_items, s.items.data(), sizeof(WorkItem) * s.items.size());
  put(s.hdr.off_mask_indptr, s.mask_indptr.data(), 4 * s.mask_indptr.size());
}

}  // namespace

namespace {

fi_status plan_common(fi_plan_t p, const int32_t* qo_indptr, const int32_t* kv_indptr,
                      const int32_t* last_page_len, int32_t batch, int32_t page_size,
                      int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                      int32_t causal, int32_t window_left, fi_dtype dtype,
                      int32_t q_len_per_req, int32_t force_kv_chunks, bool ragged,
                      const int32_t* mask_indptr, void* stream) {
  if (!p) return fail(FI_ERR_INVALID_ARG, "plan: plan is NULL");
  PlanState ns;
  fi_status st = build_plan(*p, qo_indptr, kv_indptr, last_page_len, batch, page_size,
                            num_qo_heads, num_kv_heads, head_dim, causal, window_left, dtype,
                            q_len_per_req, force_kv_chunks, ragged, mask_indptr, ns);
  if (st != FI_OK) return st;  // the previous plan stays usable
  ns.hdr.wait_limit_ns = p->wait_limit_ns;
  if (!p->host_only) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The upload copies from a host buffer that the next plan() rewrites, so
    // it cannot become a node of a captured graph.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone)
      return fail(FI_ERR_INVALID_ARG, "plan: the stream is capturing a graph (plan outside the "
                  "capture; a captured run() reads the latest plan when the graph is launched)");
    // this buffer's previous upload (two plans ago) must have left it
    const int slot = p->stage_next;
    if (p->staged_pending[slot]) {
      if (cudaEventSynchronize(p->staged[slot]) != cudaSuccess) {
        p->planned = false;
        return fail(FI_ERR_CUDA, "plan: waiting for an earlier upload failed");
      }
      p->staged_pending[slot] = false;
    }
    if (p->staging_bytes[slot] < size_t(ns.meta_bytes)) {
      if (p->staging[slot]) cudaFreeHost(p->staging[slot]);
      p->staging[slot] = nullptr;
      p->staging_bytes[slot] = 0;
      size_t want = size_t(align_up(ns.meta_bytes * 5 / 4 + 4096, 4096));
      if (cudaHostAlloc(&p->staging[slot], want, cudaHostAllocDefault) != cudaSuccess) {
        p->staging[slot] = nullptr;
        p->planned = false;
        return fail(FI_ERR_CUDA, "plan: cudaHostAlloc(%zu) failed", want);
      }
      p->staging_bytes[slot] = want;
    }
    write_staging(ns, static_cast<uint8_t*>(p->staging[slot]));
    // the workspace is rewritten only after the previous run() has read it
    cudaError_t e = cudaSuccess;
    if (p->run_recorded && p->last_run_stream != s) e = cudaStreamWaitEvent(s, p->run_done, 0);
    // from here the device copy changes: a failure leaves run() refusing
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(p->ws, p->staging[slot], size_t(ns.meta_bytes), cudaMemcpyHostToDevice,
                          s);
    if (e == cudaSuccess) e = cudaEventRecord(p->staged[slot], s);
    if (e == cudaSuccess) e = cudaEventRecord(p->upload_done, s);
    if (e != cudaSuccess) {
      p->planned = false;
      return fail(FI_ERR_CUDA, "plan: metadata upload failed: %s", cudaGetErrorString(e));
    }
    p->staged_pending[slot] = true;
    p->stage_next = slot ^ 1;
    p->upload_pending = true;
    p->upload_stream = s;
  }
  if (log_level() >= 2) {
    static const char* kname[] = {"decode", "prefill_m16", "prefill_m64", "prefill_m128"};
    std::fprintf(stderr, "[fi] plan: kernel=%s tile_rows=%d batch=%d rows=%d items=%zu "
                 "max_chunks=%d partials=%d merge_rows=%zu grid=%d graph=%d causal=%d "
                 "window_left=%d q_len_per_req=%d%s%s\n", kname[ns.kernel & 3], ns.tile_rows,
                 ns.batch, ns.total_rows, ns.items.size(), ns.max_chunks, ns.n_partials,
                 ns.merge_rows.size(), ns.grid, p->graph ? 1 : 0, ns.causal, ns.window_left,
                 ns.q_len_per_req, ns.ragged ? " ragged" : "", ns.masked ? " masked" : "");
  }
  if (p->graph && !p->frozen) {
    p->frozen = true;
    p->fz_kernel = ns.kernel; p->fz_qlpr = ns.q_len_per_req; p->fz_hq = ns.hq;
    p->fz_hk = ns.hk; p->fz_d = ns.d; p->fz_dtype = ns.dtype; p->fz_page = ns.page_size;
    p->fz_ragged = ns.ragged;
    p->fz_masked = ns.masked;
  }
  p->st = std::move(ns);
  p->planned = true;
  return ok();
}

}  // namespace

extern "C" fi_status fi_plan(fi_plan_t p, const int32_t* qo_indptr, const int32_t* kv_indptr,
                             const int32_t* last_page_len, int32_t batch, int32_t page_size,
                             int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                             int32_t causal, int32_t window_left, fi_dtype dtype,
                             int32_t q_len_per_req, int32_t force_kv_chunks, void* stream) {
  return plan_common(p, qo_indptr, kv_indptr, last_page_len, batch, page_size, num_qo_heads,
                     num_kv_heads, head_dim, causal, window_left, dtype, q_len_per_req,
                     force_kv_chunks, false, nullptr, stream);
}

extern "C" fi_status fi_plan_masked(fi_plan_t p, const int32_t* qo_indptr,
                                    const int32_t* kv_indptr, const int32_t* last_page_len,
                                    int32_t batch, int32_t page_size, int32_t num_qo_heads,
                                    int32_t num_kv_heads, int32_t head_dim, int32_t causal,
                                    int32_t window_left, fi_dtype dtype,
                                    const int32_t* mask_indptr, int32_t force_kv_chunks,
                                    void* stream) {
  if (batch > 0 && !mask_indptr)
    return fail(FI_ERR_INVALID_ARG, "plan: mask_indptr is NULL for a masked plan");
  static const int32_t zero[1] = {0};
  return plan_common(p, qo_indptr, kv_indptr, last_page_len, batch, page_size, num_qo_heads,
                     num_kv_heads, head_dim, causal, window_left, dtype, 0, force_kv_chunks,
                     false, mask_indptr ? mask_indptr : zero, stream);
}

extern "C" fi_status fi_plan_ragged(fi_plan_t p, const int32_t* qo_indptr,
                                    const int32_t* kv_indptr, int32_t batch, int32_t num_qo_heads,
                                    int32_t num_kv_heads, int32_t head_dim, int32_t causal,
                                    int32_t window_left, fi_dtype dtype, int32_t force_kv_chunks,
                                    void* stream) {
  return plan_common(p, qo_indptr, kv_indptr, nullptr, batch, kRaggedPage, num_qo_heads,
                     num_kv_heads, head_dim, causal, window_left, dtype, 0, force_kv_chunks, true,
                     nullptr, stream);
}

extern "C" fi_status fi_plan_get_info(fi_plan_t p, fi_plan_info* info, int32_t* items,
                                      int32_t items_capacity, int32_t* merge_indptr,
                                      int32_t merge_capacity) {
  if (!p) return fail(FI_ERR_INVALID_ARG, "plan_get_info: plan is NULL");
  if (!p->planned) return fail(FI_ERR_NOT_PLANNED, "plan_get_info: call fi_plan() first");
  const PlanState& s = p->st;
  if (info) {
    info->batch = s.batch;
    info->total_rows = s.total_rows;
    info->kernel = s.kernel;
    info->tile_rows = s.tile_rows;
    info->num_items = int32_t(s.items.size());
    info->num_partials = s.n_partials;
    info->num_merge_rows = int32_t(s.merge_rows.size());
    info->max_chunks = s.max_chunks;
    info->grid = s.grid;
    info->graph_mode = p->graph ? 1 : 0;
  }
  if (items) {
    if (items_capacity < int32_t(s.items.size() * kItemPublicInts))
      return fail(FI_ERR_CAPACITY, "plan_get_info: items_capacity=%d < %d", items_capacity,
                  int32_t(s.items.size() * kItemPublicInts));
    for (size_t i = 0; i < s.items.size(); ++i)  // the public fields of each item
      std::memcpy(items + i * kItemPublicInts, &s.items[i], kItemPublicInts * sizeof(int32_t));
  }
  if (merge_indptr) {
    if (merge_capacity < int32_t(s.merge_indptr.size()))
      return fail(FI_ERR_CAPACITY, "plan_get_info: merge_capacity=%d < %d", merge_capacity,
                  int32_t(s.merge_indptr.size()));
    std::memcpy(merge_indptr, s.merge_indptr.data(), s.merge_indptr.size() * 4);
  }
  return ok();
}

namespace {
// A stream that reads or writes the workspace outside run(): after the latest
// metadata upload and the latest run().
cudaError_t order_after_plan_and_run(fi_plan_t p, cudaStream_t st) {
  cudaError_t e = cudaSuccess;
  if (p->upload_pending && p->upload_stream != st) e = cudaStreamWaitEvent(st, p->upload_done, 0);
  if (e == cudaSuccess && p->run_recorded && p->last_run_stream != st)
    e = cudaStreamWaitEvent(st, p->run_done, 0);
  return e;
}
}  // namespace

extern "C" fi_status fi_plan_read_device(fi_plan_t p, int32_t* items, int32_t items_capacity,
                                         int32_t* merge_indptr, int32_t merge_capacity,
                                         void* stream) {
  if (!p) return fail(FI_ERR_INVALID_ARG, "plan_read_device: plan is NULL");
  if (!p->planned) return fail(FI_ERR_NOT_PLANNED, "plan_read_device: call fi_plan() first");
  if (p->host_only) return fail(FI_ERR_INVALID_ARG, "plan_read_device: host-only plan");
  const PlanState& s = p->st;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  std::vector<uint8_t> buf(size_t(s.meta_bytes));
  cudaError_t e = order_after_plan_and_run(p, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(buf.data(), p->ws, buf.size(), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess)
    return fail(FI_ERR_CUDA, "plan_read_device: %s", cudaGetErrorString(e));
  WsHeader h;
  std::memcpy(&h, buf.data(), sizeof h);
  if (items) {
    if (items_capacity < h.n_items * kItemPublicInts) return fail(FI_ERR_CAPACITY, "plan_read_device: items");
    for (int32_t i = 0; i < h.n_items; ++i)  // the public fields of each item
      std::memcpy(items + size_t(i) * kItemPublicInts,
                  buf.data() + h.off_items + int64_t(i) * int64_t(sizeof(WorkItem)),
                  kItemPublicInts * sizeof(int32_t));
  }
  if (merge_indptr) {
    if (merge_capacity < h.total_rows + 1) return fail(FI_ERR_CAPACITY, "plan_read_device: merge");
    std::memcpy(merge_indptr, buf.data() + h.off_merge_indptr, size_t(h.total_rows + 1) * 4);
  }
  return ok();
}

extern "C" fi_status fi_plan_device_error(fi_plan_t p, int32_t* err_flag, int clear,
                                          void* stream) {
  if (!p || !err_flag) return fail(FI_ERR_INVALID_ARG, "plan_device_error: NULL argument");
  if (!p->planned) return fail(FI_ERR_NOT_PLANNED, "plan_device_error: call fi_plan() first");
  if (p->host_only) return fail(FI_ERR_INVALID_ARG, "plan_device_error: host-only plan");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // err_flag and index_error are adjacent int32 fields of the header
  static_assert(offsetof(WsHeader, index_error) == offsetof(WsHeader, err_flag) + 4,
                "adjacent flags");
  uint8_t* flag = static_cast<uint8_t*>(p->ws) + offsetof(WsHeader, err_flag);
  int32_t v[2] = {0, 0};
  cudaError_t e = order_after_plan_and_run(p, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(v, flag, sizeof v, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess && clear) e = cudaMemsetAsync(flag, 0, sizeof v, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return fail(FI_ERR_CUDA, "plan_device_error: %s", cudaGetErrorString(e));
  *err_flag = (v[0] ? 1 : 0) | (v[1] ? 2 : 0);
  return ok();
}

extern "C" fi_status fi_plan_set_wait_limit(fi_plan_t p, uint64_t limit_ns) {
  if (!p) return fail(FI_ERR_INVALID_ARG, "plan_set_wait_limit: plan is NULL");
  p->wait_limit_ns = limit_ns;
  return ok();
}

// ------------------------------------------------------------------ run()
namespace {

const char* dtype_name(int d) {
  switch (d) {
    case FI_F16: return "f16";
    case FI_BF16: return "bf16";
    case FI_F32: return "f32";
    case FI_I32: return "i32";
    case FI_U8: return "u8";
  }
  return "?";
}

fi_status check_tensor(const fi_tensor* t, const char* name, int ndim) {
  if (!t || !t->data) return fail(FI_ERR_INVALID_ARG, "run: %s is NULL", name);
  if (t->ndim != ndim)
    return fail(FI_ERR_PLAN_MISMATCH, "run: %s rank: expected %d, got %d", name, ndim, t->ndim);
  for (int i = 0; i < ndim; ++i)
    if (t->shape[i] < 0) return fail(FI_ERR_INVALID_ARG, "run: %s shape[%d] < 0", name, i);
  // [P3 "Strided layouts"]: a strided last dim is refused, not copied
  if (t->shape[ndim - 1] > 1 && t->stride[ndim - 1] != 1)
    return fail(FI_ERR_STRIDED_LAST_DIM, "run: %s has stride(-1)=%lld, expected 1", name,
                (long long)t->stride[ndim - 1]);
  return FI_OK;
}

fi_status check_dim(const char* tname, const char* field, int64_t planned, int64_t got) {
  return fail(FI_ERR_PLAN_MISMATCH, "run: %s %s: planned %lld, got %lld", tname, field,
              (long long)planned, (long long)got);
}

fi_status check_packed(const fi_tensor* t, const char* name) {
  int64_t expect = 1;
  for (int i = t->ndim - 1; i >= 0; --i) {
    if (t->shape[i] > 1 && t->stride[i] != expect)
      return fail(FI_ERR_NONCONTIGUOUS_OUTPUT, "run: %s is not packed (stride[%d]=%lld, "
                  "expected %lld)", name, i, (long long)t->stride[i], (long long)expect);
    expect *= t->shape[i];
  }
  return FI_OK;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; }

// ragged: k / v are [rows, Hk, d] contiguous K/V (kv_indices unused) and the
// plan came from fi_plan_ragged.
fi_status run_common(fi_plan_t p, bool decode_api, bool ragged, const fi_tensor* q,
                     const fi_tensor* k, const fi_tensor* v, const fi_tensor* kv_indices,
                     const fi_tensor* custom_mask, float sm_scale, fi_tensor* out, fi_tensor* lse,
                     void* stream) {
  const char* api = ragged ? "batch_prefill_ragged"
                    : decode_api ? "batch_decode_paged"
                    : custom_mask ? "batch_prefill_paged_masked" : "batch_prefill_paged";
  if (!p) return fail(FI_ERR_INVALID_ARG, "%s: plan is NULL", api);
  // [P3 "Plan-vs-run shapes"]: a half-planned object refuses run()
  if (!p->planned) return fail(FI_ERR_NOT_PLANNED, "%s: call fi_plan() first", api);
  const PlanState& s = p->st;
  if ((custom_mask != nullptr) != (s.masked != 0))
    return fail(FI_ERR_PLAN_MISMATCH, "%s: the plan is %s (fi_plan%s)", api,
                s.masked ? "for a custom mask" : "without a custom mask",
                s.masked ? "_masked" : "");
  if (custom_mask) {
    fi_status cst = check_tensor(custom_mask, "custom_mask", 1);
    if (cst != FI_OK) return cst;
    if (custom_mask->dtype != FI_U8)
      return fail(FI_ERR_INVALID_ARG, "%s: custom_mask must be FI_U8", api);
    if (custom_mask->shape[0] < s.mask_bytes)
      return check_dim("custom_mask", "bytes (minimum, mask_indptr[batch])", s.mask_bytes,
                       custom_mask->shape[0]);
  }
  if (ragged != (s.ragged != 0))
    return fail(FI_ERR_PLAN_MISMATCH, "%s: the plan is for a %s K/V cache (fi_plan%s)", api,
                s.ragged ? "ragged" : "paged", s.ragged ? "_ragged" : "");
  if (decode_api && s.q_len_per_req < 1)
    return fail(FI_ERR_PLAN_MISMATCH, "%s: q_len_per_req: planned %d (a prefill plan), "
                "expected >= 1", api, s.q_len_per_req);
  if (!decode_api && s.q_len_per_req != 0)
    return fail(FI_ERR_PLAN_MISMATCH, "%s: q_len_per_req: planned %d (a decode plan), "
                "expected 0", api, s.q_len_per_req);
  fi_status st;
  const int kv_ndim = ragged ? 3 : 4;  // ragged: [rows, Hk, d]; paged: [pages, P, Hk, d]
  if ((st = check_tensor(q, "q", 3)) != FI_OK) return st;
  if ((st = check_tensor(k, "k_cache", kv_ndim)) != FI_OK) return st;
  if ((st = check_tensor(v, "v_cache", kv_ndim)) != FI_OK) return st;
  if (!ragged && (st = check_tensor(kv_indices, "kv_indices", 1)) != FI_OK) return st;
  if ((st = check_tensor(out, "out", 3)) != FI_OK) return st;
  if (lse && (st = check_tensor(lse, "lse", 2)) != FI_OK) return st;
  // [P3 "Plan-vs-run shapes"]: heads, head dims, page size, token minimums
  if (q->shape[0] < s.total_rows) return check_dim("q", "rows (minimum)", s.total_rows, q->shape[0]);
  if (q->shape[1] != s.hq) return check_dim("q", "num_qo_heads", s.hq, q->shape[1]);
  if (q->shape[2] != s.d) return check_dim("q", "head_dim", s.d, q->shape[2]);
  const int kh = ragged ? 1 : 2;  // index of the kv-head dim
  for (const fi_tensor* c : {k, v}) {
    const char* n = (c == k) ? "k_cache" : "v_cache";
    if (!ragged && c->shape[1] != s.page_size)
      return check_dim(n, "page_size", s.page_size, c->shape[1]);
    if (ragged && c->shape[0] < s.kv_indices_len)
      return check_dim(n, "rows (minimum, kv_indptr[batch])", s.kv_indices_len, c->shape[0]);
    if (c->shape[kh] != s.hk) return check_dim(n, "num_kv_heads", s.hk, c->shape[kh]);
    if (c->shape[kh + 1] != s.d) return check_dim(n, "head_dim", s.d, c->shape[kh + 1]);
    if (c->dtype != s.dtype)
      return fail(FI_ERR_PLAN_MISMATCH, "run: %s dtype: planned %s, got %s", n,
                  dtype_name(s.dtype), dtype_name(c->dtype));
  }
  if (k->shape[0] != v->shape[0])
    return fail(FI_ERR_INVALID_ARG, "run: k_cache has %lld pages, v_cache %lld",
                (long long)k->shape[0], (long long)v->shape[0]);
  if (q->dtype != s.dtype)
    return fail(FI_ERR_PLAN_MISMATCH, "run: q dtype: planned %s, got %s", dtype_name(s.dtype),
                dtype_name(q->dtype));
  if (out->dtype != s.dtype)
    return fail(FI_ERR_PLAN_MISMATCH, "run: out dtype: planned %s, got %s",
                dtype_name(s.dtype), dtype_name(out->dtype));
  if (!ragged) {
    if (kv_indices->dtype != FI_I32)
      return fail(FI_ERR_INVALID_ARG, "run: kv_indices must be int32");
    if (kv_indices->shape[0] < s.kv_indices_len)
      return check_dim("kv_indices", "length (minimum)", s.kv_indices_len, kv_indices->shape[0]);
  }
  if (out->shape[0] < s.total_rows)
    return check_dim("out", "rows (minimum)", s.total_rows, out->shape[0]);
  if (out->shape[1] != s.hq) return check_dim("out", "num_qo_heads", s.hq, out->shape[1]);
  if (out->shape[2] != s.d) return check_dim("out", "head_dim", s.d, out->shape[2]);
  // [P3 "Strided layouts"]: out and lse must be packed
  if ((st = check_packed(out, "out")) != FI_OK) return st;
  if (lse) {
    if (lse->dtype != FI_F32) return fail(FI_ERR_INVALID_ARG, "run: lse must be fp32");
    if (lse->shape[0] < s.total_rows)
      return check_dim("lse", "rows (minimum)", s.total_rows, lse->shape[0]);
    if (lse->shape[1] != s.hq) return check_dim("lse", "num_qo_heads", s.hq, lse->shape[1]);
    if ((st = check_packed(lse, "lse")) != FI_OK) return st;
  }
  if (!(sm_scale > 0.f) || sm_scale > 3.0e38f)
    return fail(FI_ERR_INVALID_ARG, "%s: sm_scale=%g must be positive and finite", api,
                double(sm_scale));
  // 16-byte vector loads of every row
  bool kv_strides_ok = true;
  for (int i = 0; i < kv_ndim - 1; ++i)
    if (k->stride[i] % 8 || v->stride[i] % 8) kv_strides_ok = false;
  if (!aligned16(q->data) || !aligned16(k->data) || !aligned16(v->data) || !aligned16(out->data) ||
      q->stride[0] % 8 || q->stride[1] % 8 || !kv_strides_ok)
    return fail(FI_ERR_UNSUPPORTED, "run: q/k/v/out rows must start on 16-byte boundaries "
                "(strides multiples of 8 elements)");

  // everything above is host-side validation; a host-only plan stops here
  if (p->host_only) return fail(FI_ERR_INVALID_ARG, "%s: plan has no device workspace", api);

  fi::AttnParams ap;
  ap.q = q->data; ap.q_stride_tok = q->stride[0]; ap.q_stride_head = q->stride[1];
  if (ragged) {  // one logical page of all rows: page stride unused
    ap.k = k->data; ap.k_stride_page = 0; ap.k_stride_tok = k->stride[0];
    ap.k_stride_head = k->stride[1];
    ap.v = v->data; ap.v_stride_page = 0; ap.v_stride_tok = v->stride[0];
    ap.v_stride_head = v->stride[1];
    ap.kv_indices = nullptr;
  } else {
    ap.k = k->data; ap.k_stride_page = k->stride[0]; ap.k_stride_tok = k->stride[1];
    ap.k_stride_head = k->stride[2];
    ap.v = v->data; ap.v_stride_page = v->stride[0]; ap.v_stride_tok = v->stride[1];
    ap.v_stride_head = v->stride[2];
    ap.kv_indices = static_cast<const int32_t*>(kv_indices->data);
  }
  ap.ragged = ragged ? 1 : 0;
  ap.kv_rows = ragged ? std::min(k->shape[0], v->shape[0]) : 0;
  ap.custom_mask = custom_mask ? static_cast<const uint8_t*>(custom_mask->data) : nullptr;
  ap.out = out->data;
  ap.lse = lse ? static_cast<float*>(lse->data) : nullptr;
  ap.ws = p->ws;
  ap.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  ap.num_qo_heads = s.hq;
  ap.num_kv_heads = s.hk;
  ap.page_size = s.page_size;
  ap.page_shift = -1;
  for (int sh = 0; sh < 31; ++sh)
    if ((1 << sh) == s.page_size) ap.page_shift = sh;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const bool bf16 = s.dtype == FI_BF16;
  const bool any_work = p->graph || !s.items.empty();
  // Stream order against plan() and earlier runs (outside a capture; a
  // captured run reads whatever plan the workspace holds at graph launch).
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(cs, &cap) != cudaSuccess)
    return fail(FI_ERR_CUDA, "%s: cudaStreamIsCapturing failed", api);
  const bool capturing = cap != cudaStreamCaptureStatusNone;
  if (!capturing) {
    cudaError_t e = cudaSuccess;
    if (p->upload_pending && p->upload_stream != cs) e = cudaStreamWaitEvent(cs, p->upload_done, 0);
    if (e == cudaSuccess && p->run_recorded && p->last_run_stream != cs)
      e = cudaStreamWaitEvent(cs, p->run_done, 0);
    if (e != cudaSuccess)
      return fail(FI_ERR_CUDA, "%s: ordering after plan(): %s", api, cudaGetErrorString(e));
  }
  if (log_level() >= 3)
    std::fprintf(stderr, "[fi] %s: kernel=%d grid=%d items=%zu merge_rows=%zu stream=%p%s%s\n",
                 api, s.kernel, s.grid, s.items.size(), s.merge_rows.size(),
                 static_cast<void*>(cs), capturing ? " (capturing)" : "",
                 (!ragged && check_indices_enabled()) ? " index-check" : "");
  if (!ragged && check_indices_enabled() && any_work) {
    // count page-table entries outside [0, num_pages); the attention kernels
    // and the merge read the count and do nothing when it is non-zero
    cudaError_t e = cudaMemsetAsync(static_cast<uint8_t*>(p->ws) + offsetof(WsHeader, index_error),
                                    0, sizeof(int32_t), cs);
    if (e == cudaSuccess)
      e = fi::launch_check_indices(p->ws, ap.kv_indices, k->shape[0], p->num_sms, cs);
    if (e != cudaSuccess)
      return fail(FI_ERR_CUDA, "%s: index check launch failed: %s", api, cudaGetErrorString(e));
  }
  if (any_work) {
    cudaError_t e;
    if (s.kernel == fi::kDecode)
      e = fi::launch_decode(ap, s.d, s.group, bf16, ragged ? 1 : k->shape[0], s.tile_rows,
                            s.grid, cs);
    else if (s.kernel == fi::kPrefillM128)
      e = fi::launch_prefill_tc(ap, s.d, s.group, s.tile_rows, q->shape[0],
                                ragged ? 1 : k->shape[0], bf16, s.grid, cs);
    else e = fi::launch_prefill_mma(ap, s.d, s.kernel, bf16, s.grid, cs);
    if (e != cudaSuccess)
      return fail(FI_ERR_CUDA, "%s: attention launch failed: %s", api, cudaGetErrorString(e));
  }
  if (p->graph || !s.merge_rows.empty()) {
    int merge_grid = p->graph ? p->num_sms * 4
                              : int(std::min<int64_t>(p->num_sms * 4,
                                                      (int64_t(s.merge_rows.size()) * s.hq + 7) / 8));
    cudaError_t e = fi::launch_merge_workspace(p->ws, out->data, ap.lse, s.hq, s.d, bf16,
                                               std::max(merge_grid, 1), cs);
    if (e != cudaSuccess)
      return fail(FI_ERR_CUDA, "%s: merge launch failed: %s", api, cudaGetErrorString(e));
  }
  if (!capturing) {
    cudaError_t e = cudaEventRecord(p->run_done, cs);
    if (e != cudaSuccess)
      return fail(FI_ERR_CUDA, "%s: cudaEventRecord: %s", api, cudaGetErrorString(e));
    p->run_recorded = true;
    p->last_run_stream = cs;
  }
  return ok();
}

}  // namespace

extern "C" fi_status fi_check_kv_indices(fi_plan_t p, const fi_tensor* kv_indices,
                                         int64_t num_pages, void* stream) {
  if (!p) return fail(FI_ERR_INVALID_ARG, "check_kv_indices: plan is NULL");
  if (!p->planned) return fail(FI_ERR_NOT_PLANNED, "check_kv_indices: call fi_plan() first");
  if (p->host_only) return fail(FI_ERR_INVALID_ARG, "check_kv_indices: host-only plan");
  if (p->st.ragged)
    return fail(FI_ERR_PLAN_MISMATCH, "check_kv_indices: a ragged plan has no page table");
  fi_status fs = check_tensor(kv_indices, "kv_indices", 1);
  if (fs != FI_OK) return fs;
  if (kv_indices->dtype != FI_I32)
    return fail(FI_ERR_INVALID_ARG, "check_kv_indices: kv_indices must be int32");
  if (kv_indices->shape[0] < p->st.kv_indices_len)
    return check_dim("kv_indices", "length (minimum)", p->st.kv_indices_len, kv_indices->shape[0]);
  if (num_pages < 0) return fail(FI_ERR_INVALID_ARG, "check_kv_indices: num_pages < 0");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = order_after_plan_and_run(p, st);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(static_cast<uint8_t*>(p->ws) + offsetof(WsHeader, index_error), 0,
                        sizeof(int32_t), st);
  if (e == cudaSuccess)
    e = fi::launch_check_indices(p->ws, static_cast<const int32_t*>(kv_indices->data), num_pages,
                                 p->num_sms, st);
  if (e != cudaSuccess)
    return fail(FI_ERR_CUDA, "check_kv_indices: %s", cudaGetErrorString(e));
  return ok();
}

extern "C" fi_status fi_batch_prefill_paged(fi_plan_t p, const fi_tensor* q, const fi_tensor* k,
                                            const fi_tensor* v, const fi_tensor* kv_indices,
                                            float sm_scale, fi_tensor* out, fi_tensor* lse,
                                            void* stream) {
  return run_common(p, false, false, q, k, v, kv_indices, nullptr, sm_scale, out, lse, stream);
}

extern "C" fi_status fi_batch_prefill_paged_masked(fi_plan_t p, const fi_tensor* q,
                                                   const fi_tensor* k, const fi_tensor* v,
                                                   const fi_tensor* kv_indices,
                                                   const fi_tensor* custom_mask, float sm_scale,
                                                   fi_tensor* out, fi_tensor* lse, void* stream) {
  if (!custom_mask)
    return fail(FI_ERR_INVALID_ARG, "batch_prefill_paged_masked: custom_mask is NULL");
  return run_common(p, false, false, q, k, v, kv_indices, custom_mask, sm_scale, out, lse,
                    stream);
}

extern "C" fi_status fi_batch_decode_paged(fi_plan_t p, const fi_tensor* q, const fi_tensor* k,
                                           const fi_tensor* v, const fi_tensor* kv_indices,
                                           float sm_scale, fi_tensor* out, fi_tensor* lse,
                                           void* stream) {
  return run_common(p, true, false, q, k, v, kv_indices, nullptr, sm_scale, out, lse, stream);
}

extern "C" fi_status fi_batch_prefill_ragged(fi_plan_t p, const fi_tensor* q, const fi_tensor* k,
                                             const fi_tensor* v, float sm_scale, fi_tensor* out,
                                             fi_tensor* lse, void* stream) {
  return run_common(p, false, true, q, k, v, nullptr, nullptr, sm_scale, out, lse, stream);
}

// ------------------------------------------------ speculative sampling
extern "C" fi_status fi_chain_speculative_sampling(
    const fi_tensor* draft_probs, const fi_tensor* draft_token_ids,
    const fi_tensor* target_probs, const fi_tensor* uniform_accept,
    const fi_tensor* uniform_sample, fi_tensor* output_token_ids, fi_tensor* accepted_num,
    fi_tensor* emitted_num, void* stream) {
  const char* api = "chain_speculative_sampling";
  fi_status st;
  if ((st = check_tensor(target_probs, "target_probs", 3)) != FI_OK) return st;
  const int64_t B = target_probs->shape[0];
  const int64_t n = target_probs->shape[1] - 1;
  const int64_t V = target_probs->shape[2];
  if (n < 0 || V < 1 || n > 4096)
    return fail(FI_ERR_INVALID_ARG, "%s: target_probs [B, n+1, V] needs n+1 >= 1, V >= 1", api);
  if (V > fi::chain_spec_max_vocab())
    return fail(FI_ERR_UNSUPPORTED, "%s: vocabulary %lld > %d", api, (long long)V,
                fi::chain_spec_max_vocab());
  if ((st = check_tensor(uniform_sample, "uniform_sample", 1)) != FI_OK) return st;
  if ((st = check_tensor(output_token_ids, "output_token_ids", 2)) != FI_OK) return st;
  if ((st = check_tensor(accepted_num, "accepted_num", 1)) != FI_OK) return st;
  if (emitted_num && (st = check_tensor(emitted_num, "emitted_num", 1)) != FI_OK) return st;
  if (n > 0) {
    if ((st = check_tensor(draft_probs, "draft_probs", 3)) != FI_OK) return st;
    if ((st = check_tensor(draft_token_ids, "draft_token_ids", 2)) != FI_OK) return st;
    if ((st = check_tensor(uniform_accept, "uniform_accept", 2)) != FI_OK) return st;
    if (draft_probs->shape[0] != B || draft_probs->shape[1] != n || draft_probs->shape[2] != V)
      return fail(FI_ERR_INVALID_ARG, "%s: draft_probs must be [B, n, V] = [%lld, %lld, %lld]",
                  api, (long long)B, (long long)n, (long long)V);
    if (draft_token_ids->shape[0] != B || draft_token_ids->shape[1] != n ||
        uniform_accept->shape[0] != B || uniform_accept->shape[1] != n)
      return fail(FI_ERR_INVALID_ARG, "%s: draft_token_ids and uniform_accept must be [B, n]", api);
    if (draft_probs->dtype != FI_F32 || draft_token_ids->dtype != FI_I32 ||
        uniform_accept->dtype != FI_F32)
      return fail(FI_ERR_INVALID_ARG, "%s: draft_probs / uniform_accept F32, draft_token_ids I32",
                  api);
  }
  if (target_probs->dtype != FI_F32 || uniform_sample->dtype != FI_F32 ||
      output_token_ids->dtype != FI_I32 || accepted_num->dtype != FI_I32 ||
      (emitted_num && emitted_num->dtype != FI_I32))
    return fail(FI_ERR_INVALID_ARG, "%s: probabilities and uniforms F32, outputs I32", api);
  if (uniform_sample->shape[0] != B || accepted_num->shape[0] != B ||
      (emitted_num && emitted_num->shape[0] != B) || output_token_ids->shape[0] != B ||
      output_token_ids->shape[1] != n + 1)
    return fail(FI_ERR_INVALID_ARG, "%s: uniform_sample / accepted_num / emitted_num [B], "
                "output_token_ids [B, n+1]", api);
  if ((st = check_packed(output_token_ids, "output_token_ids")) != FI_OK) return st;
  if ((st = check_packed(accepted_num, "accepted_num")) != FI_OK) return st;
  if (emitted_num && (st = check_packed(emitted_num, "emitted_num")) != FI_OK) return st;
  fi::SpecParams sp;
  sp.target_probs = static_cast<const float*>(target_probs->data);
  sp.tp_sb = target_probs->stride[0];
  sp.tp_si = target_probs->stride[1];
  sp.u_sample = static_cast<const float*>(uniform_sample->data);
  sp.draft_probs = n > 0 ? static_cast<const float*>(draft_probs->data) : nullptr;
  sp.dp_sb = n > 0 ? draft_probs->stride[0] : 0;
  sp.dp_si = n > 0 ? draft_probs->stride[1] : 0;
  sp.draft_ids = n > 0 ? static_cast<const int32_t*>(draft_token_ids->data) : nullptr;
  sp.ids_sb = n > 0 ? draft_token_ids->stride[0] : 0;
  sp.u_accept = n > 0 ? static_cast<const float*>(uniform_accept->data) : nullptr;
  sp.ua_sb = n > 0 ? uniform_accept->stride[0] : 0;
  sp.n = int32_t(n);
  sp.vocab = int32_t(V);
  sp.out_tokens = static_cast<int32_t*>(output_token_ids->data);
  sp.out_accepted = static_cast<int32_t*>(accepted_num->data);
  sp.out_emitted = emitted_num ? static_cast<int32_t*>(emitted_num->data) : nullptr;
  if (n > 0 && (draft_token_ids->stride[1] != 1 || uniform_accept->stride[1] != 1))
    return fail(FI_ERR_STRIDED_LAST_DIM, "%s: draft_token_ids / uniform_accept rows", api);
  if (uniform_sample->shape[0] > 1 && uniform_sample->stride[0] != 1)
    return fail(FI_ERR_STRIDED_LAST_DIM, "%s: uniform_sample must be contiguous", api);
  cudaError_t e = fi::launch_chain_spec_sampling(sp, int(B), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(FI_ERR_CUDA, "%s: launch failed: %s", api, cudaGetErrorString(e));
  return ok();
}

// ------------------------------------------------------------------ merges
extern "C" fi_status fi_merge_state(const fi_tensor* va, const fi_tensor* sa, const fi_tensor* vb,
                                    const fi_tensor* sb, fi_tensor* vo, fi_tensor* so,
                                    const int32_t* num_rows_dev, void* stream) {
  fi_status st;
  if ((st = check_tensor(va, "v_a", 3)) != FI_OK) return st;
  if ((st = check_tensor(vb, "v_b", 3)) != FI_OK) return st;
  if ((st = check_tensor(vo, "v_out", 3)) != FI_OK) return st;
  if ((st = check_tensor(sa, "s_a", 2)) != FI_OK) return st;
  if ((st = check_tensor(sb, "s_b", 2)) != FI_OK) return st;
  if ((st = check_tensor(so, "s_out", 2)) != FI_OK) return st;
  for (const fi_tensor* t : {vb, static_cast<const fi_tensor*>(vo)})
    for (int i = 0; i < 3; ++i)
      if (t->shape[i] != va->shape[i])
        return fail(FI_ERR_INVALID_ARG, "merge_state: v shapes differ at dim %d (%lld vs %lld)", i,
                    (long long)t->shape[i], (long long)va->shape[i]);
  for (const fi_tensor* t : {sa, sb, static_cast<const fi_tensor*>(so)})
    if (t->shape[0] != va->shape[0] || t->shape[1] != va->shape[1])
      return fail(FI_ERR_INVALID_ARG, "merge_state: s must be [rows, heads] of v");
  if (va->dtype != vb->dtype || va->dtype != vo->dtype || va->dtype == FI_I32)
    return fail(FI_ERR_INVALID_ARG, "merge_state: v_a, v_b, v_out must share one float dtype");
  if (sa->dtype != FI_F32 || sb->dtype != FI_F32 || so->dtype != FI_F32)
    return fail(FI_ERR_INVALID_ARG, "merge_state: s must be fp32");
  if ((st = check_packed(vo, "v_out")) != FI_OK) return st;
  if ((st = check_packed(so, "s_out")) != FI_OK) return st;
  if (sa->shape[1] > 1 && (sa->stride[1] != 1 || sb->stride[1] != 1))
    return fail(FI_ERR_STRIDED_LAST_DIM, "merge_state: s head stride must be 1");
  if (va->shape[0] > INT32_MAX || va->shape[1] > 65535 || va->shape[2] > 1024)
    return fail(FI_ERR_UNSUPPORTED, "merge_state: shape too large");
  fi::MergeTwoParams mp;
  mp.va = va->data; mp.vb = vb->data; mp.vo = vo->data;
  mp.sa = static_cast<const float*>(sa->data);
  mp.sb = static_cast<const float*>(sb->data);
  mp.so = static_cast<float*>(so->data);
  mp.va_sr = va->stride[0]; mp.va_sh = va->stride[1];
  mp.vb_sr = vb->stride[0]; mp.vb_sh = vb->stride[1];
  mp.sa_sr = sa->stride[0]; mp.sb_sr = sb->stride[0];
  mp.rows = int32_t(va->shape[0]); mp.heads = int32_t(va->shape[1]);
  mp.head_dim = int32_t(va->shape[2]); mp.dtype = va->dtype;
  mp.num_rows_dev = num_rows_dev;
  if (mp.rows == 0 && !num_rows_dev) return ok();
  cudaError_t e = fi::launch_merge_two(mp, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(FI_ERR_CUDA, "merge_state: %s", cudaGetErrorString(e));
  return ok();
}

extern "C" fi_status fi_merge_states(const fi_tensor* v, const fi_tensor* s,
                                     const int32_t* merge_indptr_dev, int32_t rows,
                                     fi_tensor* v_out, fi_tensor* s_out,
                                     const int32_t* num_rows_dev, void* stream) {
  fi_status st;
  if ((st = check_tensor(v, "v", 3)) != FI_OK) return st;
  if ((st = check_tensor(s, "s", 2)) != FI_OK) return st;
  if ((st = check_tensor(v_out, "v_out", 3)) != FI_OK) return st;
  if (s_out && (st = check_tensor(s_out, "s_out", 2)) != FI_OK) return st;
  if (!merge_indptr_dev) return fail(FI_ERR_INVALID_ARG, "merge_states: merge_indptr is NULL");
  if (rows < 0) return fail(FI_ERR_INVALID_ARG, "merge_states: rows=%d < 0", rows);
  if (v->dtype != FI_F32 || s->dtype != FI_F32)
    return fail(FI_ERR_INVALID_ARG, "merge_states: partial v and s must be fp32");
  if ((st = check_packed(v, "v")) != FI_OK) return st;
  if ((st = check_packed(s, "s")) != FI_OK) return st;
  if ((st = check_packed(v_out, "v_out")) != FI_OK) return st;
  if (v_out->shape[0] < rows || v_out->shape[1] != v->shape[1] || v_out->shape[2] != v->shape[2])
    return fail(FI_ERR_INVALID_ARG, "merge_states: v_out must be [>= rows, H, d] of v");
  if (s->shape[0] != v->shape[0] || s->shape[1] != v->shape[1])
    return fail(FI_ERR_INVALID_ARG, "merge_states: s must be [n, H] of v");
  if (s_out) {
    if (s_out->dtype != FI_F32) return fail(FI_ERR_INVALID_ARG, "merge_states: s_out must be fp32");
    if ((st = check_packed(s_out, "s_out")) != FI_OK) return st;
    if (s_out->shape[0] < rows || s_out->shape[1] != v->shape[1])
      return fail(FI_ERR_INVALID_ARG, "merge_states: s_out must be [>= rows, H]");
  }
  if (v_out->dtype == FI_I32) return fail(FI_ERR_INVALID_ARG, "merge_states: v_out dtype");
  if (v->shape[2] % 4 != 0 || v->shape[2] > 1024)
    return fail(FI_ERR_UNSUPPORTED, "merge_states: head_dim must be a multiple of 4, <= 1024");
  if (rows == 0 && !num_rows_dev) return ok();
  cudaError_t e = fi::launch_merge_states(
      static_cast<const float*>(v->data), static_cast<const float*>(s->data), merge_indptr_dev,
      rows, int(v->shape[1]), int(v->shape[2]), v_out->data, v_out->dtype,
      s_out ? static_cast<float*>(s_out->data) : nullptr, num_rows_dev,
      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(FI_ERR_CUDA, "merge_states: %s", cudaGetErrorString(e));
  return ok();
}
