// Batch decode that allocates nothing: its split-KV scratch (plan metadata and
// partial attention states) lives in a fixed file-scope device array instead
// of a caller-supplied workspace. For callers that may not allocate device
// memory at all - code that runs inside another framework's memory pool or a
// serving loop that reserved all memory up front, and host code that must
// not call cudaMalloc/cudaFree on the hot path.
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/fi.h"
#include "common.cuh"

namespace fi {

// Every GPU that loads the library holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};  // device address of the array, per device
std::mutex g_scratch_mu;                 // guards the first lookup on each device

// The array's device address on the current device: looked up once per
// device (with that device current) and kept; nullptr and an error message on
// failure.
void* scratch_address(const char** err) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *err = "no usable current device";
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr) {
      *err = cudaGetErrorString(e);
      return nullptr;
    }
    g_scratch_addr[dev] = ptr;
  }
  return g_scratch_addr[dev];
}

struct NoAllocLayout {
  int64_t off_qo, off_kv, off_len, off_merge, off_rows, off_items, off_lse, off_o, total;
};

int64_t up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

NoAllocLayout layout_for(int64_t batch, int64_t hk, int64_t hq, int64_t d, int64_t chunks) {
  NoAllocLayout L;
  int64_t off = kItemsOffset;
  L.off_items = off; off = up(off + int64_t(sizeof(WorkItem)) * batch * hk * chunks, 16);
  L.off_qo = off; off = up(off + 4 * (batch + 1), 16);
  L.off_kv = off; off = up(off + 4 * (batch + 1), 16);
  L.off_len = off; off = up(off + 4 * batch, 16);
  L.off_merge = off; off = up(off + 4 * (batch + 1), 16);
  L.off_rows = off; off = up(off + 4 * batch, 32);
  off = up(off, 256);
  L.off_lse = off; off = up(off + 4 * batch * chunks * hq, 256);
  L.off_o = off; off = up(off + 4 * batch * chunks * hq * d, 256);
  L.total = off;
  return L;
}

// Writes the whole plan into the scratch: header, per-request lengths from the
// device page metadata, and one work item per (request, kv head, chunk), the
// chunks cutting [0, kv_len) evenly. Nothing in the scratch is assumed to hold
// anything from an earlier call.
__global__ void noalloc_setup_kernel(uint8_t* ws, NoAllocLayout L, const int32_t* kv_indptr,
                                     const int32_t* last_page_len, int batch, int page_size,
                                     int hq, int hk, int d, int window_left, int chunks) {
  const int tid = blockIdx.x * blockDim.x + threadIdx.x;
  const int nthr = gridDim.x * blockDim.x;
  int32_t* qo = reinterpret_cast<int32_t*>(ws + L.off_qo);
  int32_t* kv = reinterpret_cast<int32_t*>(ws + L.off_kv);
  int32_t* len = reinterpret_cast<int32_t*>(ws + L.off_len);
  int32_t* merge = reinterpret_cast<int32_t*>(ws + L.off_merge);
  int32_t* rows = reinterpret_cast<int32_t*>(ws + L.off_rows);
  WorkItem* items = reinterpret_cast<WorkItem*>(ws + L.off_items);
  if (tid == 0) {
    WsHeader h;
    memset(&h, 0, sizeof h);
    h.n_items = batch * hk * chunks;
    h.n_merge_rows = chunks > 1 ? batch : 0;
    h.total_rows = batch;
    h.batch = batch;
    h.group = hq / hk;
    h.causal = 1;
    h.window_left = window_left;
    h.tile_rows = hq / hk;
    h.num_qo_heads = hq;
    h.head_dim = d;
    h.off_qo_indptr = L.off_qo;
    h.off_kv_indptr = L.off_kv;
    h.off_kv_len = L.off_len;
    h.off_merge_indptr = L.off_merge;
    h.off_merge_rows = L.off_rows;
    h.off_items = L.off_items;
    h.off_tmp_lse = L.off_lse;
    h.off_tmp_o = L.off_o;
    *reinterpret_cast<WsHeader*>(ws) = h;
  }
  for (int b = tid; b <= batch; b += nthr) {
    qo[b] = b;
    kv[b] = kv_indptr[b];
    merge[b] = chunks > 1 ? b * chunks : 0;
    if (b < batch) {
      const int pages = kv_indptr[b + 1] - kv_indptr[b];
      len[b] = pages > 0 ? (pages - 1) * page_size + last_page_len[b] : 0;
      rows[b] = b;
    }
  }
  for (int i = tid; i < batch * hk * chunks; i += nthr) {
    const int b = i / (hk * chunks);
    const int h = (i / chunks) % hk;
    const int c = i % chunks;
    const int pages = kv_indptr[b + 1] - kv_indptr[b];
    const int64_t lk = pages > 0 ? int64_t(pages - 1) * page_size + last_page_len[b] : 0;
    WorkItem it = {};
    it.b = b;
    it.kv_head = h;
    it.row0 = 0;
    it.kv_begin = int32_t(lk * c / chunks);
    it.kv_end = int32_t(lk * (c + 1) / chunks);
    it.chunk = chunks > 1 ? c : -1;
    it.num_chunks = chunks;
    it.partial_base = chunks > 1 ? b * chunks : -1;
    it.tok0 = b;
    it.lq = 1;
    it.lk = int32_t(lk);
    it.kv_start = kv_indptr[b];
    items[i] = it;
  }
}

thread_local char g_noalloc_err[256];

}  // namespace

}  // namespace fi

extern "C" const char* fi_noalloc_last_error(void) { return fi::g_noalloc_err; }

extern "C" size_t fi_noalloc_scratch_bytes(void) { return fi::kNoAllocScratchBytes; }

extern "C" fi_status fi_batch_decode_paged_noalloc(
    const fi_tensor* q, const fi_tensor* k_cache, const fi_tensor* v_cache,
    const fi_tensor* kv_indices, const int32_t* kv_indptr_dev, const int32_t* last_page_len_dev,
    int32_t batch, int32_t window_left, int32_t kv_chunks, float sm_scale, fi_tensor* out,
    fi_tensor* lse, void* stream) {
  using namespace fi;
  auto fail = [](fi_status s, const char* msg) {
    snprintf(g_noalloc_err, sizeof g_noalloc_err, "%s", msg);
    return s;
  };
  if (!q || !k_cache || !v_cache || !kv_indices || !out || !kv_indptr_dev || !last_page_len_dev ||
      !q->data || !k_cache->data || !v_cache->data || !kv_indices->data || !out->data)
    return fail(FI_ERR_INVALID_ARG, "decode_noalloc: a required pointer is NULL");
  if (q->ndim != 3 || k_cache->ndim != 4 || v_cache->ndim != 4 || out->ndim != 3 ||
      kv_indices->ndim != 1 || (lse && lse->ndim != 2))
    return fail(FI_ERR_INVALID_ARG, "decode_noalloc: q/out [B, Hq, d], caches [pages, P, Hk, d], "
                "kv_indices [n], lse [B, Hq]");
  const int hq = int(q->shape[1]), d = int(q->shape[2]);
  const int page_size = int(k_cache->shape[1]), hk = int(k_cache->shape[2]);
  if (batch < 0 || q->shape[0] < batch || out->shape[0] < batch || (lse && lse->shape[0] < batch))
    return fail(FI_ERR_INVALID_ARG, "decode_noalloc: q, out and lse need >= batch rows");
  if (hk <= 0 || hq % hk != 0)
    return fail(FI_ERR_GQA_INDIVISIBLE, "decode_noalloc: num_qo_heads is not a multiple of num_kv_heads");
  const int g = hq / hk;
  if ((g != 1 && g != 2 && g != 4) || (d != 64 && d != 128))
    return fail(FI_ERR_UNSUPPORTED, "decode_noalloc: GQA group 1, 2 or 4 and head_dim 64 or 128");
  if (q->dtype != k_cache->dtype || q->dtype != v_cache->dtype || q->dtype != out->dtype ||
      (q->dtype != FI_BF16 && q->dtype != FI_F16) || kv_indices->dtype != FI_I32 ||
      (lse && lse->dtype != FI_F32))
    return fail(FI_ERR_INVALID_ARG, "decode_noalloc: q/k/v/out share bf16 or fp16; lse is fp32");
  if (q->stride[2] != 1 || k_cache->stride[3] != 1 || v_cache->stride[3] != 1 ||
      kv_indices->stride[0] != 1)
    return fail(FI_ERR_STRIDED_LAST_DIM, "decode_noalloc: last dims must have stride 1");
  if (out->stride[2] != 1 || out->stride[1] != d || out->stride[0] != int64_t(hq) * d ||
      (lse && (lse->stride[1] != 1 || lse->stride[0] != hq)))
    return fail(FI_ERR_NONCONTIGUOUS_OUTPUT, "decode_noalloc: out and lse must be packed");
  if (k_cache->shape[0] != v_cache->shape[0])
    return fail(FI_ERR_INVALID_ARG, "decode_noalloc: k_cache and v_cache have different page counts");
  if (v_cache->shape[1] != page_size || v_cache->shape[2] != hk || v_cache->shape[3] != d ||
      k_cache->shape[3] != d || out->shape[1] != hq || out->shape[2] != d ||
      (lse && lse->shape[1] != hq))
    return fail(FI_ERR_INVALID_ARG, "decode_noalloc: shapes disagree");
  if (kv_chunks < 1 || kv_chunks > 64)
    return fail(FI_ERR_INVALID_ARG, "decode_noalloc: kv_chunks must be in [1, 64]");
  if (window_left < -1) return fail(FI_ERR_INVALID_ARG, "decode_noalloc: window_left < -1");
  if (!(sm_scale > 0.f)) return fail(FI_ERR_INVALID_ARG, "decode_noalloc: sm_scale must be > 0");
  auto a16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; };
  if (!a16(q->data) || !a16(k_cache->data) || !a16(v_cache->data) || !a16(out->data) ||
      q->stride[0] % 8 || q->stride[1] % 8 || k_cache->stride[0] % 8 || k_cache->stride[1] % 8 ||
      k_cache->stride[2] % 8 || v_cache->stride[0] % 8 || v_cache->stride[1] % 8 ||
      v_cache->stride[2] % 8)
    return fail(FI_ERR_UNSUPPORTED, "decode_noalloc: rows must start on 16-byte boundaries");
  const NoAllocLayout L = layout_for(batch, hk, hq, d, kv_chunks);
  if (L.total > int64_t(kNoAllocScratchBytes)) {
    snprintf(g_noalloc_err, sizeof g_noalloc_err,
             "decode_noalloc: batch=%d x kv_chunks=%d x heads=%d needs %lld bytes of scratch, "
             "more than the fixed %zu", batch, kv_chunks, hq, (long long)L.total,
             kNoAllocScratchBytes);
    return FI_ERR_CAPACITY;
  }
  if (batch == 0) return FI_OK;
  // once per device, with that device current: the array's device address
  // (the name g_noalloc_scratch in host code is only a stand-in for it)
  const char* why = nullptr;
  uint8_t* ws = static_cast<uint8_t*>(scratch_address(&why));
  if (!ws) {
    snprintf(g_noalloc_err, sizeof g_noalloc_err, "decode_noalloc: cudaGetSymbolAddress: %s", why);
    return FI_ERR_CUDA;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  noalloc_setup_kernel<<<64, 256, 0, s>>>(ws, L, kv_indptr_dev, last_page_len_dev, batch,
                                           page_size, hq, hk, d, window_left, kv_chunks);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(FI_ERR_CUDA, "decode_noalloc: setup launch failed");
  AttnParams ap;
  ap.q = q->data; ap.q_stride_tok = q->stride[0]; ap.q_stride_head = q->stride[1];
  ap.k = k_cache->data; ap.k_stride_page = k_cache->stride[0]; ap.k_stride_tok = k_cache->stride[1];
  ap.k_stride_head = k_cache->stride[2];
  ap.v = v_cache->data; ap.v_stride_page = v_cache->stride[0]; ap.v_stride_tok = v_cache->stride[1];
  ap.v_stride_head = v_cache->stride[2];
  ap.kv_indices = static_cast<const int32_t*>(kv_indices->data);
  ap.out = out->data;
  ap.lse = lse ? static_cast<float*>(lse->data) : nullptr;
  ap.ws = ws;
  ap.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  ap.num_qo_heads = hq;
  ap.num_kv_heads = hk;
  ap.page_size = page_size;
  ap.page_shift = -1;
  for (int sh = 0; sh < 31; ++sh)
    if ((1 << sh) == page_size) ap.page_shift = sh;
  ap.ragged = 0;
  ap.kv_rows = 0;
  ap.custom_mask = nullptr;
  const int grid = batch * hk * kv_chunks;
  e = launch_decode(ap, d, g, q->dtype == FI_BF16, k_cache->shape[0], g, grid, s);
  if (e != cudaSuccess) return fail(FI_ERR_CUDA, "decode_noalloc: decode launch failed");
  if (kv_chunks > 1) {
    e = launch_merge_workspace(ws, out->data, ap.lse, hq, d, q->dtype == FI_BF16,
                               (batch * hq + 7) / 8, s);
    if (e != cudaSuccess) return fail(FI_ERR_CUDA, "decode_noalloc: merge launch failed");
  }
  return FI_OK;
}

// The error flag of the last no-allocation decode on the current device: 1 when
// one of its bounded waits expired (that call's out / lse are not valid), else
// 0; 0 as well before the first call. Synchronises `stream`.
extern "C" fi_status fi_noalloc_device_error(int32_t* err_flag, int clear, void* stream) {
  using namespace fi;
  if (!err_flag) {
    snprintf(g_noalloc_err, sizeof g_noalloc_err, "noalloc_device_error: err_flag is NULL");
    return FI_ERR_INVALID_ARG;
  }
  *err_flag = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    snprintf(g_noalloc_err, sizeof g_noalloc_err, "noalloc_device_error: no usable current device");
    return FI_ERR_CUDA;
  }
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    base = g_scratch_addr[dev];
  }
  if (!base) return FI_OK;  // no call on this device yet
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* flag = static_cast<uint8_t*>(base) + offsetof(WsHeader, err_flag);
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, flag, sizeof v, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && clear) e = cudaMemsetAsync(flag, 0, sizeof v, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    snprintf(g_noalloc_err, sizeof g_noalloc_err, "noalloc_device_error: %s", cudaGetErrorString(e));
    return FI_ERR_CUDA;
  }
  *err_flag = v ? 1 : 0;
  return FI_OK;
}
