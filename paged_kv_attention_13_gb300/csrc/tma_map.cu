// Host side of the TMA copies: tensor maps encoded through the runtime's
// driver entry point for cuTensorMapEncodeTiled (no link against libcuda).
#include "tma.cuh"

namespace fi {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(ptr);
  }();
  return fn;
}

}  // namespace

bool encode_tensor_map(CUtensorMap* m, bool bf16, int rank, const void* base,
                       const cuuint64_t* dims, const cuuint64_t* strides_bytes,
                       const cuuint32_t* box, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  cuuint32_t(rank), const_cast<void*>(base), dims, strides_bytes, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_paged_kv_map(CUtensorMap* m, bool bf16, const void* base, int head_dim,
                         int num_kv_heads, int page_size, int64_t num_pages, int64_t stride_head,
                         int64_t stride_tok, int64_t stride_page, int box_cols, int box_rows,
                         CUtensorMapSwizzle swizzle) {
  cuuint64_t dims[4] = {cuuint64_t(head_dim), cuuint64_t(num_kv_heads), cuuint64_t(page_size),
                        cuuint64_t(num_pages)};
  cuuint64_t str[3] = {cuuint64_t(stride_head) * 2, cuuint64_t(stride_tok) * 2,
                       cuuint64_t(stride_page) * 2};
  cuuint32_t box[4] = {cuuint32_t(box_cols), 1, cuuint32_t(box_rows), 1};
  return encode_tensor_map(m, bf16, 4, base, dims, str, box, swizzle);
}

bool encode_kv_map(CUtensorMap* m, const AttnParams& p, bool is_k, bool bf16, int head_dim,
                   int64_t num_pages, int box_cols, int box_rows, CUtensorMapSwizzle swizzle) {
  const void* base = is_k ? p.k : p.v;
  const int64_t sh = is_k ? p.k_stride_head : p.v_stride_head;
  const int64_t st = is_k ? p.k_stride_tok : p.v_stride_tok;
  if (p.ragged) {
    if (p.kv_rows <= 0 || p.kv_rows > (int64_t(1) << 31)) return false;
    return encode_paged_kv_map(m, bf16, base, head_dim, p.num_kv_heads, int(p.kv_rows), 1, sh, st,
                               st * p.kv_rows, box_cols, box_rows, swizzle);
  }
  const int64_t sp = is_k ? p.k_stride_page : p.v_stride_page;
  return encode_paged_kv_map(m, bf16, base, head_dim, p.num_kv_heads, p.page_size, num_pages, sh,
                             st, sp, box_cols, box_rows, swizzle);
}

}  // namespace fi
