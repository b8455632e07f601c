// Short-query attention: the launchers of the kernels in decode_kernel.cuh
// (the ring, the producer and both consumers are described there).
#include "decode_kernel.cuh"

namespace fi {
namespace {

// the tensor-core consumer for groups 1, 2, 4, 8, 16: one or two row halves
// of one M tile (the 32-row pair consumer launches from decode_pair.cu)
template <int D, bool BF16>
cudaError_t launch_mma(const AttnParams& p, int group, int rh, int grid, const CUtensorMap& tk,
                       const CUtensorMap& tv, int box_rows, cudaStream_t s) {
#define FI_MMA_CASE(G)                                                                     \
  case G:                                                                                  \
    return rh == 1 ? launch_k<D, G, BF16, true, 1>(p, grid, tk, tv, box_rows, s)           \
                   : launch_k<D, G, BF16, true, 2>(p, grid, tk, tv, box_rows, s);
  switch (group) {
    FI_MMA_CASE(1)
    FI_MMA_CASE(2)
    FI_MMA_CASE(4)
    FI_MMA_CASE(8)
    case 16: return launch_k<D, 16, BF16, true, 2>(p, grid, tk, tv, box_rows, s);
    default: return cudaErrorInvalidValue;
  }
#undef FI_MMA_CASE
}

template <int D, bool BF16>
cudaError_t launch_shuffle(const AttnParams& p, int group, int grid, const CUtensorMap& tk,
                           const CUtensorMap& tv, int box_rows, cudaStream_t s) {
  switch (group) {
    case 1: return launch_k<D, 1, BF16, false, 1>(p, grid, tk, tv, box_rows, s);
    case 2: return launch_k<D, 2, BF16, false, 1>(p, grid, tk, tv, box_rows, s);
    case 4: return launch_k<D, 4, BF16, false, 1>(p, grid, tk, tv, box_rows, s);
    default: return cudaErrorInvalidValue;
  }
}

int gcd_int(int a, int b) {
  while (b) {
    const int t = a % b;
    a = b;
    b = t;
  }
  return a;
}

int stage_keys(int head_dim) { return head_dim == 128 ? TmaCfg<128, true>::KT : TmaCfg<64, true>::KT; }

}  // namespace

bool decode_mma_supports(int head_dim, int page_size, int group) {
  if (head_dim != 64 && head_dim != 128) return false;
  if (group != 1 && group != 2 && group != 4 && group != 8 && group != 16) return false;
  return gcd_int(page_size, stage_keys(head_dim)) >= 8;
}

bool decode_shuffle_supports(int head_dim, int group) {
  return (head_dim == 64 || head_dim == 128) && (group == 1 || group == 2 || group == 4);
}

int decode_ctas_per_sm(int head_dim, int page_size, int group) {
  const bool mma = decode_mma_supports(head_dim, page_size, group);
  if (head_dim == 64) return mma ? TmaCfg<64, true>::MINB : TmaCfg<64, false>::MINB;
  return mma ? TmaCfg<128, true>::MINB : TmaCfg<128, false>::MINB;
}

cudaError_t launch_decode(const AttnParams& p, int head_dim, int group, bool bf16,
                          int64_t num_pages, int tile_rows, int grid, cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  if (head_dim != 128 && head_dim != 64) return cudaErrorInvalidValue;
  // Boxes of gcd(page_size, KT) slots never cross a page: every box starts
  // at a multiple of that size (tiles start at lo rounded down to it).
  const int box_rows = gcd_int(p.page_size, stage_keys(head_dim));
  const bool mma = decode_mma_supports(head_dim, p.page_size, group);
  if (!mma && !(decode_shuffle_supports(head_dim, group) && tile_rows == group))
    return cudaErrorInvalidValue;
  if (tile_rows < 1 || tile_rows > (mma ? 32 : 16)) return cudaErrorInvalidValue;
  const int rh = tile_rows > 16 ? 4 : tile_rows > 8 ? 2 : 1;
  const int box_cols = mma ? 64 : head_dim;
  const CUtensorMapSwizzle swz = mma ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  CUtensorMap tk, tv;
  if ((!p.ragged && num_pages <= 0) ||
      !encode_kv_map(&tk, p, true, bf16, head_dim, num_pages, box_cols, box_rows, swz) ||
      !encode_kv_map(&tv, p, false, bf16, head_dim, num_pages, box_cols, box_rows, swz))
    return cudaErrorInvalidValue;
  if (mma && rh == 4)
    return launch_decode_pair(p, head_dim, group, bf16, grid, tk, tv, box_rows, stream);
  if (mma) {
    if (head_dim == 128)
      return bf16 ? launch_mma<128, true>(p, group, rh, grid, tk, tv, box_rows, stream)
                  : launch_mma<128, false>(p, group, rh, grid, tk, tv, box_rows, stream);
    return bf16 ? launch_mma<64, true>(p, group, rh, grid, tk, tv, box_rows, stream)
                : launch_mma<64, false>(p, group, rh, grid, tk, tv, box_rows, stream);
  }
  if (head_dim == 128)
    return bf16 ? launch_shuffle<128, true>(p, group, grid, tk, tv, box_rows, stream)
                : launch_shuffle<128, false>(p, group, grid, tk, tv, box_rows, stream);
  return bf16 ? launch_shuffle<64, true>(p, group, grid, tk, tv, box_rows, stream)
              : launch_shuffle<64, false>(p, group, grid, tk, tv, box_rows, stream);
}

}  // namespace fi
