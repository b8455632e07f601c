// Launches of the short-query kernel's 32-row pair consumer
// (decode_kernel.cuh), in a translation unit of their own.
#include "decode_kernel.cuh"

namespace fi {

cudaError_t launch_decode_pair(const AttnParams& p, int head_dim, int group, bool bf16, int grid,
                               const CUtensorMap& tk, const CUtensorMap& tv, int box_rows,
                               cudaStream_t s) {
#define FI_PAIR_CASE(D, BF)                                                                 \
  switch (group) {                                                                          \
    case 1: return launch_k<D, 1, BF, true, 4>(p, grid, tk, tv, box_rows, s);               \
    case 2: return launch_k<D, 2, BF, true, 4>(p, grid, tk, tv, box_rows, s);               \
    case 4: return launch_k<D, 4, BF, true, 4>(p, grid, tk, tv, box_rows, s);               \
    case 8: return launch_k<D, 8, BF, true, 4>(p, grid, tk, tv, box_rows, s);               \
    case 16: return launch_k<D, 16, BF, true, 4>(p, grid, tk, tv, box_rows, s);             \
    default: return cudaErrorInvalidValue;                                                  \
  }
  if (head_dim == 128) {
    if (bf16) { FI_PAIR_CASE(128, true) }
    FI_PAIR_CASE(128, false)
  }
  if (head_dim == 64) {
    if (bf16) { FI_PAIR_CASE(64, true) }
    FI_PAIR_CASE(64, false)
  }
#undef FI_PAIR_CASE
  return cudaErrorInvalidValue;
}

}  // namespace fi
