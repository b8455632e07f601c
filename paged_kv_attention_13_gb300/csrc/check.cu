// Opt-in range check of a plan's page table (FI_CHECK_INDICES, and the
// fi_check_kv_indices entry point). A page index outside the cache is what
// turns a wrong page table into a memory fault ("Refuse attention inputs the
// ROCm kernels would compute wrongly" (#399) and "Support speculative-decode
// verify on ROCm ..." (#362), "Review notes": a wrong indptr faults the
// merge). Here such an entry is counted in the workspace header instead; the
// attention kernels and the merge of the same run read the count and do no
// work, and fi_plan_device_error reports it. Nothing traps.
#include "fi_internal.h"

namespace fi {
namespace {

// Entries [0, kv_indptr[batch]) of the page table, the count read from the
// plan's workspace on the device, so a captured run checks each re-plan's
// table.
__global__ void __launch_bounds__(256) check_indices_kernel(void* ws, const int32_t* kv_indices,
                                                            int64_t num_pages) {
  WsHeader* hdr = static_cast<WsHeader*>(ws);
  const int32_t* kv_indptr = ws_ptr<const int32_t>(ws, hdr->off_kv_indptr);
  const int64_t n = kv_indptr[hdr->batch];
  int bad = 0;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int32_t v = __ldg(kv_indices + i);
    bad += (v < 0 || int64_t(v) >= num_pages) ? 1 : 0;
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, off);
  if ((threadIdx.x & 31) == 0 && bad) atomicAdd(&hdr->index_error, bad);
}

}  // namespace

cudaError_t launch_check_indices(void* ws, const int32_t* kv_indices, int64_t num_pages,
                                 int num_sms, cudaStream_t stream) {
  check_indices_kernel<<<num_sms > 0 ? num_sms : 1, 256, 0, stream>>>(ws, kv_indices, num_pages);
  return cudaGetLastError();
}

}  // namespace fi
