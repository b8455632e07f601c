// Tensor Memory Accelerator (TMA) copies and mbarrier waits shared by the
// kernels that stage K/V pages with cp.async.bulk.tensor, plus the host side
// that encodes the tensor maps.
//
// Every wait is bounded in time: on expiry it raises the CTA's abort flag and
// returns false, so a kernel never spins forever on a copy that does not land.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "common.cuh"

namespace fi {

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per wait

// Shared by the threads of one CTA: the abort flag that an expired wait
// raises (every later wait then returns false at once) and the limit of each
// wait. The limit comes from the workspace header (0 there means kWaitLimitNs);
// waits that drain a CTA's own copies before it exits use a private block with
// the default limit, so they still wait for those copies.
struct WaitCtl {
  int abort;
  int pad;
  unsigned long long limit_ns;
};

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `parity` to complete; false on timeout or abort.
// try_wait itself suspends the thread for a while before it reports that
// the phase is still open, so the abort flag and the clock are looked at
// after every failed poll.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile WaitCtl* ctl) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (ctl->abort) return false;
    if (globaltimer() - t0 > ctl->limit_ns) {
      ctl->abort = 1;
      return false;
    }
  }
}

// The wait limit of a launch: the header's, or kWaitLimitNs when it is 0.
__device__ __forceinline__ unsigned long long wait_limit_of(const WsHeader* hdr) {
  const unsigned long long l = hdr->wait_limit_ns;
  return l ? l : kWaitLimitNs;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y, int z, int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}

// Plain bulk copy global -> shared (no tensor map); both addresses 16-byte
// aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// Host: cuTensorMapEncodeTiled through the runtime's driver entry point (no
// link against libcuda). 16-bit elements; false when the driver refuses the
// shape, strides or box.
bool encode_tensor_map(CUtensorMap* m, bool bf16, int rank, const void* base,
                       const cuuint64_t* dims, const cuuint64_t* strides_bytes,
                       const cuuint32_t* box, CUtensorMapSwizzle swizzle);

// Host: the 4-D map over a paged K or V cache, dims (innermost first)
// [head_dim, kv head, slot in page, page], with a box of `box_cols` dims x
// `box_rows` slots of one head of one page.
bool encode_paged_kv_map(CUtensorMap* m, bool bf16, const void* base, int head_dim,
                         int num_kv_heads, int page_size, int64_t num_pages, int64_t stride_head,
                         int64_t stride_tok, int64_t stride_page, int box_cols, int box_rows,
                         CUtensorMapSwizzle swizzle);

// Host: the 4-D map of K (is_k) or V for a run: over the paged cache as
// above, or, with a ragged cache, over [rows, kv head, dim] as one logical
// page of p.kv_rows slots (dims [head_dim, kv head, rows, 1]).
bool encode_kv_map(CUtensorMap* m, const AttnParams& p, bool is_k, bool bf16, int head_dim,
                   int64_t num_pages, int box_cols, int box_rows, CUtensorMapSwizzle swizzle);

}  // namespace fi
