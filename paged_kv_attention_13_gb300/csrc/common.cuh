// Device helpers shared by the libfi kernels: 16-bit float conversion, cached
// and streaming loads, cp.async, ldmatrix / mma.sync wrappers, exp2.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "fi_internal.h"

namespace fi {

constexpr float kLn2 = 0.69314718055994530942f;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// 2^x on the SFU (the PTX ex2.approx instruction; -inf -> +0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

template <bool BF16> struct Dt;
template <> struct Dt<true> {
  using T = __nv_bfloat16;
  using T2 = __nv_bfloat162;
  __device__ __forceinline__ static float lo(uint32_t w) { return __uint_as_float(w << 16); }
  __device__ __forceinline__ static float hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
  __device__ __forceinline__ static uint32_t pack(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ __forceinline__ static T from_float(float x) { return __float2bfloat16_rn(x); }
};
template <> struct Dt<false> {
  using T = __half;
  using T2 = __half2;
  __device__ __forceinline__ static float lo(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu)));
  }
  __device__ __forceinline__ static float hi(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
  }
  __device__ __forceinline__ static uint32_t pack(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ __forceinline__ static T from_float(float x) { return __float2half_rn(x); }
};

// 16-byte load that bypasses L1 allocation (KV is read once per item).
__device__ __forceinline__ uint4 ld_stream16(const void* ptr) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(ptr));
  return r;
}

__device__ __forceinline__ uint4 ld_nc16(const void* ptr) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(ptr));
  return r;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// cp.async 16 bytes; src_bytes = 0 zero-fills the destination.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A(16x16, row) * B(16x8, col), fp32 accumulate.
template <bool BF16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// Bit (i * lk + j) of a request's custom mask, whose bits start at byte
// `base` (least significant bit first).
__device__ __forceinline__ bool custom_mask_bit(const uint8_t* mask, int base, int i, int j,
                                                int lk) {
  const int64_t n = int64_t(i) * lk + j;
  return (__ldg(mask + base + (n >> 3)) >> (n & 7)) & 1;
}

// 32 consecutive bits n0 .. n0+31 of a request's custom mask (least
// significant bit first within each byte), as bits 0..31 of the result; bits
// at or past nbits (the segment's Lq * Lk bits) and before 0 read as 0.
__device__ __forceinline__ uint32_t custom_mask_word(const uint8_t* seg, int64_t nbits,
                                                     int64_t n0) {
  const int64_t b0 = n0 >> 3;
  const int64_t nbytes = (nbits + 7) >> 3;
  uint64_t w = 0;
#pragma unroll
  for (int q = 0; q < 5; ++q) {
    const int64_t bi = b0 + q;
    const uint64_t v = (bi >= 0 && bi < nbytes) ? __ldg(seg + bi) : 0u;
    w |= v << (8 * q);
  }
  return uint32_t(w >> (n0 & 7));
}

// Key j of a request: its row in the cache (page from the page table), or
// with a ragged cache, row kv_start + j.
__device__ __forceinline__ int64_t kv_row_offset(const int32_t* pages, int32_t j, int page_size,
                                                 int page_shift, int64_t stride_page,
                                                 int64_t stride_tok, bool ragged, int kv_start) {
  if (ragged) return int64_t(kv_start + j) * stride_tok;
  int32_t pi, slot;
  if (page_shift >= 0) {
    pi = j >> page_shift;
    slot = j & ((1 << page_shift) - 1);
  } else {
    pi = j / page_size;
    slot = j - pi * page_size;
  }
  const int64_t page = __ldg(pages + pi);
  return page * stride_page + int64_t(slot) * stride_tok;
}

}  // namespace fi
