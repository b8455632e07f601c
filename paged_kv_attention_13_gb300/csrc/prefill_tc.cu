// Prefill kernel on the 5th-generation tensor cores: TMA page gathers into
// 128B-swizzled shared memory, tcgen05.mma with S, P and O in tensor memory,
// one thread per query row for the online softmax.
//
// A work item is two 128-row Q tiles (packed rows: query row x head in the
// GQA group, all heads of one kv head) against a range of 128-key tiles,
// head_dim 64 or 128, bf16 or fp16 in, fp32 accumulate. Both Q tiles use every
// K/V tile staged in shared memory. An item carries its request's metadata.
//
// Roles inside one CTA (384 threads, one CTA per SM, persistent over the work
// items of the plan):
//   warp 0      TMA producer of the two Q tiles (3-D map over [tokens, heads,
//               dim]) and, per key tile, one box per page of K (4-D map over
//               [pages, slot, kv head, dim]) straight from the paged cache;
//               it also prefetches the next item's Q tiles into L2;
//   warp 2      TMA producer of V, the same way, at its own pace (two K and
//               two V stages, released separately);
//   warp 1      MMA issuer (one thread): S_x = Q_x K^T into TMEM, then
//               O_x += P_x V with P_x read from TMEM, alternating the tiles so
//               the tensor core works on one tile while the other's softmax
//               runs; warp 3 only gives up its registers;
//   warps 4-7   softmax of tile A, warps 8-11 softmax of tile B: a thread owns
//               one row (its TMEM lane), masks boundary tiles, keeps the
//               running max / sum in registers, rescales O in TMEM only when
//               the max grows by more than 2^8, writes P over its S columns,
//               and runs the epilogue, whose output rows pass through a
//               per-warp shared-memory staging buffer.
// Every mbarrier wait is bounded in time; on expiry the CTA records an error
// in the workspace header, stops issuing work, waits for its own copies and
// MMAs in flight, frees its tensor memory and exits.
//
// Mask ("Route non-causal windowed prefill to AITER's masked kernel" (#339),
// "Why window_size_right stays -1"; "Support speculative-decode verify on
// ROCm ..." (#362), "Summary"): key j of query row i is kept when
// (!causal || j <= i + Lk - Lq) && (wl < 0 || j + Lq + wl >= Lk + i). Key
// tiles outside the item's live range are never loaded; the per-element
// test runs on tiles that straddle a bound only.
#include <type_traits>

#include "tma.cuh"

namespace fi {
namespace {

constexpr int kTcThreads = 384;  // 4 control warps + 2 softmax warpgroups
constexpr int kBlk = 128 * 128;  // 128 rows x 128 bytes: one 64-column swizzled block

// K and V stages (a third V or a third K stage, 32 KB more shared memory,
// measured no faster on the long-context split prefill once K and V have
// their own producer warps)
constexpr int kNK = 2, kNV = 2;
static_assert(kNK <= 4 && kNV <= 4, "a producer's stage bits");

// Shared-memory layout for head_dim D (64 or 128): a tile is 128 rows of D
// 16-bit columns, D / 64 swizzled blocks; Q tiles A and B, the K and V
// stages, the barriers, and the rows handed between the warpgroups.
template <int D>
struct TcLayout {
  static constexpr int kH = D / 64;
  static constexpr int kTile = kH * kBlk;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 2 * kTile;
  static constexpr int kOffV = kOffK + kNK * kTile;
  static constexpr int kOffBar = kOffV + kNV * kTile;
  static constexpr int kOffMl = kOffBar + 256;
  // per softmax warp, 32 rows x 128 bytes: output rows pass through it so the
  // stores to global memory cover whole 128-byte lines
  static constexpr int kOffStage = kOffMl + 1024;
  static constexpr int kSmem = kOffStage + 8 * 4096 + 1024;  // + alignment slack
};

// barrier slots
constexpr int B_QFULL = 0, B_QEMPTY = 1, B_KFULL = 2, B_KEMPTY = B_KFULL + kNK,
              B_VFULL = B_KEMPTY + kNK, B_VEMPTY = B_VFULL + kNV, B_SFULL = B_VEMPTY + kNV,
              B_PFULL = B_SFULL + 2, B_ODONE = B_PFULL + 2, B_OFREE = B_ODONE + 2,
              B_FINAL = B_OFREE + 2, B_MLFULL = B_FINAL + 1, B_MLFREE = B_MLFULL + 1,
              N_BARS = B_MLFREE + 1;
static_assert(8 * N_BARS + 8 + 16 <= 256, "barriers, the TMEM slot and the wait control fit");

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// Wait for outstanding TMEM loads; the registers of `r` are tied to the wait,
// so no use of them can be scheduled above it.
__device__ __forceinline__ void tmem_wait_ld_tied(uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
        "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
        "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
        "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
        "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
      :
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start, leading and stride
// byte offsets in 16-byte units, version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFFu);
  d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
  d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(2) << 61;
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulate, A/B fp16 or bf16, A
// K-major, B K-major (S = Q K^T) or MN-major (O += P V), M x N.
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, bool b_mn_major, int M, int N) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((b_mn_major ? 1u : 0u) << 16) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

struct ItemGeom {
  int b, hk, token0, lq, lk, n_rows, i0, kv_lo, kv_hi, t_start, n_tiles;
  int chunk, num_chunks, partial_base, row0;
  int kv_start;   // the request's first page-table entry (ragged cache: first K/V row)
  int mask_base;  // first byte of the request's custom mask
};

// A work item in four 16-byte loads issued together: it carries its
// request's metadata, so nothing else is read before its geometry is known.
__device__ __forceinline__ WorkItem load_item(const WorkItem* items, int w) {
  WorkItem it;
  const int4* src = reinterpret_cast<const int4*>(items + w);
  int4* dst = reinterpret_cast<int4*>(&it);
#pragma unroll
  for (int i = 0; i < 4; ++i) dst[i] = __ldg(src + i);
  return it;
}

__device__ __forceinline__ ItemGeom item_geom(const WorkItem& it, int g, int tile_rows,
                                              int causal, int wl, int align) {
  ItemGeom G;
  G.b = it.b; G.hk = it.kv_head; G.row0 = it.row0;
  G.token0 = it.tok0;
  G.lq = it.lq;
  G.lk = it.lk;
  G.n_rows = min(tile_rows, G.lq * g - it.row0);
  G.i0 = it.row0 / g;
  const int i1 = (it.row0 + G.n_rows) / g - 1;
  const int hi_t = causal ? min(G.lk, i1 + G.lk - G.lq + 1) : G.lk;
  const int lo_t = wl >= 0 ? max(0, G.lk - G.lq + G.i0 - wl) : 0;
  G.kv_lo = max(it.kv_begin, lo_t);
  G.kv_hi = min(it.kv_end, hi_t);
  // the first key tile starts on the TMA box boundary at or below the first
  // live key (a box never crosses a page), not on a multiple of 128, so it
  // holds at most align - 1 keys before the first live one: a sliding window
  // of 127 keys over 64 query tokens then takes 2 tiles, not 2 or 3
  G.t_start = (G.kv_lo / align) * align;
  G.n_tiles = G.kv_lo < G.kv_hi ? (G.kv_hi - G.t_start + 127) / 128 : 0;
  G.chunk = it.chunk; G.num_chunks = it.num_chunks; G.partial_base = it.partial_base;
  G.kv_start = it.kv_start;
  G.mask_base = it.mask_base;
  return G;
}

// Bring a 3-D box of a tensor map into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}

// 16 packed columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// O += P V with P (the A operand) read from tensor memory.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// Two Q tiles per CTA (A: packed rows [row0, row0+tr), B: the next tr rows)
// share every K/V tile, which halves the K/V bytes per FLOP. The tensor core
// alternates between them - S_A(j+1) and PV_B(j) run while softmax A works,
// PV_A(j+1) and S_B(j+1) while softmax B works - and P is written back into
// tensor memory over the S columns it came from.
// An item of one Q tile and at least two key tiles is split instead: both
// warpgroups run the same rows, A on the even key tiles and B on the odd
// ones, each with its own S/P and O in tensor memory, and at the end A
// combines the two states (m, l, O) by their maxima and writes the output.
// MASKED: the plan carries a custom mask (a separate build of the kernel, so
// the unmasked softmax keeps its registers).
template <bool BF16, int D, bool MASKED>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tq,
                      const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                      int kv_box_rows) {
  using DT = Dt<BF16>;
  using T = typename DT::T;
  using L = TcLayout<D>;
  constexpr int kH = L::kH, kTile = L::kTile, kOffQ = L::kOffQ, kOffK = L::kOffK,
                kOffV = L::kOffV, kOffBar = L::kOffBar, kOffMl = L::kOffMl,
                kOffStage = L::kOffStage;
  // the page table failed the index check: the whole CTA leaves before any
  // barrier, tensor-memory allocation or copy
  if (static_cast<const WsHeader*>(p.ws)->index_error) return;
  extern __shared__ uint8_t smem_raw[];
  uint32_t sbase = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (sbase & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  sbase += pad;
  const uint32_t bar0 = sbase + kOffBar;
  auto BAR = [&](int i) { return bar0 + 8u * uint32_t(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * N_BARS);
  volatile WaitCtl* ctl = reinterpret_cast<volatile WaitCtl*>(smem + kOffBar + 8 * N_BARS + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const WsHeader* hdr = static_cast<const WsHeader*>(p.ws);
  const int n_items = hdr->n_items;
  const WorkItem* items = ws_ptr<const WorkItem>(p.ws, hdr->off_items);
  float* tmp_lse = ws_ptr<float>(p.ws, hdr->off_tmp_lse);
  float* tmp_o = ws_ptr<float>(p.ws, hdr->off_tmp_o);
  const int g = hdr->group;
  const int causal = hdr->causal;
  const int wl = hdr->window_left;
  const int tile_rows = hdr->tile_rows;  // two Q tiles
  const int tr = tile_rows / 2;          // rows of one Q tile
  const int Hq = p.num_qo_heads;

  if (threadIdx.x == 0) {
    mbar_init(BAR(B_QFULL), 1);
    mbar_init(BAR(B_QEMPTY), 1);
    for (int s = 0; s < kNV; ++s) {
      mbar_init(BAR(B_VFULL + s), 1);
      mbar_init(BAR(B_VEMPTY + s), 1);
    }
    for (int s = 0; s < kNK; ++s) {
      mbar_init(BAR(B_KFULL + s), 1);
      mbar_init(BAR(B_KEMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(BAR(B_SFULL + s), 1);
      mbar_init(BAR(B_PFULL + s), 128);
      mbar_init(BAR(B_ODONE + s), 1);
      mbar_init(BAR(B_OFREE + s), 128);
    }
    mbar_init(BAR(B_FINAL), 1);
    mbar_init(BAR(B_MLFULL), 128);
    mbar_init(BAR(B_MLFREE), 128);
    ctl->abort = 0;
    ctl->limit_ns = wait_limit_of(hdr);
    mbar_init_fence();
  }
  // K/V stages start zeroed so rows no copy has written yet hold finite values
  for (int i = threadIdx.x; i < ((kNK + kNV) * kTile) / 16; i += kTcThreads)
    reinterpret_cast<uint4*>(smem + kOffK)[i] = make_uint4(0, 0, 0, 0);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                     smem_u32(tmem_slot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Register split: the control warpgroup (producer, MMA issuer, two idle
  // warps) gives registers to the two softmax warpgroups, which hold a whole
  // 128-column score row: 128 x 104 + 256 x 200 = 64512 = 384 x 168 launched.
  // The compiler allocates each side to its own limit; at 192 the softmax
  // spilled to local memory.
  if (warp < 4) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 104;" ::: "memory");
  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------ producers
    // Warp 0 loads the Q tiles and the K tiles, warp 2 the V tiles, each at
    // its own pace: a V stage is released only after its P V product, long
    // after the K stage of the same tile, and one warp issuing both waited
    // on V slots while K slots stood free (split items of the long-context
    // batch streamed at 0.7 of the HBM rate). Lane 0 owns the warp's
    // barriers; for each tile every lane fetches one page index (up to 8
    // pages per tile) and issues that page's boxes.
    const int which_w = warp == 0 ? 0 : 1;
    int gcnt = 0, qc = 0;
    // stage (which, st) at bit 4 * which + st: armed at least once, and the
    // parity of its latest arming (bit masks, so they stay in registers)
    uint32_t armed = 0, apar = 0;
    bool q_armed = false;
    uint32_t q_par = 0;
    bool ok = true;
    const int npg = 128 / kv_box_rows;
    // page and slot of key k (page_shift >= 0: a power-of-two page size)
    const int pshift = p.page_shift, pmask = pshift >= 0 ? (1 << pshift) - 1 : 0;
    auto page_of = [&](int k) { return pshift >= 0 ? (k >> pshift) : k / p.page_size; };
    auto slot_of = [&](int k) { return pshift >= 0 ? (k & pmask) : k % p.page_size; };
    const int tiles_per_batch = 32 / npg;  // page indices the warp holds per batch of tiles
    // issue K (which = 0) or V (which = 1) of tile t, whose page index this
    // lane holds in `page` (valid when `has`)
    auto load = [&](int which, const ItemGeom& G, int t, int cntr, bool has, int page,
                    int nvalid) {
      const int ns = which ? kNV : kNK;
      const int st = cntr % ns, fill = cntr / ns;  // the stage's fill-th use
      const int t0 = G.t_start + t * 128;
      const int full = which ? B_VFULL : B_KFULL, empty = which ? B_VEMPTY : B_KEMPTY;
      bool okl = true;
      if (lane == 0) {
        if (fill >= 1 && !mbar_wait(BAR(empty + st), (fill - 1) & 1, ctl)) okl = false;
        if (okl) {
          mbar_expect_tx(BAR(full + st), uint32_t(nvalid) * uint32_t(kv_box_rows) * uint32_t(D) * 2u);
          const uint32_t bit = 1u << (4 * which + st);
          armed |= bit;
          apar = (fill & 1) ? (apar | bit) : (apar & ~bit);
        }
      }
      okl = __shfl_sync(0xffffffffu, okl, 0);
      if (okl && has) {
        // box `lane` covers keys t0 + lane * kv_box_rows onwards, inside one
        // page (kv_box_rows divides the page size); ragged: one logical page
        // per request, the slot is the row
        const int slot0 = p.ragged ? G.kv_start + t0 : slot_of(t0 + lane * kv_box_rows);
        const uint32_t roff = uint32_t(lane * kv_box_rows) * 128u;
        const uint32_t dst = sbase + (which ? kOffV : kOffK) + st * kTile + roff;
        for (int h = 0; h < kH; ++h)
          tma_load_4d(dst + h * kBlk, which ? &tv : &tk, BAR(full + st), h * 64, G.hk, slot0, page);
      }
      return okl;
    };
    WorkItem nit{};
    nit.b = -1;
    if (int(blockIdx.x) < n_items) nit = load_item(items, blockIdx.x);
    for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
      const WorkItem it = nit;  // this item, loaded one item ahead
      if (w + int(gridDim.x) < n_items) nit = load_item(items, w + gridDim.x);
      if (it.b < 0) continue;  // schedule padding
      const ItemGeom G = item_geom(it, g, tile_rows, causal, wl, kv_box_rows);
      if (G.n_tiles == 0) continue;
      const bool hasB = G.n_rows > tr;
      const int32_t* pages = p.ragged ? nullptr : p.kv_indices + G.kv_start;
      // the request's pages (every page but the last is full); ragged: rows
      const int n_pages = p.ragged ? G.lk : (G.lk + p.page_size - 1) / p.page_size;
      // page index of lane L for batch bt: tile bt * tiles_per_batch + L / npg,
      // its page L % npg (0 when past the request)
      auto fetch = [&](int bt) {
        const int t = bt * tiles_per_batch + lane / npg;
        const int pg = page_of(G.t_start + t * 128 + (lane % npg) * kv_box_rows);
        if (p.ragged) return 0;
        return (t < G.n_tiles && pg < n_pages && lane < tiles_per_batch * npg) ? __ldg(pages + pg) : 0;
      };
      int idx_cur = fetch(0), idx_nxt = fetch(1);
      if (which_w == 0 && lane == 0) {
        if (qc > 0 && !mbar_wait(BAR(B_QEMPTY), (qc - 1) & 1, ctl)) ok = false;
        if (ok) {
          mbar_expect_tx(BAR(B_QFULL), (hasB ? 2u : 1u) * uint32_t(tr) * uint32_t(D) * 2u);
          q_armed = true;
          q_par = qc & 1;
          for (int x = 0; x < (hasB ? 2 : 1); ++x)
            for (int h = 0; h < kH; ++h)
              tma_load_3d(sbase + kOffQ + x * kTile + h * kBlk, &tq, BAR(B_QFULL), h * 64,
                          G.hk * g, G.token0 + G.i0 + x * (tr / g));
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ++qc;
      for (int step = 0; step < G.n_tiles && ok; ++step) {
        const int bt = step / tiles_per_batch, k = step % tiles_per_batch;
        if (k == 0 && bt > 0) {  // move to the next batch, prefetch the one after
          idx_cur = idx_nxt;
          idx_nxt = fetch(bt + 1);
        }
        const bool has = lane < npg && page_of(G.t_start + step * 128 + lane * kv_box_rows) < n_pages;
        const int page = __shfl_sync(0xffffffffu, idx_cur, (k * npg + lane) & 31);
        const int nvalid = __popc(__ballot_sync(0xffffffffu, has));
        ok = load(which_w, G, step, gcnt, has, page, nvalid);
        ++gcnt;
      }
      // once this item's K tiles are issued, the Q tiles of the CTA's next
      // item go to L2, so their copy into shared memory, which waits for this
      // item's last S product, is an L2 read rather than an HBM one
      if (which_w == 0 && lane == 0 && ok) {
        for (int w2 = w + gridDim.x; w2 < n_items; w2 += gridDim.x) {
          const WorkItem it2 = load_item(items, w2);
          if (it2.b < 0) continue;
          const ItemGeom G2 = item_geom(it2, g, tile_rows, causal, wl, kv_box_rows);
          if (G2.n_tiles == 0) continue;
          for (int x = 0; x < (G2.n_rows > tr ? 2 : 1); ++x)
            for (int h = 0; h < kH; ++h)
              tma_prefetch_3d(&tq, h * 64, G2.hk * g, G2.token0 + G2.i0 + x * (tr / g));
          break;
        }
      }
    }
    // before exit: every copy this warp started has landed (these waits
    // ignore the abort flag but keep the time bound)
    if (lane == 0) {
      volatile WaitCtl drain = {0, 0, kWaitLimitNs};
      if (q_armed) mbar_wait(BAR(B_QFULL), q_par, &drain);
      for (int which = 0; which < 2; ++which)
        for (int s = 0; s < (which ? kNV : kNK); ++s)
          if ((armed >> (4 * which + s)) & 1)
            mbar_wait(BAR((which ? B_VFULL : B_KFULL) + s), (apar >> (4 * which + s)) & 1, &drain);
      if (drain.abort) ctl->abort = 1;  // an expired drain wait is reported too
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Lane 0 runs the schedule, its waits and every tcgen05 operation. The
    // shared-memory descriptors are made once: a descriptor's start address
    // is its low 14 bits (address / 16), so the descriptor of an address plus
    // an offset is the base descriptor plus offset / 16 (shared addresses stay
    // below 256 KB). Building both descriptors per instruction cost about 130
    // cycles per 128 x 128 x 16 MMA, twice the tensor core's 64.
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16(BF16, false, 128, 128);
      constexpr uint32_t kIdO = idesc_f16(BF16, true, 128, D);
      const uint64_t dQ = sdesc_sw128(sbase + kOffQ, 16, 1024);
      const uint64_t dK = sdesc_sw128(sbase + kOffK, 16, 1024);
      const uint64_t dV = sdesc_sw128(sbase + kOffV, kBlk, 1024);
      constexpr uint64_t kTile16 = kTile >> 4;
      // S_x = Q_xq K^T into the S columns of warpgroup x (xq = x, or Q tile
      // A for both warpgroups of a split item)
      auto issue_s = [&](int x, int st, int xq) {
        const uint32_t d = tmem + uint32_t(x) * 128u;
        const uint64_t a0 = dQ + uint64_t(xq) * kTile16, b0 = dK + uint64_t(st) * kTile16;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {  // the head dim in steps of 16
          const uint64_t off = uint64_t((kk >> 2) * kBlk + (kk & 3) * 32) >> 4;
          tc_mma(d, a0 + off, b0 + off, kIdS, kk > 0 ? 1u : 0u);
        }
        tc_commit(BAR(B_SFULL + x));
      };
      auto issue_pv = [&](int x, int st, bool acc) {  // O_x += P_x V
        const uint32_t d = tmem + 256u + uint32_t(x) * 128u;
        const uint32_t a = tmem + uint32_t(x) * 128u;
        const uint64_t b0 = dV + uint64_t(st) * kTile16;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_ts(d, a + uint32_t(kk) * 8u, b0 + uint64_t(kk) * (2048 >> 4), kIdO,
                    (acc || kk > 0) ? 1u : 0u);
      };
      int gt = 0, qc = 0, cnt0 = 0, cnt1 = 0, itc0 = 0, itc1 = 0;
      bool ok = true;
      WorkItem nit{};
      nit.b = -1;
      if (int(blockIdx.x) < n_items) nit = load_item(items, blockIdx.x);
      for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
        const WorkItem it = nit;  // this item, loaded one item ahead
        if (w + int(gridDim.x) < n_items) nit = load_item(items, w + gridDim.x);
        if (it.b < 0) continue;  // schedule padding
        const ItemGeom G = item_geom(it, g, tile_rows, causal, wl, kv_box_rows);
        if (G.n_tiles == 0) continue;
        const bool hasB = G.n_rows > tr;
        const int n = G.n_tiles;
        if (!mbar_wait(BAR(B_QFULL), qc & 1, ctl)) { ok = false; break; }
        if (!hasB && n >= 2) {
          // split item: key tile j goes to warpgroup j & 1, both on Q tile A
          for (int j0 = 0; j0 < 2 && ok; ++j0) {
            const int g0 = gt + j0;
            if (!mbar_wait(BAR(B_KFULL + g0 % kNK), (g0 / kNK) & 1, ctl)) { ok = false; break; }
            tc_fence_after();
            issue_s(j0, g0 % kNK, 0);
            tc_commit(BAR(B_KEMPTY + g0 % kNK));
          }
          if (!ok) break;
          if (n == 2) tc_commit(BAR(B_QEMPTY));
          for (int j = 0; j < n && ok; ++j) {
            const int xw = j & 1, jx = j >> 1, g1 = gt + j, sv = g1 % kNV;
            const int itc_x = xw ? itc1 : itc0, cnt_x = xw ? cnt1 : cnt0;
            if (jx == 0 && itc_x > 0 &&
                !mbar_wait(BAR(B_OFREE + xw), (itc_x - 1) & 1, ctl)) { ok = false; break; }
            if (!mbar_wait(BAR(B_PFULL + xw), (cnt_x + jx) & 1, ctl)) { ok = false; break; }
            if (!mbar_wait(BAR(B_VFULL + sv), (g1 / kNV) & 1, ctl)) { ok = false; break; }
            tc_fence_after();
            issue_pv(xw, sv, jx > 0);
            if (j >= n - 2) tc_commit(BAR(B_ODONE + xw));  // the warpgroup's last tile
            tc_commit(BAR(B_VEMPTY + sv));
            if (j + 2 < n) {  // tile j + 2, on this warpgroup's S columns
              const int sk = (g1 + 2) % kNK;
              if (!mbar_wait(BAR(B_KFULL + sk), ((g1 + 2) / kNK) & 1, ctl)) { ok = false; break; }
              tc_fence_after();
              issue_s(xw, sk, 0);
              tc_commit(BAR(B_KEMPTY + sk));
              if (j + 2 == n - 1) tc_commit(BAR(B_QEMPTY));
            }
          }
          gt += n;
          ++qc;
          cnt0 += (n + 1) / 2;
          cnt1 += n / 2;
          ++itc0;
          ++itc1;
          continue;
        }
        if (!mbar_wait(BAR(B_KFULL + gt % kNK), (gt / kNK) & 1, ctl)) { ok = false; break; }
        tc_fence_after();
        issue_s(0, gt % kNK, 0);
        if (hasB) issue_s(1, gt % kNK, 1);
        tc_commit(BAR(B_KEMPTY + gt % kNK));
        if (n == 1) tc_commit(BAR(B_QEMPTY));
        for (int j = 0; j < n && ok; ++j) {
          const int g1 = gt + j, sv = g1 % kNV, st1 = (g1 + 1) % kNK;
          // ---- tile A
          if (j == 0 && itc0 > 0 && !mbar_wait(BAR(B_OFREE), (itc0 - 1) & 1, ctl)) { ok = false; break; }
          if (!mbar_wait(BAR(B_PFULL), (cnt0 + j) & 1, ctl)) { ok = false; break; }
          if (!mbar_wait(BAR(B_VFULL + sv), (g1 / kNV) & 1, ctl)) { ok = false; break; }
          tc_fence_after();
          issue_pv(0, sv, j > 0);
          if (j == n - 1) tc_commit(BAR(B_ODONE));
          if (!hasB) tc_commit(BAR(B_VEMPTY + sv));
          if (j + 1 < n) {
            if (!mbar_wait(BAR(B_KFULL + st1), ((g1 + 1) / kNK) & 1, ctl)) { ok = false; break; }
            tc_fence_after();
            issue_s(0, st1, 0);
            if (!hasB) {
              tc_commit(BAR(B_KEMPTY + st1));
              if (j + 1 == n - 1) tc_commit(BAR(B_QEMPTY));
            }
          }
          // ---- tile B
          if (hasB) {
            if (j == 0 && itc1 > 0 && !mbar_wait(BAR(B_OFREE + 1), (itc1 - 1) & 1, ctl)) { ok = false; break; }
            if (!mbar_wait(BAR(B_PFULL + 1), (cnt1 + j) & 1, ctl)) { ok = false; break; }
            tc_fence_after();
            issue_pv(1, sv, j > 0);
            tc_commit(BAR(B_VEMPTY + sv));
            if (j == n - 1) tc_commit(BAR(B_ODONE + 1));
            if (j + 1 < n) {
              issue_s(1, st1, 1);
              tc_commit(BAR(B_KEMPTY + st1));
              if (j + 1 == n - 1) tc_commit(BAR(B_QEMPTY));
            }
          }
        }
        gt += n;
        ++qc;
        cnt0 += n;
        ++itc0;
        if (hasB) {
          cnt1 += n;
          ++itc1;
        }
      }
      // every MMA this thread issued has completed before tensor memory is freed
      tc_commit(BAR(B_FINAL));
      volatile WaitCtl drain = {0, 0, kWaitLimitNs};
      if (!mbar_wait(BAR(B_FINAL), 0, &drain)) ctl->abort = 1;
    }
    __syncwarp();
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 200;" ::: "memory");
    // ------------------------------------------------------------ softmax + epilogue
    const int x = (warp - 4) >> 2;         // Q tile of this warpgroup
    const int sw = warp & 3;               // TMEM lane quadrant
    const int r = sw * 32 + lane;          // row within the Q tile
    const uint32_t lane_addr = uint32_t(sw * 32) << 16;
    const uint32_t tS = tmem + lane_addr + uint32_t(x) * 128u;
    const uint32_t tO = tmem + lane_addr + 256u + uint32_t(x) * 128u;
    const float scale = p.sm_scale_log2;
    // every wait here is warp-uniform, so a timeout never splits a warp in
    // front of a .sync.aligned instruction
    auto wwait = [&](uint32_t bar, uint32_t parity) {
      const bool okl = mbar_wait(bar, parity, ctl);
      return __all_sync(0xffffffffu, okl);
    };
    float* sml = reinterpret_cast<float*>(smem + kOffMl);  // [2][128]: B's row max, row sum
    // gt: key tiles of the CTA so far (stage and phase); cnt, itc: S tiles and
    // items of this warpgroup; itc_b: items of warpgroup B (its O phases);
    // nsplit: split items (the exchange phases)
    int gt = 0, cnt = 0, itc = 0, itc_b = 0, nsplit = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
      const WorkItem it = load_item(items, w);
      if (it.b < 0) continue;  // schedule padding
      const ItemGeom G = item_geom(it, g, tile_rows, causal, wl, kv_box_rows);
      const bool hasB = G.n_rows > tr;
      const int n = G.n_tiles;
      const bool split = !hasB && n >= 2;
      const int xr = split ? 0 : x;  // the Q tile whose rows this warpgroup runs
      const int nx = xr == 0 ? min(tr, G.n_rows) : max(0, G.n_rows - tr);  // rows of that tile
      const bool active = n > 0 && (x == 0 || hasB || split);
      const bool row_ok = r < nx;
      const int pr = G.row0 + xr * tr + r;
      const int qi = pr / g;
      const int tok = G.token0 + qi;
      const int head = G.hk * g + pr % g;
      const bool direct = G.chunk < 0;
      const int slot = direct ? 0 : G.partial_base + (qi - G.i0) * G.num_chunks + G.chunk;
      // custom (tree) mask: request b's bits start on byte mbase (-1: none)
      const int mbase = MASKED ? G.mask_base : -1;
      if (!active) {
        if (n == 0 && row_ok) {  // no live key: o = 0, lse = -inf
          if (direct) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(p.out) + (int64_t(tok) * Hq + head) * D);
            for (int q = 0; q < D / 8; ++q) dst[q] = make_uint4(0, 0, 0, 0);
            if (p.lse) p.lse[int64_t(tok) * Hq + head] = neg_inf();
          } else {
            float4* dst = reinterpret_cast<float4*>(tmp_o + (int64_t(slot) * Hq + head) * D);
            for (int q = 0; q < D / 4; ++q) dst[q] = make_float4(0.f, 0.f, 0.f, 0.f);
            tmp_lse[int64_t(slot) * Hq + head] = neg_inf();
          }
        }
        gt += n;
        continue;
      }
      // this row's live keys: [jmin, jmax]
      int jmin = G.kv_lo, jmax = G.kv_hi - 1;
      if (wl >= 0) jmin = max(jmin, G.lk - G.lq + qi - wl);
      if (causal) jmax = min(jmax, qi + G.lk - G.lq);
      const int ix0 = (G.row0 + xr * tr) / g;              // first / last query row of my tile
      const int ix1 = (G.row0 + xr * tr + nx) / g - 1;
      // key tiles of this warpgroup: all of them, or every other one (split)
      const int nt = split ? (n - x + 1) / 2 : n;
      float m_run = neg_inf(), l_run = 0.f;
      for (int jj = 0; jj < nt; ++jj) {
        const int j = split ? 2 * jj + x : jj;
        const int g1 = gt + j;
        const int t0 = G.t_start + j * 128;
        if (!wwait(BAR(B_SFULL + x), (cnt + jj) & 1)) { ok = false; break; }
        tc_fence_after();
        const bool need_mask = MASKED || (t0 < G.kv_lo) || (t0 + 128 > G.kv_hi) ||
                               (causal && t0 + 127 > ix0 + G.lk - G.lq) ||
                               (wl >= 0 && t0 < G.lk - G.lq + ix1 - wl);
        // The row's 128 scores end up in registers (sv). P = exp2(s * scale -
        // m) is packed in pairs over the first 64 S columns; the scaling and
        // the row sum run as packed fp32 pairs. (Computing a share of the
        // exponentials on the FMA pipe instead of the SFU measured slower.)
        uint32_t sv[4][32];
        const float2 sc2 = make_float2(scale, scale);
        float2 ps2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        auto mask_chunk = [&](auto cc) {
          constexpr int c = decltype(cc)::value;
          // the keys of this chunk the row keeps, as a bit mask: those in
          // [jmin, jmax], ANDed with the custom mask's bits (bit qi * Lk +
          // key of the request's segment; bits past it read as 0, and keys
          // past Lk are outside jmax anyway). A warp whose rows keep the whole
          // chunk skips the per-element pass.
          const int base = t0 + c * 32;
          const int lo = max(jmin - base, 0), hi = min(jmax - base, 31);
          uint32_t keep = lo > hi ? 0u : ((0xFFFFFFFFu >> (31 - (hi - lo))) << lo);
          if constexpr (MASKED)
            keep &= custom_mask_word(p.custom_mask + mbase, int64_t(G.lq) * G.lk,
                                     int64_t(qi) * G.lk + base);
          if (__all_sync(0xffffffffu, keep == 0xFFFFFFFFu)) return;
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (!(keep & (1u << e))) sv[c][e] = __float_as_uint(neg_inf());
        };
        auto exp_chunk = [&](auto cc, float2 nmu2) {
          constexpr int c = decltype(cc)::value;
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 xx = __ffma2_rn(
                make_float2(__uint_as_float(sv[c][2 * e]), __uint_as_float(sv[c][2 * e + 1])), sc2,
                nmu2);
            const float2 pp = make_float2(ex2(xx.x), ex2(xx.y));
            ps2[e & 1] = __fadd2_rn(ps2[e & 1], pp);
            pk[e] = DT::pack(pp.x, pp.y);
          }
          tmem_st16(tS + uint32_t(c) * 16u, pk);
        };
        using C0 = std::integral_constant<int, 0>;
        using C1 = std::integral_constant<int, 1>;
        using C2 = std::integral_constant<int, 2>;
        using C3 = std::integral_constant<int, 3>;
        // Warm rows (a finite running max) take their exponentials against
        // the running max straight away, with no max pass over the tile, and
        // the second half of the row is still loading while the first half is
        // exponentiated. If the tile's sum stays at most 2^8, no p exceeds
        // 2^8, the bound the lazy rescale keeps, and the tile is done. Else
        // (and for a warp with a cold row: the first tile, or a row whose keys
        // have all been masked so far) the row max is taken and the tile
        // follows the lazy rule: a new reference when the max exceeds the old
        // by more than 2^8, O rescaled, P recomputed. Every choice is
        // warp-uniform (the tensor-memory accesses are .sync.aligned).
        const bool cold = __any_sync(0xffffffffu, m_run == neg_inf());
        bool redo = cold;
        if (!cold) {
          tmem_ld32(tS, sv[0]);
          tmem_ld32(tS + 32u, sv[1]);
          tmem_wait_ld_tied(sv[0]);
          tmem_wait_ld_tied(sv[1]);
          tmem_ld32(tS + 64u, sv[2]);
          tmem_ld32(tS + 96u, sv[3]);
          const float2 nm2 = make_float2(-m_run, -m_run);
          if (need_mask) {
            mask_chunk(C0());
            mask_chunk(C1());
          }
          exp_chunk(C0(), nm2);
          exp_chunk(C1(), nm2);
          tmem_wait_ld_tied(sv[2]);
          tmem_wait_ld_tied(sv[3]);
          if (need_mask) {
            mask_chunk(C2());
            mask_chunk(C3());
          }
          exp_chunk(C2(), nm2);
          exp_chunk(C3(), nm2);
          const float tsum = (ps2[0].x + ps2[1].x) + (ps2[0].y + ps2[1].y);
          redo = __any_sync(0xffffffffu, tsum > 256.f);
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(tS + uint32_t(c) * 32u, sv[c]);
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_wait_ld_tied(sv[c]);
          if (need_mask) {
            mask_chunk(C0());
            mask_chunk(C1());
            mask_chunk(C2());
            mask_chunk(C3());
          }
        }
        float m_new = m_run, corr = 1.f;
        if (redo) {
          // row max of the raw scores: eight independent chains of
          // three-input maxima
          float mp[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) mp[q] = neg_inf();
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 16; ++e)
              mp[e & 7] = fmax3(mp[e & 7], __uint_as_float(sv[c][2 * e]),
                                __uint_as_float(sv[c][2 * e + 1]));
          const float mraw = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                                   fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
          const float mx = mraw * scale;  // scale > 0
          if (mx > m_run + 8.f || (m_run == neg_inf() && mraw != neg_inf())) m_new = mx;
          corr = (m_new == m_run) ? 1.f : ex2(m_run - m_new);
          // a warm warp whose rows all keep their reference keeps its P
          if (cold || __any_sync(0xffffffffu, m_new != m_run)) {
            // O rescale: S_x(j) is complete, so the P V product before it is too
            if (jj > 0 && __any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll 1
              for (int c = 0; c < D / 32; ++c) {
                uint32_t ov[32];
                tmem_ld32(tO + uint32_t(c) * 32u, ov);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * corr);
                tmem_st32(tO + uint32_t(c) * 32u, ov);
              }
            }
            const float mu = (m_new == neg_inf()) ? 0.f : m_new;
            const float2 nmu2 = make_float2(-mu, -mu);
            ps2[0] = ps2[1] = make_float2(0.f, 0.f);
            exp_chunk(C0(), nmu2);
            exp_chunk(C1(), nmu2);
            exp_chunk(C2(), nmu2);
            exp_chunk(C3(), nmu2);
          }
        }
        bool zeroed = false;
        if ((x == 0 || split) && t0 + 128 > G.lk) {  // the tile's first (or only) reader
          // rows of V past the request's last key may hold anything: zero them
          if (!wwait(BAR(B_VFULL + g1 % kNV), (g1 / kNV) & 1)) { ok = false; break; }
          if (t0 + r >= G.lk) {
#pragma unroll
            for (int h = 0; h < kH; ++h) {
              uint4* row = reinterpret_cast<uint4*>(smem + kOffV + (g1 % kNV) * kTile + h * kBlk +
                                                    r * 128);
#pragma unroll
              for (int q = 0; q < 8; ++q) row[q] = make_uint4(0, 0, 0, 0);
            }
          }
          zeroed = true;
        }
        tmem_wait_st();
        l_run = l_run * corr + ((ps2[0].x + ps2[1].x) + (ps2[0].y + ps2[1].y));
        m_run = m_new;
        if (zeroed) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        mbar_arrive(BAR(B_PFULL + x));
      }
      if (!ok) break;
      if (split && x == 1) {
        // hand this warpgroup's row state to A, which reads O_B from tensor
        // memory and releases it
        if (nsplit > 0 && !wwait(BAR(B_MLFREE), (nsplit - 1) & 1)) { ok = false; break; }
        sml[r] = m_run;
        sml[128 + r] = l_run;
        mbar_arrive(BAR(B_MLFULL));
        gt += n;
        cnt += nt;
        ++itc;
        ++nsplit;
        continue;
      }
      // epilogue; for a split item, combine with B's state first:
      //   m = max(m_A, m_B), O = O_A 2^(m_A - m) + O_B 2^(m_B - m), same for l
      float fa = 1.f, fb = 0.f;
      if (split) {
        if (!wwait(BAR(B_MLFULL), nsplit & 1)) { ok = false; break; }
        const float mb = sml[r], lb = sml[128 + r];
        mbar_arrive(BAR(B_MLFREE));
        const float m = fmaxf(m_run, mb);
        fa = m_run == neg_inf() ? 0.f : ex2(m_run - m);
        fb = mb == neg_inf() ? 0.f : ex2(mb - m);
        l_run = l_run * fa + lb * fb;
        m_run = m;
      }
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const float lse = l_run > 0.f ? (m_run + __log2f(l_run)) * kLn2 : neg_inf();
      fa *= inv;
      fb *= inv;
      if (!wwait(BAR(B_ODONE + x), itc & 1)) { ok = false; break; }
      if (split && !wwait(BAR(B_ODONE + 1), itc_b & 1)) { ok = false; break; }
      tc_fence_after();
      const uint32_t tOb = tmem + lane_addr + 384u;  // O of warpgroup B
      // The rows leave through this warp's staging buffer: a thread writes
      // its row's 128-byte blocks there (16-byte pieces in XOR-swizzled
      // order, so neither side has bank conflicts), then each store
      // instruction sends four rows' blocks, 8 lanes per block. A thread
      // storing its own row wrote 16-byte pieces of 32 rows per instruction.
      uint8_t* stg = smem + kOffStage + (warp - 4) * 4096;
      char* my_dst = nullptr;  // this thread's output row (none past the tile)
      if (row_ok)
        my_dst = direct ? reinterpret_cast<char*>(static_cast<T*>(p.out) + (int64_t(tok) * Hq + head) * D)
                        : reinterpret_cast<char*>(tmp_o + (int64_t(slot) * Hq + head) * D);
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(tO + uint32_t(c) * 32u, ov);
        tmem_wait_ld();
        if (split) {
          uint32_t ob[32];
          tmem_ld32(tOb + uint32_t(c) * 32u, ob);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e)
            ov[e] = __float_as_uint(__uint_as_float(ov[e]) * fa + __uint_as_float(ob[e]) * fb);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * fa);
        }
        // this chunk's 16-byte pieces q of the row's 128-byte block: the
        // 16-bit output packs two chunks per block, fp32 partials one
        if (direct) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int q = (c & 1) * 4 + i;
            *reinterpret_cast<uint4*>(stg + lane * 128 + ((q ^ (lane & 7)) << 4)) = make_uint4(
                DT::pack(__uint_as_float(ov[8 * i + 0]), __uint_as_float(ov[8 * i + 1])),
                DT::pack(__uint_as_float(ov[8 * i + 2]), __uint_as_float(ov[8 * i + 3])),
                DT::pack(__uint_as_float(ov[8 * i + 4]), __uint_as_float(ov[8 * i + 5])),
                DT::pack(__uint_as_float(ov[8 * i + 6]), __uint_as_float(ov[8 * i + 7])));
          }
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<uint4*>(stg + lane * 128 + ((q ^ (lane & 7)) << 4)) =
                make_uint4(ov[4 * q], ov[4 * q + 1], ov[4 * q + 2], ov[4 * q + 3]);
        }
        if (!direct || (c & 1)) {
          __syncwarp();
          const int blk = direct ? (c >> 1) : c;  // the 128-byte block of each row
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int row = k * 4 + (lane >> 3), q = lane & 7;
            char* dst = reinterpret_cast<char*>(
                __shfl_sync(0xffffffffu, reinterpret_cast<long long>(my_dst), row));
            const uint4 v = *reinterpret_cast<const uint4*>(stg + row * 128 + ((q ^ (row & 7)) << 4));
            if (dst) *reinterpret_cast<uint4*>(dst + blk * 128 + q * 16) = v;
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      mbar_arrive(BAR(B_OFREE + x));
      if (split) mbar_arrive(BAR(B_OFREE + 1));  // O_B is read too
      if (row_ok) {
        if (direct) {
          if (p.lse) p.lse[int64_t(tok) * Hq + head] = lse;
        } else {
          tmp_lse[int64_t(slot) * Hq + head] = lse;
        }
      }
      gt += n;
      cnt += nt;
      ++itc;
      if (hasB || split) ++itc_b;
      if (split) ++nsplit;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0 && ctl->abort) {
    int* err = const_cast<int*>(&hdr->err_flag);
    atomicExch(err, 1);
  }
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

}  // namespace

namespace {
int gcd_i(int a, int b) {
  while (b) {
    const int t = a % b;
    a = b;
    b = t;
  }
  return a;
}

template <bool BF16, int D, bool MASKED>
cudaError_t launch_tc_m(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv, int box_rows, int grid, cudaStream_t s) {
  // the shared-memory limit: once per device, before any capture
  static std::atomic<uint64_t> done{0};
  constexpr int kSmem = TcLayout<D>::kSmem;
  auto k = prefill_tc_kernel<BF16, D, MASKED>;
  const cudaError_t attr = smem_attr_once(k, kSmem, done);
  if (attr != cudaSuccess) return attr;
  k<<<grid, kTcThreads, kSmem, s>>>(p, tq, tk, tv, box_rows);
  return cudaGetLastError();
}

template <bool BF16, int D>
cudaError_t launch_tc(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                      const CUtensorMap& tv, int box_rows, int grid, cudaStream_t s) {
  return p.custom_mask ? launch_tc_m<BF16, D, true>(p, tq, tk, tv, box_rows, grid, s)
                       : launch_tc_m<BF16, D, false>(p, tq, tk, tv, box_rows, grid, s);
}
}  // namespace

// head_dim 64 or 128; K/V boxes of gcd(page_size, 128) slots must be whole
// 8-row swizzle atoms, so the page size is a multiple of 8 (any multiple:
// a box never crosses a page because its size divides the page size).
bool prefill_tc_supports(int head_dim, int page_size, int group) {
  if ((head_dim != 128 && head_dim != 64) || group < 1 || group > 128) return false;
  return page_size >= 8 && page_size % 8 == 0;
}

cudaError_t launch_prefill_tc(const AttnParams& p, int head_dim, int group, int tile_rows,
                              int64_t q_rows, int64_t num_pages, bool bf16, int grid,
                              cudaStream_t s) {
  if (grid <= 0) return cudaSuccess;
  if (!prefill_tc_supports(head_dim, p.page_size, group)) return cudaErrorInvalidValue;
  CUtensorMap tq, tk, tv;
  const int box_rows = gcd_i(p.page_size, 128);
  {
    cuuint64_t dims[3] = {cuuint64_t(head_dim), cuuint64_t(p.num_qo_heads), cuuint64_t(q_rows)};
    cuuint64_t str[2] = {cuuint64_t(p.q_stride_head) * 2, cuuint64_t(p.q_stride_tok) * 2};
    cuuint32_t box[3] = {64, cuuint32_t(group), cuuint32_t(tile_rows / 2 / group)};
    if (!encode_tensor_map(&tq, bf16, 3, p.q, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  if (!encode_kv_map(&tk, p, true, bf16, head_dim, num_pages, 64, box_rows,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_kv_map(&tv, p, false, bf16, head_dim, num_pages, 64, box_rows,
                     CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (head_dim == 128)
    return bf16 ? launch_tc<true, 128>(p, tq, tk, tv, box_rows, grid, s)
                : launch_tc<false, 128>(p, tq, tk, tv, box_rows, grid, s);
  return bf16 ? launch_tc<true, 64>(p, tq, tk, tv, box_rows, grid, s)
              : launch_tc<false, 64>(p, tq, tk, tv, box_rows, grid, s);
}

}  // namespace fi
