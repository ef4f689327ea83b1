// Inline-PTX building blocks for sm_103a: mbarrier pipes, TMA tile loads,
// tcgen05 (tensor-core MMA with TMEM accumulators) and TMEM load/store.
//
// Everything here is a thin wrapper over one PTX instruction (or a fixed
// group of them); the warp-specialised kernels are composed from these.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace attn {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity.  Returns true when the
// phase completed.  Gives up (returns false) when the abort flag (an int in
// shared memory at shared-window address `abort_sa`) is already set by
// another role, or after `limit_ns` of wall time, in which case it sets the
// flag, ORs `site` into the device error word `err` and returns false.
// Every role that sees false leaves its loop, so the CTA drains and exits
// instead of hanging.
__device__ __forceinline__ bool abort_set(uint32_t abort_sa) {
  int v;
  asm volatile("ld.volatile.shared.b32 %0, [%1];" : "=r"(v) : "r"(abort_sa) : "memory");
  return v != 0;
}
__device__ __forceinline__ void abort_raise(uint32_t abort_sa) {
  asm volatile("st.volatile.shared.b32 [%0], %1;" ::"r"(abort_sa), "r"(1) : "memory");
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t abort_sa,
                                          unsigned int* err, uint32_t site, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0u) {
      if (abort_set(abort_sa)) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        abort_raise(abort_sa);
        atomicOr(err, site);
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------- TMA (tensor tile copies)
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// 3-D tiled load global -> shared, completion counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// The same, executed by a whole converged warp with warp-uniform operands;
// elect.sync picks the one thread that issues the copy (as for the MMAs
// below: cheaper for the warp than a single-thread branch).
__device__ __forceinline__ void tma_load_3d_elect(void* dst, const CUtensorMap* map,
                                                  uint64_t* bar, int c0, int c1, int c2,
                                                  uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;\n\t}" ::"r"(smem_u32(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// mbar_arrive_expect_tx by one elected thread of a converged warp.
__device__ __forceinline__ void mbar_arrive_expect_tx_elect(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

// Generic-proxy shared-memory accesses ordered before later async-proxy ones.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- cluster launch control
// Asks the hardware to cancel a CTA of this grid that has not started yet
// and to hand its work to the calling CTA: the 16-byte response lands at
// shared address `resp` and completes 16 transaction bytes on `bar`.
__device__ __forceinline__ void clc_try_cancel(uint32_t resp, uint64_t* bar) {
  asm volatile(
      "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 "
      "[%0], [%1];" ::"r"(resp),
      "r"(smem_u32(bar))
      : "memory");
}
// clc_try_cancel by one elected thread of a converged warp.
__device__ __forceinline__ void clc_try_cancel_elect(uint32_t resp, uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 "
      "[%0], [%1];\n\t}" ::"r"(resp),
      "r"(smem_u32(bar))
      : "memory");
}
// Reads a response: the x block index of the CTA taken over, or -1 when the
// request found no CTA left to take.
__device__ __forceinline__ int clc_response_ctaid_x(uint32_t resp) {
  uint32_t ok, x = 0;
  asm volatile(
      "{\n\t.reg .b128 r;\n\t.reg .pred p;\n\t"
      "ld.shared.b128 r, [%2];\n\t"
      "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t"
      "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, r;\n\t}"
      : "=r"(ok), "+r"(x)
      : "r"(resp)
      : "memory");
  return ok ? static_cast<int>(x) : -1;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// 16-byte global store marked evict-first in L2.
__device__ __forceinline__ void st_global_v4_evict_first(void* addr, uint32_t a, uint32_t b,
                                                         uint32_t c, uint32_t d) {
  asm volatile(
      "{\n\t.reg .b64 pol;\n\t"
      "createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
      "st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, pol;\n\t}" ::"l"(addr),
      "r"(a), "r"(b), "r"(c), "r"(d)
      : "memory");
}

// ---------------------------------------------------------------- register reallocation
template <uint32_t N>
__device__ __forceinline__ void reg_alloc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void reg_dealloc() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ---------------------------------------------------------------- tcgen05: TMEM allocation
// Executed by one full warp.  Writes the TMEM base address to *dst (shared).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05: descriptors
// Instruction descriptor, kind::f16: bf16 x bf16 -> fp32, dense.
//   [4,6) D format (1 = f32), [7,10) A format (1 = bf16), [10,13) B format,
//   bit 15 A major (0 = K-major), bit 16 B major (1 = MN-major),
//   [17,23) N >> 3, [24,29) M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Instruction descriptor, kind::f8f6f4: e4m3 x e4m3 -> fp32, dense, both
// operands K-major: [4,6) D format (1 = f32), A and B formats 0 (= E4M3).
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(uint32_t M, uint32_t N) {
  return (1u << 4) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand.
//   [0,14) start >> 4, [16,30) leading byte offset >> 4, [32,46) stride byte
//   offset >> 4, [46,49) = 0b001, [49,52) base offset (0: tiles are 1024-B
//   aligned), [61,64) swizzle mode (2 = 128B).
// K-major: rows of 128 B, 8-row groups `sbo` apart (lbo unused).
// MN-major: 64-element MN chunks `lbo` apart, 8-row K groups `sbo` apart.
// Every descriptor of these kernels has sbo = 1024, so the upper word
// (kSdescHi) is the same for all; only the lower word (start address,
// leading byte offset) varies, and the MMA wrappers take that 32-bit word and
// rebuild the descriptor inside the instruction group.
constexpr uint64_t kSdescHi = (static_cast<uint64_t>(1024 >> 4) << 32) |
                              (static_cast<uint64_t>(1) << 46) | (static_cast<uint64_t>(2) << 61);
__device__ __forceinline__ uint32_t sdesc_sw128_lo(uint32_t saddr, uint32_t lbo) {
  return ((saddr & 0x3FFFFu) >> 4) | (((lbo >> 4) & 0x3FFFu) << 16);
}

// D[tmem] (+)= A[smem desc] * B[smem desc] (mma_ss) or A[tmem] * B[smem
// desc] (mma_ts), kind::f16 (bf16 operands) or kind::f8f6f4 (e4m3).  Every
// per-instruction offset and the instruction descriptor are compile-time
// constants, the offsets added inside the instruction group -- TMEM columns of D (and of A for mma_ts) to the TMEM
// base, 16-byte descriptor units to the descriptors' start addresses -- so
// an unrolled sequence of MMAs keeps only the TMEM base and one descriptor
// word live.  The whole (converged) warp executes these wrappers with
// warp-uniform operands, and elect.sync picks the one thread that issues:
// issued that way an MMA costs the warp far fewer cycles than from a
// single-thread branch (one thread's issue of an N = 64 MMA took about as
// long as an N = 128 one), and the issue rate holds up next to busy warps
// on the same SMSP.  elect.sync elects the same thread every time for the
// same member mask (the full warp here), so mma_commit, elected the same
// way, is issued by the thread that issued the MMAs it tracks.
#define ATTN_MMA_SS(KIND)                                                                    \
  asm volatile(                                                                             \
      "{\n\t.reg .pred p, e;\n\t.reg .b32 dt, al, bl;\n\t.reg .b64 da, db;\n\t"        \
      "elect.sync _|e, 0xffffffff;\n\t"                                                   \
      "add.u32 dt, %0, %5;\n\t"                                                           \
      "add.u32 al, %1, %6;\n\t"                                                           \
      "add.u32 bl, %2, %7;\n\t"                                                           \
      "cvt.u64.u32 da, al;\n\t"                                                           \
      "cvt.u64.u32 db, bl;\n\t"                                                           \
      "or.b64 da, da, %8;\n\t"                                                            \
      "or.b64 db, db, %8;\n\t"                                                            \
      "setp.ne.b32 p, %4, 0;\n\t"                                                         \
      "@e tcgen05.mma.cta_group::1." KIND " [dt], da, db, %3, p;\n\t}" ::"r"(tmem),         \
      "r"(a_lo), "r"(b_lo), "n"(kIdesc), "r"(accumulate), "n"(kColD), "n"(kOffA), "n"(kOffB), \
      "n"(kSdescHi)                                                                         \
      : "memory")
#define ATTN_MMA_TS(KIND)                                                                    \
  asm volatile(                                                                             \
      "{\n\t.reg .pred p, e;\n\t.reg .b32 dt, at, bl;\n\t.reg .b64 db;\n\t"            \
      "elect.sync _|e, 0xffffffff;\n\t"                                                   \
      "add.u32 dt, %0, %4;\n\t"                                                           \
      "add.u32 at, %0, %5;\n\t"                                                           \
      "add.u32 bl, %1, %6;\n\t"                                                           \
      "cvt.u64.u32 db, bl;\n\t"                                                           \
      "or.b64 db, db, %7;\n\t"                                                            \
      "setp.ne.b32 p, %3, 0;\n\t"                                                         \
      "@e tcgen05.mma.cta_group::1." KIND " [dt], [at], db, %2, p;\n\t}" ::"r"(tmem),       \
      "r"(b_lo), "n"(kIdesc), "r"(accumulate), "n"(kColD), "n"(kColA), "n"(kOffB),          \
      "n"(kSdescHi)                                                                         \
      : "memory")
// D at TMEM column kColD, A and B descriptors (lower words) + kOffA, kOffB,
// instruction descriptor kIdesc
template <bool kF8, uint32_t kColD, uint32_t kOffA, uint32_t kOffB, uint32_t kIdesc>
__device__ __forceinline__ void mma_ss(uint32_t tmem, uint32_t a_lo, uint32_t b_lo,
                                       uint32_t accumulate) {
  if constexpr (kF8)
    ATTN_MMA_SS("kind::f8f6f4");
  else
    ATTN_MMA_SS("kind::f16");
}
// D at TMEM column kColD, A at TMEM column kColA, B descriptor (lower word) + kOffB,
// instruction descriptor kIdesc
template <bool kF8, uint32_t kColD, uint32_t kColA, uint32_t kOffB, uint32_t kIdesc>
__device__ __forceinline__ void mma_ts(uint32_t tmem, uint32_t b_lo, uint32_t accumulate) {
  if constexpr (kF8)
    ATTN_MMA_TS("kind::f8f6f4");
  else
    ATTN_MMA_TS("kind::f16");
}
#undef ATTN_MMA_SS
#undef ATTN_MMA_TS

// Copy a 128-row x 256-bit slice of a shared-memory matrix (descriptor lower
// word d_lo + kOff; upper word kSdescHi) into TMEM lanes 0..127, columns
// kCol..kCol+7 of the base: row r lands in lane r, its 16 bf16 in column
// order, two per column, the lower element in the low half -- the layout
// an A operand in TMEM has.  Warp-wide, one elected thread issues; runs in
// the tensor pipe in issue order with the MMAs of the same thread.
template <uint32_t kCol, uint32_t kOff>
__device__ __forceinline__ void tmem_cp_128x256b(uint32_t tmem, uint32_t d_lo) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 dt, dl;\n\t.reg .b64 d;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "add.u32 dt, %0, %2;\n\t"
      "add.u32 dl, %1, %3;\n\t"
      "cvt.u64.u32 d, dl;\n\t"
      "or.b64 d, d, %4;\n\t"
      "@e tcgen05.cp.cta_group::1.128x256b [dt], d;\n\t}" ::"r"(tmem),
      "r"(d_lo), "n"(kCol), "n"(kOff), "n"(kSdescHi)
      : "memory");
}

// Arrive on `bar` once every tcgen05 op issued so far by the issuing thread
// completed.  Executed by the whole converged warp, like the MMA wrappers;
// elect.sync over the full warp picks the thread that issued them.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------- tcgen05: TMEM <-> registers
// 16 lanes x 32 bits, two halves: thread t of the warp gets lane
// (lane_base + t % 16) and columns [col + (t / 16) * kHalf, + 32 or 64).  The
// two threads t and t + 16 share one TMEM lane (one row) and split its columns.
#define ATTN_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
    "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
template <uint32_t kHalf>
__device__ __forceinline__ void tmem_ld_pair64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, "
      "%45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, "
      "%62, %63}, [%64], %65;\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : ATTN_R8(0), ATTN_R8(8), ATTN_R8(16), ATTN_R8(24), ATTN_R8(32), ATTN_R8(40), ATTN_R8(48),
        ATTN_R8(56)
      : "r"(taddr), "n"(kHalf)
      : "memory");
}
template <uint32_t kHalf>
__device__ __forceinline__ void tmem_ld_pair32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32], %33;\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : ATTN_R8(0), ATTN_R8(8), ATTN_R8(16), ATTN_R8(24)
      : "r"(taddr), "n"(kHalf)
      : "memory");
}
template <uint32_t kHalf>
__device__ __forceinline__ void tmem_ld_pair16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16], %17;\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : ATTN_R8(0), ATTN_R8(8)
      : "r"(taddr), "n"(kHalf)
      : "memory");
}
#undef ATTN_R8
#define ATTN_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), \
    "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])
template <uint32_t kHalf>
__device__ __forceinline__ void tmem_st_pair32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x32bx2.x32.b32 [%0], %33, {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
      "%10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, "
      "%27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      ATTN_W8(0), ATTN_W8(8), ATTN_W8(16), ATTN_W8(24), "n"(kHalf)
      : "memory");
}
#undef ATTN_W8

template <uint32_t kHalf>
__device__ __forceinline__ void tmem_st_pair16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x32bx2.x16.b32 [%0], %17, {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
      "%10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "n"(kHalf)
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- small math
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Three-input max (sm_100+).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Packed fp32 pairs (sm_100+ f32x2 arithmetic): lo in the low half.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Four floats -> four e4m3 codes (round to nearest even, saturating to the
// largest finite value), p0 in the lowest byte.
__device__ __forceinline__ uint32_t pack_e4m3x4(float p0, float p1, float p2, float p3) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(p0), "f"(p1), "f"(p2), "f"(p3));
  return r;
}

}  // namespace attn
