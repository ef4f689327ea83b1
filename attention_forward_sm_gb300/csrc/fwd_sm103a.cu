// Attention forward (prefill) for sm_103a: tiled, IO-aware, online softmax,
// per-row log-sum-exp, causal mask and grouped KV heads.  The causal mask can
// sit at a global row offset (p.q_offset: row i of the launch is row
// q_offset + i of the sequence), for a rank's block of a sequence-parallel
// prefill.
//
// Method.  FlashAttention computes softmax(scale * Q K^T) V tile by tile
// without writing the N x N score matrix to HBM ("FlashAttention-3 vs Triton
// Kernels", introduction).  Each query row keeps a running max m and running
// sum l; when m grows the accumulated output is rescaled ("correction"
// partition in "Warp Specialization in Triton: Design and Roadmap", "How the
// compiler does it").  The kernel is warp-specialised: loads, MMAs and the
// softmax (with the correction and the epilogue) run in different warps and
// talk through mbarrier producer/consumer pipes, so loads, tensor-core work
// and exponentials overlap (same note, and the pipeline diagram and
// "Hardware Mechanics" of the FlashAttention-3 page, which describe the
// Hopper version of the idea).
//
// GB300 design (not the Hopper layout of the pages):
//   * one CTA = 2 query tiles of 128 rows of one (batch, head); the two tiles
//     are independent MMA chains (the autoWS note's "data partitioning"), so
//     the tensor core works on one tile while the softmax of the other runs;
//   * tcgen05.mma (kind::f16, M=128) issued from one warp, one elected
//     thread per instruction; S = Q K^T and O accumulate in tensor memory
//     (TMEM), not registers: S0, S1, O0, O1 occupy 128 + 128 + D + D of the
//     512 TMEM columns.  At D = 64 and for e4m3 the next key tile's
//     Q K^T is issued in two halves, the upper one while the softmax still
//     works on the current S;
//   * P (bf16) is written back over S in TMEM and fed to the P*V MMA as the
//     A operand straight from TMEM;
//   * a TMA load warp streams K and V tiles (128 keys x D, 128-byte swizzle)
//     through a STAGES-deep shared-memory ring;
//   * sixteen softmax warps, eight per query tile: two warps share each
//     32-lane TMEM quarter (16 rows each) and the two half-warps split a row's
//     128 scores, so a thread handles 64 columns; row max (one shuffle),
//     exp2, row sum in fp32, P packed to bf16 into TMEM.  The same warps
//     rescale O in TMEM, only when some row's max rose by more than 2^8
//     (otherwise the stale max stays: exact, because the final division uses
//     the same max), and run the epilogue (O / l -> bf16 -> global, and LSE);
//   * setmaxnreg moves registers from the load/MMA warps to the softmax warps;
//   * a running CTA takes over CTAs that have not started yet (cluster
//     launch control) and works through their units in turn, its TMEM,
//     barriers and K/V ring carrying over, so the next unit's loads and first
//     Q K^T overlap the current unit's tail.
#include <cuda_bf16.h>
#include <math_constants.h>

#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kBM = 128;          // query rows per tile
constexpr int kBN = 128;          // keys per K/V tile
constexpr int kThreads = 640;     // 20 warps: 16 softmax/epilogue + load, MMA, 2 idle
constexpr int kWarpLoad = 16;
constexpr int kWarpMma = 17;
constexpr int kClcReaders = 18;   // loader, MMA issuer, 16 softmax warps
// setmaxnreg split of the 61440 registers the launch gets (640 threads x 96):
// 4 softmax warpgroups + 1 warpgroup for load / MMA / idle warps.
constexpr uint32_t kRegSoftmax = 112, kRegOther = 32;
static_assert(4 * 128 * kRegSoftmax + 128 * kRegOther <= 640 * 96, "register split");

template <int D, bool kFp8 = false>
struct Cfg {
  static constexpr int kElemBytes = kFp8 ? 1 : 2;
  static constexpr int kTileBytes = kBM * D * kElemBytes;  // a 128 x D tile (Q, K; V or V^T)
  static constexpr int kAtomElems = 128 / kElemBytes;      // elements per 128-byte swizzle row
  static constexpr int kChunks = D * kElemBytes / 128;     // 128-byte swizzle chunks per tile row
  static constexpr int kStages = (D == 128) ? 4 : 8;       // K/V ring depth
  static constexpr int kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 256 + D;
  // Q K^T in two N = 64 halves, keys [64, 128) issued while the softmax
  // still works on the previous S (see the MMA warp).  With Q in shared
  // memory each half re-reads all of Q, so the halves cost 3/4 of a full
  // MMA's time each; that pays where the tensor pipe has slack (e4m3, and
  // D = 64, whose Q moreover sits in TMEM) and not at D = 128 bf16, where
  // the pipe is already busy ~3/4 of the time.
  static constexpr bool kSplitS = (D == 64) || kFp8;
  // D = 64 (bf16) has TMEM columns to spare: Q_t is copied there once per
  // unit (kColQ0, kColQ1: D / 2 columns each) and every Q K^T reads A from
  // TMEM, so an N = 64 half reads only its 2 KB of K from shared memory per
  // k-step instead of 6 KB; Q's shared-memory buffers are free once copied.
  static constexpr bool kQInTmem = (D == 64) && !kFp8;
  static constexpr int kColQ0 = 2 * 128 + 2 * D, kColQ1 = kColQ0 + D / 2;
  static constexpr int kTmemCols = 512;
  static_assert(!kQInTmem || kColQ1 + D / 2 <= kTmemCols, "TMEM columns");
  // P = 2^(s - m + kPBias) and the running max moves when it rises by more
  // than kRescale (log2 units).  bf16 P has fp32's range: any bias works, a
  // wide threshold saves O rescales.  E4M3 P saturates at 448 < 2^9, so
  // p <= 2^(kPBias + kRescale) must stay <= 2^8; the bias lifts small
  // weights out of the subnormal range (normal E4M3 starts at 2^-6).
  static constexpr float kPBias = kFp8 ? 6.f : 0.f;
  static constexpr float kRescale = kFp8 ? 2.f : 8.f;
  // dynamic shared memory map (offsets from a 1024-byte aligned base): the
  // two Q tiles, the K/V ring (barriers are static shared memory)
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = 2 * kTileBytes;
  static constexpr int kSmemBytes = kOffKV + kStages * kTileBytes + 1024;  // + alignment slack
  static_assert(!kFp8 || D == kBN, "the FP8 V^T tile is D x 128 keys: D must be 128");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

struct Misc {
  uint64_t q_full;        // the unit's Q tiles arrived (one phase per unit)
  uint64_t q_empty;       // the unit's Q tiles were read (its last Q K^T, or with Q in
                          // TMEM the copies, retired): Q buffers reusable
  uint64_t s_full[2];     // S_t = Q_t K^T in TMEM (MMA commit)
  uint64_t s_read[2];     // S_t loaded by the tile's softmax warps (one arrival per warp)
  uint64_t p_full[2];     // P_t in TMEM (one arrival per softmax warp of the tile)
  uint64_t o_done[2];     // every MMA of the unit's O_t retired (one phase per unit)
  uint64_t mma_done;
  uint64_t kv_full[8], kv_empty[8];
  uint64_t clc_full[2];   // next-unit response k in slot k % 2 arrived
  uint64_t clc_empty[2];  // every role has read response k (kClcReaders arrivals)
  uint4 clc_resp[2];      // cluster-launch-control responses
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xFFFFFFFFu, v); }

// Optional event trace (compile with -DATTN_TRACE): clock64 stamps of the
// pipeline events of the first CTAs, for latency analysis.  Off by default.
#ifdef ATTN_TRACE
constexpr int kTraceCtas = 16;
__device__ unsigned long long g_attn_trace[kTraceCtas * 1024];
#define ATTN_TRACE_EV(E, t, j)                                                     \
  do {                                                                            \
    if (blockIdx.x < kTraceCtas && (j) < 64)                                      \
      g_attn_trace[blockIdx.x * 1024 + ((E) * 2 + (t)) * 64 + (j)] = clock64();   \
  } while (0)
#else
#define ATTN_TRACE_EV(E, t, j) \
  do {                         \
  } while (0)
#endif

// Wait used only while tearing down after an abort: ignores the abort flag and
// gives up after a bounded number of polls (each poll suspends briefly), so
// copies and MMAs already in flight retire before the CTA exits.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  for (int spin = 0; spin < (1 << 20); ++spin)
    if (mbar_try_wait(bar, parity)) return;
}

// S = Q K^T over the head dimension into TMEM columns kColD, one MMA per 32
// bytes of a row (16 bf16 or 32 e4m3 columns); inside a 128-byte swizzle
// chunk a k-step advances the start address by 32 bytes, the next chunk
// starts 128 rows * 128 bytes further.  kOffB moves the K operand by whole
// rows: kKeyHalf selects keys [64, 128) of the tile (64 rows * 128 bytes,
// eight 1024-byte swizzle atoms).
constexpr uint32_t kKeyHalf = (64 * 128) >> 4;
// kColQ = 0: A (Q) from shared memory; otherwise A from TMEM columns
// kColQ.. (Q copied there once per unit, 8 columns per k-step).
template <bool kFp8, uint32_t kColD, uint32_t kOffA, uint32_t kColQ, uint32_t kOffB,
          uint32_t kIdesc, int KK, int NK>
__device__ __forceinline__ void issue_s_rec(uint32_t tmem, uint32_t a0, uint32_t b0) {
  if constexpr (KK < NK) {
    constexpr uint32_t off = ((KK >> 2) * (kBM * 128) + (KK & 3) * 32) >> 4;
    if constexpr (kColQ != 0)
      mma_ts<kFp8, kColD, kColQ + KK * 8, off + kOffB, kIdesc>(tmem, b0, KK > 0 ? 1u : 0u);
    else
      mma_ss<kFp8, kColD, off + kOffA, off + kOffB, kIdesc>(tmem, a0, b0, KK > 0 ? 1u : 0u);
    issue_s_rec<kFp8, kColD, kOffA, kColQ, kOffB, kIdesc, KK + 1, NK>(tmem, a0, b0);
  }
}
// N = 128 (all keys of the tile) or, with kHalf = 1 or 2, N = 64 over keys
// [0, 64) or [64, 128) into the same columns of S as the full product.  The
// A (Q) descriptor is a0 + kOffA (a constant, modulo 2^32, from the K ring's
// descriptor, so that no second descriptor register stays live), or, with
// kColQ != 0, Q is read from TMEM columns kColQ..
template <int D, bool kFp8, uint32_t kColS, uint32_t kOffA, int kHalf = 0, uint32_t kColQ = 0>
__device__ __forceinline__ void issue_s_steps(uint32_t tmem, uint32_t a0, uint32_t b0) {
  constexpr uint32_t kN = kHalf ? kBN / 2 : kBN;
  constexpr uint32_t kIdesc = kFp8 ? idesc_e4m3_f32(128, kN) : idesc_bf16_f32(128, kN, false);
  constexpr uint32_t kColD = kColS + (kHalf == 2 ? kBN / 2 : 0);
  constexpr uint32_t kOffB = kHalf == 2 ? kKeyHalf : 0;
  issue_s_rec<kFp8, kColD, kOffA, kColQ, kOffB, kIdesc, 0, D * (kFp8 ? 1 : 2) / 32>(tmem, a0,
                                                                                   b0);
}
// O (TMEM columns kColD) += P (TMEM columns kColP) V over the 128 keys of a
// tile, one MMA per 8 TMEM columns of P (16 bf16 or 32 e4m3 keys).  bf16: V
// is MN-major, a step advances 16 rows * 128 bytes.  e4m3: V^T (D rows of
// 128 keys) is K-major, a step advances 32 bytes inside the 128-byte row.
template <bool kFp8, uint32_t kColD, uint32_t kColP, uint32_t kOffB, uint32_t kIdesc, int KK>
__device__ __forceinline__ void issue_pv_rec(uint32_t tmem, uint32_t b0, uint32_t acc) {
  constexpr int kSteps = kFp8 ? kBN / 32 : kBN / 16;
  if constexpr (KK < kSteps) {
    constexpr uint32_t off = kFp8 ? ((KK * 32) >> 4) : ((KK * 16 * 128) >> 4);
    mma_ts<kFp8, kColD, kColP + KK * 8, off + kOffB, kIdesc>(tmem, b0, KK > 0 ? 1u : acc);
    issue_pv_rec<kFp8, kColD, kColP, kOffB, kIdesc, KK + 1>(tmem, b0, acc);
  }
}
template <int D, bool kFp8, uint32_t kColD, uint32_t kColP, uint32_t kOffB>
__device__ __forceinline__ void issue_pv_steps(uint32_t tmem, uint32_t b0, uint32_t acc) {
  constexpr uint32_t kIdesc = kFp8 ? idesc_e4m3_f32(128, D) : idesc_bf16_f32(128, D, true);
  issue_pv_rec<kFp8, kColD, kColP, kOffB, kIdesc, 0>(tmem, b0, acc);
}

// Work unit u: (batch*head, pair of 128-row query tiles).  Non-causal:
// head-major.  Causal: heads in groups of p.group_heads (sized on the host
// so a group's K/V stays in L2); inside a group all units longest first, so
// the CTAs, which take units in order, end every group, and the grid, on
// short units.
struct Unit {
  int bh, q_base, n_kv;
};
__device__ __forceinline__ Unit decode_unit(const FwdParams& p, int u, int nqb) {
  int qblk, bh;
  if (p.causal) {
    const int BH = p.B * p.Hq;
    const int per_group = p.group_heads * nqb;
    const int g = u / per_group;
    const int idx = u % per_group;
    const int heads = min(p.group_heads, BH - g * p.group_heads);
    qblk = nqb - 1 - idx / heads;
    bh = g * p.group_heads + idx % heads;
  } else {
    qblk = u % nqb;
    bh = u / nqb;
  }
  Unit w;
  w.bh = bh;
  w.q_base = qblk * 2 * kBM;
  w.n_kv = (p.Nk + kBN - 1) / kBN;
  if (p.causal) w.n_kv = min(w.n_kv, (w.q_base + p.q_offset + 2 * kBM + kBN - 1) / kBN);
  return w;
}
__device__ __forceinline__ int kv_head(const FwdParams& p, int bh) {
  return (bh / p.Hq) * p.Hkv + (bh % p.Hq) / (p.Hq / p.Hkv);
}

// The grid has one CTA per unit, in unit order, but a running CTA takes over
// CTAs that have not started yet (cluster launch control) and does their
// units itself, in the order the hardware would have started them: the
// loader asks for the next unit once it has issued the current unit's
// loads, and every role reads the answer (response k in slot k % 2) when it
// finishes unit k.  TMEM, barriers and the K/V ring live across units: every
// barrier phase and the ring position run on, so the next unit's K/V and Q
// loads and its first Q K^T overlap the current unit's last steps and
// epilogue.
template <int D, bool kFp8>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = Cfg<D, kFp8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  // barriers in static shared memory: their addresses are constants, which
  // keeps them out of the registers of the 32-register warps
  __shared__ Misc ms;
  const uint32_t abort_flag = smem_u32(&ms.abort_flag);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // (recomputed where used rather than kept live into the roles)
#define ATTN_NQB ((p.Nq + 2 * kBM - 1) / (2 * kBM))
#define ATTN_UNITS (ATTN_NQB * p.B * p.Hq)

  // ---- setup: barriers (loader warp), TMEM (MMA warp)
  if (warp == kWarpLoad && lane == 0) {
    mbar_init(&ms.q_full, 1);
    mbar_init(&ms.q_empty, 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&ms.s_full[t], 1);
      mbar_init(&ms.s_read[t], 8);
      mbar_init(&ms.p_full[t], 8);
      mbar_init(&ms.o_done[t], 1);
    }
    mbar_init(&ms.mma_done, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ms.clc_full[i], 1);
      mbar_init(&ms.clc_empty[i], kClcReaders);
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&ms.kv_full[s], 1);
      mbar_init(&ms.kv_empty[s], 1);
    }
    ms.abort_flag = 0;
    fence_mbar_init();
    // The first unit's Q tiles and first K tile start loading now, before the
    // CTA-wide barrier and the TMEM allocation: they are the first MMA's
    // operands.
    const Unit w = decode_unit(p, static_cast<int>(blockIdx.x), ATTN_NQB);
    mbar_arrive_expect_tx(&ms.q_full, 2 * C::kTileBytes);
    for (int t = 0; t < 2; ++t)
      for (int ch = 0; ch < C::kChunks; ++ch)
        tma_load_3d(smem + C::kOffQ + t * C::kTileBytes + ch * (kBM * 128), &p.tmap_q,
                    &ms.q_full, ch * C::kAtomElems, w.q_base + t * kBM, w.bh,
                    l2_policy_evict_first());
    mbar_arrive_expect_tx(&ms.kv_full[0], C::kTileBytes);
    for (int ch = 0; ch < C::kChunks; ++ch)
      tma_load_3d(smem + C::kOffKV + ch * (kBM * 128), &p.tmap_k, &ms.kv_full[0],
                  ch * C::kAtomElems, 0, kv_head(p, w.bh), l2_policy_evict_last());
    tma_prefetch_desc(&p.tmap_v);
  }
  if (warp == kWarpMma) {
    tmem_alloc(&ms.tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;

  if (warp < 16) {
    // =====================================================================
    // softmax + epilogue: warps 8t .. 8t + 7 serve query tile t.  Two warps
    // share each 32-lane TMEM quarter (16 rows each), and the two threads
    // t and t + 16 of a warp share one row: thread half c holds key columns
    // [64c, 64c + 64) of the row.  Per SMSP that puts two warps of a tile on
    // the exponentials at once, and the row max needs one shuffle.
    // =====================================================================
    reg_alloc<kRegSoftmax>();
    const int t = warp >> 3;
    const int lbase = (warp & 3) * 32 + ((warp >> 2) & 1) * 16;  // first TMEM lane of the warp
    const int r = lbase + (lane & 15);                              // row within the tile
    const int c = lane >> 4;                                        // column half of the row
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(lbase) << 16);
    const uint32_t s_addr = lane_addr + (t ? C::kColS1 : C::kColS0);
    const uint32_t o_addr = lane_addr + (t ? C::kColO1 : C::kColO0);
    const bool tracer = (warp & 7) == 0 && lane == 0;
    uint32_t step = 0;  // key tiles of this CTA's earlier units: barrier phases run on
    bool ok = true;
    for (int u = static_cast<int>(blockIdx.x), k = 0; u >= 0 && ok; ++k) {
      const Unit w = decode_unit(p, u, ATTN_NQB);
      const int tile_row0 = w.q_base + t * kBM;
      const int row = tile_row0 + r;
      const int vis = p.causal ? min(row + 1 + p.q_offset, p.Nk) : p.Nk;  // keys [0, vis)
      float m = -CUDART_INF_F, l = 0.f;  // l: sum over this thread's half of the row
      for (int j = 0; j < w.n_kv; ++j) {
        if (!warp_all(mbar_wait(&ms.s_full[t], (step + j) & 1, abort_flag, p.err,
                                kErrWaitSoftmax, p.wait_limit_ns))) {
          ok = false;
          break;
        }
        if (tracer && k == 0) ATTN_TRACE_EV(0, t, j);
        tc_fence_after();
        float s[64];
        {
          uint32_t sr[64];
          tmem_ld_pair64<64>(s_addr, sr);
#pragma unroll
          for (int i = 0; i < 64; ++i) s[i] = __uint_as_float(sr[i]);
        }
        if (tracer && k == 0) ATTN_TRACE_EV(1, t, j);
        const int kb = j * kBN + c * 64;  // key index of this thread's first column
        const bool need_mask =
            (j * kBN + kBN > p.Nk) || (p.causal && j * kBN + kBN - 1 > tile_row0 + p.q_offset);
        if (need_mask) {
          const int lim_c = vis - kb;  // columns [0, lim_c) valid
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (i >= lim_c) s[i] = -CUDART_INF_F;
        }
        float mx;
        {
          float a0 = fmaxf(s[0], s[1]), a1 = fmaxf(s[2], s[3]);
          float a2 = fmaxf(s[4], s[5]), a3 = fmaxf(s[6], s[7]);
#pragma unroll
          for (int i = 8; i < 64; i += 8) {
            a0 = max3f(a0, s[i], s[i + 1]);
            a1 = max3f(a1, s[i + 2], s[i + 3]);
            a2 = max3f(a2, s[i + 4], s[i + 5]);
            a3 = max3f(a3, s[i + 6], s[i + 7]);
          }
          mx = max3f(a0, a1, fmaxf(a2, a3));
          mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 16));  // the row's other half
        }
        if constexpr (C::kSplitS) {
          // S_t has been read (and used): the MMA warp may now write the next
          // key tile's keys [64, 128) over columns 64..127 of S_t, which P
          // does not use
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ms.s_read[t]);
        }
        // running max in log2 units (scale >= 0, so max commutes with scaling)
        const float m_tile = (mx == -CUDART_INF_F) ? -CUDART_INF_F : mx * p.scale_log2;
        float alpha = 1.f;
        if (m_tile > m + C::kRescale || m == -CUDART_INF_F) {
          alpha = ex2_approx(m - m_tile);  // 0 on the first tile
          m = m_tile;
        }
        if (tracer && k == 0) ATTN_TRACE_EV(2, t, j);
        // p = 2^(s*scale*log2e - m + bias), masked entries exactly 0; packed
        // to bf16 pairs (32 words) or e4m3 quads (16 words), low key first
        const float neg_m = C::kPBias - m;
        float rsum;
        uint32_t pk[kFp8 ? 16 : 32];
        auto pack4 = [&](int i, float p0, float p1, float p2, float p3) {
          if constexpr (kFp8) {
            pk[i / 4] = pack_e4m3x4(p0, p1, p2, p3);
          } else {
            pk[i / 2] = pack_bf16x2(p0, p1);
            pk[i / 2 + 1] = pack_bf16x2(p2, p3);
          }
        };
        if (need_mask) {
          float r0 = 0.f, r1 = 0.f;
#pragma unroll
          for (int i = 0; i < 64; i += 4) {
            float pp[4];
#pragma unroll
            for (int v = 0; v < 4; ++v)
              pp[v] = (s[i + v] == -CUDART_INF_F)
                          ? 0.f
                          : ex2_approx(fmaf(s[i + v], p.scale_log2, neg_m));
            r0 += pp[0] + pp[2];
            r1 += pp[1] + pp[3];
            pack4(i, pp[0], pp[1], pp[2], pp[3]);
          }
          rsum = r0 + r1;
        } else {
          // packed fp32x2: one FMA and one add per pair of columns
          const uint64_t scale2 = f32x2(p.scale_log2, p.scale_log2);
          const uint64_t negm2 = f32x2(neg_m, neg_m);
          uint64_t acc0 = f32x2(0.f, 0.f), acc1 = acc0;
#pragma unroll
          for (int i = 0; i < 64; i += 4) {
            float x0, x1, x2, x3;
            unpack_f32x2(fma_f32x2(f32x2(s[i], s[i + 1]), scale2, negm2), x0, x1);
            unpack_f32x2(fma_f32x2(f32x2(s[i + 2], s[i + 3]), scale2, negm2), x2, x3);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
            acc0 = add_f32x2(acc0, f32x2(p0, p1));
            acc1 = add_f32x2(acc1, f32x2(p2, p3));
            pack4(i, p0, p1, p2, p3);
          }
          float u0f, u1f;
          unpack_f32x2(add_f32x2(acc0, acc1), u0f, u1f);
          rsum = u0f + u1f;
        }
        l = fmaf(l, alpha, rsum);
        if (tracer && k == 0) ATTN_TRACE_EV(3, t, j);
        // Rescale O_t when a row's max rose past the threshold.  Every P*V of
        // KV tiles < j has retired: it was issued before S_t(j), whose
        // completion woke this warp.  The P*V of tile j waits for p_full below.
        // Thread half c owns O columns [c*D/2, (c+1)*D/2) of its row.
        if (j > 0 && __any_sync(0xFFFFFFFFu, alpha != 1.f)) {
          // 16 columns at a time: P (pk) stays live across this rare path
#pragma unroll 1
          for (int kk = 0; kk < D / 32; ++kk) {
            uint32_t v[16];
            tmem_ld_pair16<D / 2>(o_addr + kk * 16, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            tmem_st_pair16<D / 2>(o_addr + kk * 16, v);
          }
          tmem_st_wait();
        }
        // P over the first 64 (bf16) or 32 (e4m3) columns of S: this half's
        // 32 or 16 columns
        if constexpr (kFp8)
          tmem_st_pair16<16>(s_addr, pk);
        else
          tmem_st_pair32<32>(s_addr, pk);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ms.p_full[t]);
        if (tracer && k == 0) ATTN_TRACE_EV(4, t, j);
      }
      step += w.n_kv;
      // ---- epilogue of tile t: O / l -> bf16 -> global (a thread writes the
      // D/2 columns it owns of its row; evict-first in L2, since nothing here
      // reads O again and the K/V tiles being reused should keep the space),
      // and LSE.  The TMEM reads of O_t
      // complete here, before these warps publish the next unit's first P of
      // this tile, which the MMA that overwrites O_t waits for.
      ok = ok && warp_all(mbar_wait(&ms.o_done[t], k & 1, abort_flag, p.err, kErrWaitCorr, p.wait_limit_ns));
      if (!ok) break;
      tc_fence_after();
      const float l_row = l + __shfl_xor_sync(0xFFFFFFFFu, l, 16);
      const float inv = p.o_scale / l_row;
      uint4* orow = reinterpret_cast<uint4*>(
          static_cast<__nv_bfloat16*>(p.o) +
          (static_cast<size_t>(w.bh) * p.Nq + static_cast<size_t>(row)) * D + c * (D / 2));
#pragma unroll
      for (int kk = 0; kk < D / 64; ++kk) {
        // columns c*D/2 + [32kk, 32kk + 32) of the row
        uint32_t v[32];
        tmem_ld_pair32<D / 2>(o_addr + kk * 32, v);
        uint32_t wv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          wv[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * inv,
                              __uint_as_float(v[2 * i + 1]) * inv);
        if (row < p.Nq) {
#pragma unroll
          for (int g = 0; g < 4; ++g)
            st_global_v4_evict_first(orow + kk * 4 + g, wv[4 * g], wv[4 * g + 1], wv[4 * g + 2],
                                     wv[4 * g + 3]);
        }
      }
      if (c == 0 && row < p.Nq)
        p.lse[static_cast<size_t>(w.bh) * p.Nq + row] =
            (m - C::kPBias + __log2f(l_row)) * 0.69314718055994530942f;
      // the next unit: response k
      if (!warp_all(mbar_wait(&ms.clc_full[k & 1], (k >> 1) & 1, abort_flag, p.err,
                              kErrWaitCorr, p.wait_limit_ns))) {
        ok = false;
        break;
      }
      const int nu = clc_response_ctaid_x(smem_u32(&ms.clc_resp[k & 1]));
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ms.clc_empty[k & 1]);
      u = nu < ATTN_UNITS ? nu : -1;
    }
  } else if (warp == kWarpLoad) {
    // =====================================================================
    // TMA loader: per unit the Q tiles (once the previous unit's last Q K^T
    // has read them), then K_j, V_j through the ring.  Ring item numbers run
    // on across units: a unit's step j loads items 2(step + j), +1.  The
    // whole warp runs the loop (waits are warp-wide votes, so control flow
    // stays uniform); one elected thread issues each copy, arrival and
    // next-unit request.
    // =====================================================================
    reg_dealloc<kRegOther>();
    {
      uint32_t item = 0;    // ring items of earlier units
      uint32_t g = 1;       // next ring item (the first unit's K_0 was issued during setup)
      uint32_t q_phase = 0;  // q_full phase of the last Q load issued
      bool ok = true;
      int clc_k = -1;        // last next-unit request issued
      int u = static_cast<int>(blockIdx.x);
      for (int k = 0; ok; ++k) {
        const Unit w = decode_unit(p, u, ATTN_NQB);
        const int bhkv = kv_head(p, w.bh);
        const uint32_t item_end = item + 2u * static_cast<uint32_t>(w.n_kv);
        for (; g < item_end; ++g) {
          const uint32_t it = g - item;  // item within the unit: K_{it/2} or V_{it/2}
          const uint32_t s = g % C::kStages;
          if (!warp_all(mbar_wait(&ms.kv_empty[s], ((g / C::kStages) & 1u) ^ 1u, abort_flag,
                                  p.err, kErrWaitLoad, p.wait_limit_ns))) {
            ok = false;
            break;
          }
          if (lane == 0 && k == 0) ATTN_TRACE_EV(7, it & 1, it >> 1);
          mbar_arrive_expect_tx_elect(&ms.kv_full[s], C::kTileBytes);
          uint8_t* dst = smem + C::kOffKV + s * C::kTileBytes;
          const int jt = static_cast<int>(it >> 1);
          if (kFp8 && (it & 1)) {
            // V^T [D rows, keys]: rows 0..D-1, keys of tile jt
            tma_load_3d_elect(dst, &p.tmap_v, &ms.kv_full[s], jt * kBN, 0, bhkv,
                              l2_policy_evict_last());
          } else {
            const CUtensorMap* map = (it & 1) ? &p.tmap_v : &p.tmap_k;
            for (int ch = 0; ch < C::kChunks; ++ch)
              tma_load_3d_elect(dst + ch * (kBM * 128), map, &ms.kv_full[s], ch * C::kAtomElems,
                                jt * kBN, bhkv, l2_policy_evict_last());
          }
          if (it == 0 && k > 0) {
            // the Q tiles of this unit, once the previous unit's last Q K^T
            // retired (its K_0 is already on the way)
            if (!warp_all(mbar_wait(&ms.q_empty, (k - 1) & 1, abort_flag, p.err, kErrWaitLoad,
                                    p.wait_limit_ns))) {
              ok = false;
              ++g;
              break;
            }
            const Unit wq = decode_unit(p, u, ATTN_NQB);
            q_phase = k & 1;
            mbar_arrive_expect_tx_elect(&ms.q_full, 2 * C::kTileBytes);
            for (int t = 0; t < 2; ++t)
              for (int ch = 0; ch < C::kChunks; ++ch)
                tma_load_3d_elect(smem + C::kOffQ + t * C::kTileBytes + ch * (kBM * 128),
                                  &p.tmap_q, &ms.q_full, ch * C::kAtomElems,
                                  wq.q_base + t * kBM, wq.bh, l2_policy_evict_first());
          }
        }
        item = item_end;
        if (!ok) break;
        // every load of unit k is issued: ask for the next unit (slot k % 2,
        // free once every role has read response k - 2)
        if (k >= 2 && !warp_all(mbar_wait(&ms.clc_empty[k & 1], ((k >> 1) + 1) & 1, abort_flag,
                                          p.err, kErrWaitLoad, p.wait_limit_ns))) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx_elect(&ms.clc_full[k & 1], 16);
        clc_try_cancel_elect(smem_u32(&ms.clc_resp[k & 1]), &ms.clc_full[k & 1]);
        clc_k = k;
        if (!warp_all(mbar_wait(&ms.clc_full[k & 1], (k >> 1) & 1, abort_flag, p.err,
                                kErrWaitLoad, p.wait_limit_ns))) {
          ok = false;
          break;
        }
        const int nu = clc_response_ctaid_x(smem_u32(&ms.clc_resp[k & 1]));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ms.clc_empty[k & 1]);
        if (nu < 0 || nu >= ATTN_UNITS) break;
        u = nu;
      }
      if (abort_set(abort_flag)) {
        // drain: wait (bounded) for the copies still in flight before exiting:
        // the last Q load and the ring items issued last (items < g)
        drain_wait(&ms.q_full, q_phase);
        if (clc_k >= 0) drain_wait(&ms.clc_full[clc_k & 1], (clc_k >> 1) & 1);
        for (uint32_t it = g > C::kStages ? g - C::kStages : 0u; it < g; ++it)
          drain_wait(&ms.kv_full[it % C::kStages], (it / C::kStages) & 1u);
      }
    }
  } else if (warp == kWarpMma) {
    // =====================================================================
    // MMA issuer: S_t = Q_t K_j^T, O_t += P_t V_j.  The whole warp runs this
    // loop (waits are warp-wide votes, so control flow stays uniform); one
    // elected thread issues each MMA and commit.
    // =====================================================================
    reg_dealloc<kRegOther>();
    {
      constexpr uint32_t kTileDesc = C::kTileBytes >> 4;  // one tile in descriptor units
      // Descriptors are built once; every k-step only adds a constant to the
      // start-address field, so issuing an MMA costs a couple of instructions.
      // Q and V differ from K by compile-time constants (start address; V:
      // bf16 MN-major with 64-column chunks kBM * 128 bytes apart, e4m3 V^T
      // K-major), so one descriptor stays live.
      const uint32_t desc_k = sdesc_sw128_lo(smem_u32(smem + C::kOffKV), 16);
      constexpr uint32_t kQFromK = static_cast<uint32_t>((C::kOffKV - C::kOffQ) >> 4);
      constexpr uint32_t kVFromK = kFp8 ? 0u : static_cast<uint32_t>(((kBM * 128) >> 4) - 1) << 16;
      constexpr uint32_t kS = C::kStages;  // power of two
      static_assert((kS & (kS - 1)) == 0, "ring depth must be a power of two");
      // Q_t's descriptor relative to the K ring's (a constant modulo 2^32)
      constexpr uint32_t kQ0 = 0u - kQFromK, kQ1 = kQ0 + kTileDesc;
      // S_t = Q_t K^T from the K tile in ring slot `slot`
      constexpr uint32_t kTQ0 = C::kQInTmem ? C::kColQ0 : 0, kTQ1 = C::kQInTmem ? C::kColQ1 : 0;
      auto issue_s = [&](int t, uint32_t slot) {
        const uint32_t b0 = desc_k + slot * kTileDesc;
        if (t)
          issue_s_steps<D, kFp8, C::kColS1, kQ1, 0, kTQ1>(tmem, desc_k, b0);
        else
          issue_s_steps<D, kFp8, C::kColS0, kQ0, 0, kTQ0>(tmem, desc_k, b0);
      };
      // keys [64h, 64h + 64) of S_t = Q_t K^T into columns [64h, 64h + 64) of
      // S_t.  Half 1 goes in as soon as the softmax warps have read S_t of the
      // previous key tile (P_t takes columns below 64 only), half 0 after the
      // P_t V that reads P_t from those columns: the tile's wait for its next
      // S holds only the P V and half the Q K^T.
      auto issue_s_half = [&](int t, uint32_t slot, int h) {
        const uint32_t b0 = desc_k + slot * kTileDesc;
        if (t) {
          if (h)
            issue_s_steps<D, kFp8, C::kColS1, kQ1, 2, kTQ1>(tmem, desc_k, b0);
          else
            issue_s_steps<D, kFp8, C::kColS1, kQ1, 1, kTQ1>(tmem, desc_k, b0);
        } else {
          if (h)
            issue_s_steps<D, kFp8, C::kColS0, kQ0, 2, kTQ0>(tmem, desc_k, b0);
          else
            issue_s_steps<D, kFp8, C::kColS0, kQ0, 1, kTQ0>(tmem, desc_k, b0);
        }
      };
      // O_t (+)= P_t V from the V tile in ring slot `slot`; P_t is in TMEM over S_t
      auto issue_pv = [&](int t, uint32_t slot, uint32_t acc) {
        const uint32_t b0 = desc_k + slot * kTileDesc;
        if (t)
          issue_pv_steps<D, kFp8, C::kColO1, C::kColS1, kVFromK>(tmem, b0, acc);
        else
          issue_pv_steps<D, kFp8, C::kColO0, C::kColS0, kVFromK>(tmem, b0, acc);
      };
      int k = 0;  // units done
      // wait for P_t of global step gs (O_t is already rescaled when it arrives)
      auto wait_p = [&](int t, uint32_t gs, int jv) -> bool {
        if (!warp_all(mbar_wait(&ms.p_full[t], gs & 1u, abort_flag, p.err, kErrWaitMma,
                                p.wait_limit_ns)))
          return false;
        if (lane == 0 && k == 0) ATTN_TRACE_EV(5, t, jv);
        tc_fence_after();
        return true;
      };
      // wait until the softmax warps of tile t have read S_t of global step gs
      auto wait_s_read = [&](int t, uint32_t gs) -> bool {
        if (!warp_all(mbar_wait(&ms.s_read[t], gs & 1u, abort_flag, p.err, kErrWaitMma,
                                p.wait_limit_ns)))
          return false;
        tc_fence_after();
        return true;
      };
      uint32_t step = 0;  // key tiles of earlier units: ring items 2*step.., barrier phases
      bool ok = true;
      int u = static_cast<int>(blockIdx.x);
      for (; ok; ++k) {
        const uint32_t step_end = step + static_cast<uint32_t>(decode_unit(p, u, ATTN_NQB).n_kv);
        ok = warp_all(mbar_wait(&ms.q_full, k & 1, abort_flag, p.err, kErrWaitMma, p.wait_limit_ns));
        if constexpr (C::kQInTmem) {
          // Q_0, Q_1 into TMEM (one 128 x 16 slice per copy; D = 64 is one
          // 128-byte swizzle row, a slice advances 32 bytes).  The copies
          // run in the tensor pipe ahead of this unit's Q K^T; they overwrite
          // the previous unit's Q only once every MMA of that unit retired
          // (its last P V, committed to o_done[1] after all its Q K^T), and
          // Q's shared memory is free once they retire.
          if (ok && k > 0)
            ok = warp_all(mbar_wait(&ms.o_done[1], (k - 1) & 1, abort_flag, p.err, kErrWaitMma,
                                    p.wait_limit_ns));
          if (ok) {
            tc_fence_after();
            static_assert(D == 64, "one swizzle chunk per row");
            const uint32_t q0 = desc_k + kQ0, q1 = desc_k + kQ1;
            tmem_cp_128x256b<C::kColQ0 + 0, 0>(tmem, q0);
            tmem_cp_128x256b<C::kColQ0 + 8, 2>(tmem, q0);
            tmem_cp_128x256b<C::kColQ0 + 16, 4>(tmem, q0);
            tmem_cp_128x256b<C::kColQ0 + 24, 6>(tmem, q0);
            tmem_cp_128x256b<C::kColQ1 + 0, 0>(tmem, q1);
            tmem_cp_128x256b<C::kColQ1 + 8, 2>(tmem, q1);
            tmem_cp_128x256b<C::kColQ1 + 16, 4>(tmem, q1);
            tmem_cp_128x256b<C::kColQ1 + 24, 6>(tmem, q1);
            mma_commit(&ms.q_empty);
          }
        }
        // global step gs = step + j: K_j is ring item 2 gs, V_j item 2 gs + 1
        for (uint32_t gs = step; gs < step_end && ok; ++gs) {
          const uint32_t sk = (2u * gs) % kS, sv = (2u * gs - 1u) % kS;
          ok = warp_all(mbar_wait(&ms.kv_full[sk], ((2u * gs) / kS) & 1u, abort_flag, p.err,
                                  kErrWaitMma, p.wait_limit_ns));
          if (ok && gs > step)
            ok = warp_all(mbar_wait(&ms.kv_full[sv], ((2u * gs - 1u) / kS) & 1u, abort_flag, p.err,
                                    kErrWaitMma, p.wait_limit_ns));
          if (!ok) break;
          tc_fence_after();
          for (int t = 0; t < 2 && ok; ++t) {
            if (gs > step && C::kSplitS) {
              ok = wait_s_read(t, gs - 1);
              if (!ok) break;
              issue_s_half(t, sk, 1);
              ok = wait_p(t, gs - 1, static_cast<int>(gs - step) - 1);
              if (!ok) break;
              // the accumulate flag as a constant in each branch keeps this
              // path within the MMA warp's 32 registers (no spill at D = 64)
              if (gs > step + 1)
                issue_pv(t, sv, 1u);
              else
                issue_pv(t, sv, 0u);
              issue_s_half(t, sk, 0);
            } else {
              if (gs > step) {
                ok = wait_p(t, gs - 1, static_cast<int>(gs - step) - 1);
                if (!ok) break;
                issue_pv(t, sv, gs > step + 1 ? 1u : 0u);
              }
              issue_s(t, sk);
            }
            mma_commit(&ms.s_full[t]);
            if (lane == 0 && k == 0) ATTN_TRACE_EV(6, t, gs - step);
          }
          if (!ok) break;
          mma_commit(&ms.kv_empty[sk]);
          if (gs > step) mma_commit(&ms.kv_empty[sv]);
        }
        // the unit's last Q K^T is issued: Q's buffers are free once it retires
        if (ok && !C::kQInTmem) mma_commit(&ms.q_empty);
        if (ok) {
          const uint32_t gs = step_end - 1;
          const uint32_t sv = (2u * gs + 1u) % kS;
          ok = warp_all(mbar_wait(&ms.kv_full[sv], ((2u * gs + 1u) / kS) & 1u, abort_flag, p.err,
                                  kErrWaitMma, p.wait_limit_ns));
          if (ok) {
            tc_fence_after();
            for (int t = 0; t < 2 && ok; ++t) {
              ok = (!C::kSplitS || wait_s_read(t, gs)) && wait_p(t, gs, static_cast<int>(gs - step));
              if (ok) {
                issue_pv(t, sv, gs > step ? 1u : 0u);
                mma_commit(&ms.o_done[t]);
              }
            }
            if (ok) mma_commit(&ms.kv_empty[sv]);
          }
        }
        step = step_end;
        if (!ok) break;
        // the next unit: response k
        ok = warp_all(mbar_wait(&ms.clc_full[k & 1], (k >> 1) & 1, abort_flag, p.err, kErrWaitMma,
                                p.wait_limit_ns));
        if (!ok) break;
        const int nu = clc_response_ctaid_x(smem_u32(&ms.clc_resp[k & 1]));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ms.clc_empty[k & 1]);
        if (nu < 0 || nu >= ATTN_UNITS) break;
        u = nu;
      }
      // all issued MMAs retire before the CTA releases TMEM
      mma_commit(&ms.mma_done);
      drain_wait(&ms.mma_done, 0);
    }
  } else {
    reg_dealloc<kRegOther>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
#undef ATTN_NQB
#undef ATTN_UNITS
}

// Causal unit order: query heads per group, whole KV-head groups, so that
// the group's K and V (read by every unit of its heads) take at most about
// a third of the 129 MB L2.
int causal_group_heads(const FwdParams& p) {
  const int G = p.Hq / p.Hkv;
  const double kv_bytes = 2.0 * p.Nk * p.D * (p.fp8 ? 1 : 2);  // K and V of one KV head
  int kv_heads = static_cast<int>(40.0e6 / kv_bytes);
  kv_heads = max(1, min(kv_heads, p.B * p.Hkv));
  return kv_heads * G;
}

template <int D, bool kFp8>
cudaError_t launch_d(const FwdParams& p_in, cudaStream_t stream) {
  FwdParams p = p_in;
  p.group_heads = causal_group_heads(p);
  using C = Cfg<D, kFp8>;
  // the shared-memory opt-in is a per-device property of the function
  static std::atomic<bool> attr_done[64];  // zero-initialised: false
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(attn_fwd_kernel<D, kFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done[dev].store(true, std::memory_order_release);
  }
  // one CTA per unit; running CTAs take over the ones not started yet
  const long long nqb = (p.Nq + 2 * kBM - 1) / (2 * kBM);
  const long long grid = nqb * p.B * p.Hq;
  attn_fwd_kernel<D, kFp8><<<static_cast<unsigned>(grid), kThreads, C::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

size_t fwd_smem_bytes(int D, bool fp8) {
  if (fp8) return Cfg<128, true>::kSmemBytes;
  return D == 128 ? Cfg<128>::kSmemBytes : Cfg<64>::kSmemBytes;
}

cudaError_t launch_fwd(const FwdParams& p, cudaStream_t stream) {
  if (p.fp8) return p.D == 128 ? launch_d<128, true>(p, stream) : cudaErrorInvalidValue;
  if (p.D == 128) return launch_d<128, false>(p, stream);
  if (p.D == 64) return launch_d<64, false>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn

#ifdef ATTN_TRACE
// Trace builds only: copies the event stamps of the last traced launch to
// host memory (n words at most); returns the number copied or -1.
extern "C" int attn_trace_copy(unsigned long long* host, int n) {
  n = n < attn::kTraceCtas * 1024 ? n : attn::kTraceCtas * 1024;
  return cudaMemcpyFromSymbol(host, attn::g_attn_trace, n * sizeof(unsigned long long)) ==
                 cudaSuccess
             ? n
             : -1;
}
#endif
