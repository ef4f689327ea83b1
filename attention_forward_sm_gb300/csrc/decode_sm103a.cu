// Split-KV decode for sm_103a: one query row per (batch, query head), the
// whole K/V cache visible, cut into nsplit key chunks whose partial states
// (normalised output O_c and lse_c) are recombined through their log-sum-exp
// weights by a second kernel.
//
// Method: the smzdm digest ("Attention cannot be split like GEMM", section 5)
// -- a key shard's partial output can only be merged with the others through
// its lse state; adding raw partials is wrong because each shard's softmax
// has its own denominator.  SP FlashDecode exchanges exactly one
// [V_DIM + 1] state per (batch, q head) per shard; here the shards are key
// chunks on one GPU and the state is (O_c in fp32, lse_c).
//
// The split kernel is bound by HBM bandwidth (every K/V byte is read once and
// used for G = Hq/Hkv query heads), so it streams the cache with 128-bit
// read-only loads, keeps the G query rows in registers and does the dot
// products on the FMA pipe; no tensor cores.
#include <cuda_bf16.h>
#include <math_constants.h>

#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kDecThreads = 224;               // consumer threads (7 warps); + 1 producer warp
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kStageKeys = 8 * kDecWarps;      // keys per ring stage: 8 per consumer warp
constexpr int kStages = 3;                     // ring depth: 3 x 2 x 14 KB in flight (D = 128)

__device__ __forceinline__ bool warp_all_dec(bool v) { return __all_sync(0xFFFFFFFFu, v); }

// Contiguous global -> shared bulk copy (no tensor map), completion counted
// in bytes on `bar`; addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

struct alignas(16) Vec16 {
  uint32_t x, y, z, w;
};

// 8 bf16 (one 16-byte vector) -> 8 floats.  bf16 is the top half of a
// binary32, so the widening is a shift / mask.
__device__ __forceinline__ void widen8(const Vec16& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Same, as 4 packed pairs (element 2i in the low half of pair i).
__device__ __forceinline__ void widen8x2(const Vec16& v, uint64_t (&f)[4]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    f[i] = f32x2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
}

// Lanes [g*TPK, (g+1)*TPK) hold partial dot products of one key row with GT
// query heads (v[h]).  Reduce over the TPK lanes while halving the number of
// values per lane at each of the first log2(GT) steps (each lane keeps the
// half selected by its lane bit and adds the partner's copy of that half).
// Afterwards every lane holds the full sum for one head, head_of_lane().
template <int GT, int TPK>
__device__ __forceinline__ float reduce_heads(float (&v)[GT], int lane) {
  int n = GT;
#pragma unroll
  for (int delta = TPK / 2; delta >= 1; delta /= 2) {
    if (n > 1) {
      const bool upper = (lane & delta) != 0;
      const int half = n / 2;
#pragma unroll
      for (int i = 0; i < GT / 2; ++i) {
        if (i < half) {
          const float send = upper ? v[i] : v[i + half];
          const float keep = upper ? v[i + half] : v[i];
          v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, delta);
        }
      }
      n = half;
    } else {
      v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], delta);
    }
  }
  return v[0];
}

template <int GT, int TPK>
__device__ __forceinline__ int head_of_lane(int lane) {
  int h = 0, n = GT;
#pragma unroll
  for (int delta = TPK / 2; delta >= 1; delta /= 2) {
    if (n > 1) {
      if (lane & delta) h += n / 2;
      n /= 2;
    }
  }
  return h;
}

// Offset (within a TPK lane group) of the lowest lane holding head h.
template <int GT, int TPK>
__device__ __forceinline__ int rep_lane_of_head(int h) {
  int off = 0, n = GT;
#pragma unroll
  for (int delta = TPK / 2; delta >= 1; delta /= 2) {
    if (n > 1) {
      if (h >= n / 2) {
        off += delta;
        h -= n / 2;
      }
      n /= 2;
    }
  }
  return off;
}

// Lanes that are the lowest copy of their head value (the rest of the lane
// group duplicates it).
template <int GT, int TPK>
__device__ __forceinline__ bool is_rep_lane(int lane) {
  int n = GT, dup_mask = 0;
#pragma unroll
  for (int delta = TPK / 2; delta >= 1; delta /= 2) {
    if (n > 1)
      n /= 2;
    else
      dup_mask |= delta;
  }
  return (lane & dup_mask) == 0;
}

// grid (nsplit, Hkv * (G / GT), B); one CTA per (key chunk, kv head, group of
// GT query heads, batch).  A producer warp streams the chunk's K and V rows
// (contiguous in the cache) into a kStages-deep shared-memory ring with bulk
// async copies, kStageKeys keys per stage, so the loads in flight do not
// depend on registers or on how far the consumers are.  Each of the 7
// consumer warps takes 8 keys of every stage and runs its own online
// softmax; the warp states are merged at the end into the chunk's
// (O_c, lse_c).
template <int D, int GT>
__global__ void __launch_bounds__(kDecThreads + 32, (GT >= 8 ? 1 : 2))
    decode_split_kernel(const DecodeParams p) {
  constexpr int TPK = D / 8;      // lanes per key row, 16 bytes each
  constexpr int KPW = 32 / TPK;   // key rows per warp-wide shared-memory load
  constexpr int kWarpKeys = kStageKeys / kDecWarps;  // keys of a stage per warp
  constexpr int kU = kWarpKeys / KPW;                // loads per lane per stage and tensor
  constexpr int kRowBytes = D * 2;
  constexpr int kStageBytes = kStageKeys * kRowBytes;  // one tensor's part of a stage
  static_assert(GT <= TPK, "head group larger than the lane group");
  static_assert(kWarpKeys % KPW == 0, "stage split");

  extern __shared__ __align__(128) uint8_t dsmem[];
  uint8_t* ring = dsmem;  // [kStages][K rows | V rows]
  __shared__ uint64_t full_bar[kStages], empty_bar[kStages];
  __shared__ int abort_flag;
  __shared__ float sm_m[kDecWarps][GT];
  __shared__ float sm_l[kDecWarps][GT];
  __shared__ float sm_o[kDecWarps][GT][D];

  const int G = p.Hq / p.Hkv;
  const int ngroups = G / GT;
  const int split = blockIdx.x;
  const int hkv = blockIdx.y / ngroups;
  const int hq0 = hkv * G + (blockIdx.y % ngroups) * GT;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int C = (p.Nk + p.nsplit - 1) / p.nsplit;
  const int k0 = split * C;
  const int k1 = min(k0 + C, p.Nk);
  const int nstage = k1 > k0 ? (k1 - k0 + kStageKeys - 1) / kStageKeys : 0;
  const size_t head_off = (static_cast<size_t>(b) * p.Hkv + hkv) * static_cast<size_t>(p.Nk) * D;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kDecWarps);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const uint32_t abort_p = smem_u32(&abort_flag);

  if (warp == kDecWarps) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();  // every byte is read once
      const uint8_t* kg = static_cast<const uint8_t*>(p.k) + head_off * 2;
      const uint8_t* vg = static_cast<const uint8_t*>(p.v) + head_off * 2;
      int issued = 0;
      for (int i = 0; i < nstage; ++i) {
        const int slot = i % kStages;
        if (!mbar_wait(&empty_bar[slot], ((i / kStages) & 1) ^ 1, abort_p, p.err, kErrWaitLoad,
                       p.wait_limit_ns))
          break;
        const int key = k0 + i * kStageKeys;
        const uint32_t bytes = static_cast<uint32_t>(min(kStageKeys, k1 - key)) * kRowBytes;
        mbar_arrive_expect_tx(&full_bar[slot], 2 * bytes);
        uint8_t* dst = ring + slot * 2 * kStageBytes;
        bulk_load(dst, kg + static_cast<size_t>(key) * kRowBytes, bytes, &full_bar[slot], pol);
        bulk_load(dst + kStageBytes, vg + static_cast<size_t>(key) * kRowBytes, bytes,
                  &full_bar[slot], pol);
        issued = i + 1;
      }
      if (abort_set(abort_p)) {  // let the copies still in flight land before the CTA exits
        for (int i = max(0, issued - kStages); i < issued; ++i)
          for (int spin = 0; spin < (1 << 20); ++spin)
            if (mbar_try_wait(&full_bar[i % kStages], (i / kStages) & 1)) break;
      }
    }
  } else {
    // ---------------------------------------------------------------- consumers
    const int sub = lane / TPK;
    const int dc = lane % TPK;
    // query rows pre-scaled by scale*log2 e, so scores are in log2 units;
    // consecutive pairs of the lane's 8 dims packed for f32x2 arithmetic
    uint64_t qf2[GT][4];
    {
      const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(p.q) +
                                (static_cast<size_t>(b) * p.Hq + hq0) * D + dc * 8;
#pragma unroll
      for (int h = 0; h < GT; ++h) {
        float qf[8];
        widen8(*reinterpret_cast<const Vec16*>(qb + static_cast<size_t>(h) * D), qf);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          qf2[h][i] = f32x2(qf[2 * i] * p.scale_log2, qf[2 * i + 1] * p.scale_log2);
      }
    }
    const int hsel = head_of_lane<GT, TPK>(lane);
    float m_run = -CUDART_INF_F, l_run = 0.f;
    uint64_t acc2[GT][4];  // unnormalised output, pairs of dims
#pragma unroll
    for (int h = 0; h < GT; ++h)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc2[h][i] = f32x2(0.f, 0.f);

    for (int i = 0; i < nstage; ++i) {
      const int slot = i % kStages;
      if (!warp_all_dec(mbar_wait(&full_bar[slot], (i / kStages) & 1, abort_p, p.err,
                                  kErrWaitSoftmax, p.wait_limit_ns)))
        break;
      const int kbase = k0 + i * kStageKeys + warp * kWarpKeys;  // first key of this warp
      if (kbase < k1) {
        const uint8_t* ks = ring + slot * 2 * kStageBytes +
                            (warp * kWarpKeys + sub) * kRowBytes + dc * 16;
        const uint8_t* vs = ks + kStageBytes;
        float s[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int key = kbase + u * KPW + sub;
          uint64_t kf2[4];
          widen8x2(*reinterpret_cast<const Vec16*>(ks + u * KPW * kRowBytes), kf2);
          float part[GT];
#pragma unroll
          for (int h = 0; h < GT; ++h) {
            uint64_t a2 = mul_f32x2(qf2[h][0], kf2[0]);
#pragma unroll
            for (int i = 1; i < 4; ++i) a2 = fma_f32x2(qf2[h][i], kf2[i], a2);
            float lo, hi;
            unpack_f32x2(a2, lo, hi);
            part[h] = lo + hi;
          }
          s[u] = reduce_heads<GT, TPK>(part, lane);
          if (key >= k1) s[u] = -CUDART_INF_F;  // rows past the chunk end are stale data
        }
        // max of head hsel over the warp's keys of this stage
        float mx = s[0];
#pragma unroll
        for (int u = 1; u < kU; ++u) mx = fmaxf(mx, s[u]);
#pragma unroll
        for (int off = TPK; off < 32; off *= 2)
          mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
        const float m_new = fmaxf(m_run, mx);  // finite: key kbase is valid
        const float alpha = ex2_approx(m_run - m_new);
        m_run = m_new;
        float pu[kU], psum = 0.f;
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          pu[u] = ex2_approx(s[u] - m_new);
          psum += pu[u];
        }
        l_run = fmaf(l_run, alpha, psum);
#pragma unroll
        for (int h = 0; h < GT; ++h) {
          const float ah = __shfl_sync(0xFFFFFFFFu, alpha, rep_lane_of_head<GT, TPK>(h));
          const uint64_t ah2 = f32x2(ah, ah);
#pragma unroll
          for (int i = 0; i < 4; ++i) acc2[h][i] = mul_f32x2(acc2[h][i], ah2);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          Vec16 vraw = *reinterpret_cast<const Vec16*>(vs + u * KPW * kRowBytes);
          // rows past the chunk end hold stale data: their weight is exactly 0,
          // but 0 * NaN would not be, so zero the values too
          if (kbase + u * KPW + sub >= k1) vraw = Vec16{0, 0, 0, 0};
          uint64_t vf2[4];
          widen8x2(vraw, vf2);
#pragma unroll
          for (int h = 0; h < GT; ++h) {
            const float ph =
                __shfl_sync(0xFFFFFFFFu, pu[u], sub * TPK + rep_lane_of_head<GT, TPK>(h));
            const uint64_t ph2 = f32x2(ph, ph);
#pragma unroll
            for (int i = 0; i < 4; ++i) acc2[h][i] = fma_f32x2(ph2, vf2[i], acc2[h][i]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[slot]);
    }

    // let the combine kernel start launching while this CTA finishes
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    float acc[GT][8];
#pragma unroll
    for (int h = 0; h < GT; ++h)
#pragma unroll
      for (int i = 0; i < 4; ++i) unpack_f32x2(acc2[h][i], acc[h][2 * i], acc[h][2 * i + 1]);
    // merge the KPW key sub-groups of the warp (same running max)
#pragma unroll
    for (int off = TPK; off < 32; off *= 2) {
      l_run += __shfl_xor_sync(0xFFFFFFFFu, l_run, off);
#pragma unroll
      for (int h = 0; h < GT; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[h][e] += __shfl_xor_sync(0xFFFFFFFFu, acc[h][e], off);
    }
    if (sub == 0) {
#pragma unroll
      for (int h = 0; h < GT; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) sm_o[warp][h][dc * 8 + e] = acc[h][e];
      if (is_rep_lane<GT, TPK>(lane)) {
        sm_m[warp][hsel] = m_run;
        sm_l[warp][hsel] = l_run;
      }
    }
  }
  __syncthreads();

  // merge the warps: chunk state (O_c normalised, lse_c in natural log)
  for (int t = threadIdx.x; t < GT * D; t += kDecThreads + 32) {
    const int h = t / D, d = t % D;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, sm_m[w][h]);
    const size_t row = static_cast<size_t>(b) * p.Hq + hq0 + h;
    float out = 0.f, lse = -CUDART_INF_F;
    if (M != -CUDART_INF_F) {
      float L = 0.f, o = 0.f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float wgt = ex2_approx(sm_m[w][h] - M);
        L = fmaf(sm_l[w][h], wgt, L);
        o = fmaf(sm_o[w][h][d], wgt, o);
      }
      out = o / L;
      lse = (M + __log2f(L)) * 0.69314718055994530942f;
    }
    p.ws_o[(row * p.nsplit + split) * D + d] = out;
    if (d == 0) p.ws_lse[row * p.nsplit + split] = lse;
  }
}

// grid (B*Hq), D threads: log-sum-exp combine of the nsplit chunk states.
//   L = max_c lse_c + ln sum_c exp(lse_c - max),  O = sum_c exp(lse_c - L) O_c
template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const DecodeParams p) {
  // programmatic dependent launch: wait for the split kernel's results
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const size_t row = blockIdx.x;
  const int d = threadIdx.x;
  const float* lse_in = p.ws_lse + row * p.nsplit;
  constexpr float kLog2e = 1.4426950408889634f;
  float M = -CUDART_INF_F;
  for (int c = 0; c < p.nsplit; ++c) M = fmaxf(M, lse_in[c]);
  float S = 0.f;
  for (int c = 0; c < p.nsplit; ++c) S += ex2_approx((lse_in[c] - M) * kLog2e);
  const float L = M + __logf(S);
  float o = 0.f;
  const float* o_in = p.ws_o + row * p.nsplit * D + d;
  for (int c = 0; c < p.nsplit; ++c)
    o = fmaf(ex2_approx((lse_in[c] - L) * kLog2e), o_in[static_cast<size_t>(c) * D], o);
  if (p.o_state)
    p.o_state[row * D + d] = o;  // unrounded state for a further combine
  else
    static_cast<__nv_bfloat16*>(p.o)[row * D + d] = __float2bfloat16_rn(o);
  if (d == 0) p.lse[row] = L;
}

template <int D>
int pick_gt(int G) {
  constexpr int TPK = D / 8;
  int gt = 1;
  while (gt * 2 <= TPK && gt * 2 <= 8 && G % (gt * 2) == 0) gt *= 2;
  return gt;
}

template <int D>
constexpr int split_smem_bytes() {
  return kStages * 2 * kStageKeys * D * 2;
}

template <int D, int GT>
cudaError_t launch_split_t(const DecodeParams& p, cudaStream_t stream) {
  constexpr int smem = split_smem_bytes<D>();
  // the shared-memory opt-in is a per-device property of the function
  static std::atomic<bool> attr_done[64];  // zero-initialised: false
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(decode_split_kernel<D, GT>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_done[dev].store(true, std::memory_order_release);
  }
  const int G = p.Hq / p.Hkv;
  dim3 grid(p.nsplit, p.Hkv * (G / GT), p.B);
  decode_split_kernel<D, GT><<<grid, kDecThreads + 32, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_split_d(const DecodeParams& p, cudaStream_t stream) {
  switch (pick_gt<D>(p.Hq / p.Hkv)) {
    case 1: return launch_split_t<D, 1>(p, stream);
    case 2: return launch_split_t<D, 2>(p, stream);
    case 4: return launch_split_t<D, 4>(p, stream);
    case 8: return launch_split_t<D, 8>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool decode_supported(int G, int D) { return G >= 1 && (D == 64 || D == 128); }

cudaError_t launch_decode_split(const DecodeParams& p, cudaStream_t stream) {
  if (p.D == 128) return launch_split_d<128>(p, stream);
  if (p.D == 64) return launch_split_d<64>(p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_combine(const DecodeParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.B * p.Hq));
  cfg.blockDim = dim3(static_cast<unsigned>(p.D));
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.D == 128) return cudaLaunchKernelEx(&cfg, decode_combine_kernel<128>, p);
  if (p.D == 64) return cudaLaunchKernelEx(&cfg, decode_combine_kernel<64>, p);
  return cudaErrorInvalidValue;
}

}  // namespace attn
