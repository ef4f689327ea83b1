// C ABI of libattn.so: argument validation, TMA tensor-map encoding, launches
// and error mapping.  The declarations and their contracts are in
// include/attn.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <limits.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "../../include/attn.h"
#include "internal.h"
#include "ptx.cuh"

namespace attn {

// Device error word: bits set by a kernel whose bounded wait ran out.
__device__ unsigned int g_error_word = 0;

namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: no healthy wait comes near it

struct DeviceState {
  std::once_flag once;
  bool is_sm103 = false;
  unsigned int* err_word = nullptr;
  cudaError_t init_error = cudaSuccess;
};
DeviceState g_dev[kMaxDevices];

std::once_flag g_encode_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Per-device checks, done once per device: compute capability 10.3, the
// device error word's address, the kernels' shared-memory opt-in.
int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_DEVICE;
  DeviceState& st = g_dev[dev];
  std::call_once(st.once, [&st, dev] {
    int major = 0, minor = 0;
    st.init_error = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (st.init_error == cudaSuccess)
      st.init_error = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    st.is_sm103 = (major == 10 && minor == 3);
    if (st.init_error == cudaSuccess && st.is_sm103)
      st.init_error = cudaGetSymbolAddress(reinterpret_cast<void**>(&st.err_word), g_error_word);
  });
  if (st.init_error != cudaSuccess) return ATTN_ERR_CUDA;
  if (!st.is_sm103) return ATTN_ERR_DEVICE;
  *out = &st;
  return ATTN_OK;
}

int encode_fn(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::call_once(g_encode_once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  if (!g_encode) return ATTN_ERR_CUDA;
  *fn = g_encode;
  return ATTN_OK;
}

// 3-D view [BH, N, D] of a contiguous bf16 tensor, box {64, 128, 1},
// 128-byte swizzle (the layout the MMA descriptors expect).
int encode_3d(CUtensorMap* map, const void* base, int D, int N, long long BH) {
  PFN_cuTensorMapEncodeTiled_v12000 fn;
  if (int rc = encode_fn(&fn)) return rc;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                           static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(D) * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_TMA;
}

// 3-D view [BH, rows, inner] of a contiguous e4m3 tensor (bytes), box
// {128, 128, 1}, 128-byte swizzle.  `inner` * 1 byte must be a multiple of 16.
int encode_3d_e4m3(CUtensorMap* map, const void* base, int inner, int rows, long long BH) {
  PFN_cuTensorMapEncodeTiled_v12000 fn;
  if (int rc = encode_fn(&fn)) return rc;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner),
                           static_cast<cuuint64_t>(rows) * static_cast<cuuint64_t>(inner)};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_TMA;
}

// One CTA waits, through the same bounded wait the pipelines use, on an
// mbarrier that nothing ever arrives at; the wait gives up after `limit_ns`
// and records `kErrSelfTest` in the device error word.
__global__ void selftest_wait_kernel(unsigned int* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  mbar_wait(&bar, 0, smem_u32(&abort_flag), err, kErrSelfTest, limit_ns);
}

}  // namespace

unsigned int* device_error_word() {
  DeviceState* st = nullptr;
  return device_state(&st) == ATTN_OK ? st->err_word : nullptr;
}

uint64_t wait_limit_ns() { return kWaitLimitNs; }

int decode_prepare(const void* q, const void* kcache, const void* vcache, void* o, float* o_state,
                   float* lse, int B, int Hq, int Hkv, int Nk, int D, int nsplit,
                   DecodeParams* p) {
  if (!q || !kcache || !vcache || !(o || o_state) || !lse) return ATTN_ERR_NULL;
  if (B < 1 || Hq < 1 || Hkv < 1 || Nk < 1 || Hq % Hkv != 0) return ATTN_ERR_SHAPE;
  if (D != 64 && D != 128) return ATTN_ERR_SHAPE;
  if (nsplit < 1 || nsplit > Nk) return ATTN_ERR_SHAPE;
  if (B > 65535 || Hq > 65535) return ATTN_ERR_SHAPE;
  if (!decode_supported(Hq / Hkv, D)) return ATTN_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o) ||
      !aligned16(o_state) || !aligned16(lse))
    return ATTN_ERR_ALIGN;
  *p = DecodeParams{};
  p->q = q;
  p->k = kcache;
  p->v = vcache;
  p->o = o;
  p->o_state = o_state;
  p->lse = lse;
  p->B = B;
  p->Hq = Hq;
  p->Hkv = Hkv;
  p->Nk = Nk;
  p->D = D;
  p->nsplit = nsplit;
  p->scale_log2 = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(D)));
  p->wait_limit_ns = kWaitLimitNs;
  return ATTN_OK;
}

int decode_bind_device(DecodeParams* p) {
  DeviceState* st = nullptr;
  if (int rc = device_state(&st)) return rc;
  p->err = st->err_word;
  return ATTN_OK;
}

size_t decode_scratch_bytes(const DecodeParams& p, size_t* o_bytes) {
  *o_bytes = static_cast<size_t>(p.B) * p.Hq * p.nsplit * p.D * sizeof(float);
  return *o_bytes + static_cast<size_t>(p.B) * p.Hq * p.nsplit * sizeof(float);
}

}  // namespace attn

using namespace attn;

extern "C" {

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_NULL: return "ATTN_ERR_NULL: a required pointer is NULL";
    case ATTN_ERR_ALIGN: return "ATTN_ERR_ALIGN: a pointer is not 16-byte aligned";
    case ATTN_ERR_SHAPE: return "ATTN_ERR_SHAPE: a size is out of range";
    case ATTN_ERR_DEVICE: return "ATTN_ERR_DEVICE: the current device is not sm_103";
    case ATTN_ERR_LAUNCH: return "ATTN_ERR_LAUNCH: kernel launch failed";
    case ATTN_ERR_ALLOC: return "ATTN_ERR_ALLOC: scratch allocation failed";
    case ATTN_ERR_TMA: return "ATTN_ERR_TMA: tensor map encoding failed";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA: a CUDA runtime call failed";
    case ATTN_ERR_SCRATCH:
      return "ATTN_ERR_SCRATCH: the problem needs more than the fixed no-allocation scratch";
    default: return "unknown attn status";
  }
}

long long attn_decode_workspace_bytes(int B, int Hq, int D, int nsplit) {
  if (B < 1 || Hq < 1 || D < 1 || nsplit < 1) return 0;
  return static_cast<long long>(B) * Hq * nsplit * (D + 1) * 4;
}

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
             int Hkv, int Nq, int Nk, int D, int causal, float scale, cudaStream_t stream) {
  return attn_fwd_rows(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, causal, 0, scale, stream);
}

int attn_fwd_rows(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                  int Hkv, int Nq, int Nk, int D, int causal, int q_offset, float scale,
                  cudaStream_t stream) {
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_NULL;
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nk < 1 || Hq % Hkv != 0) return ATTN_ERR_SHAPE;
  if (D != 64 && D != 128) return ATTN_ERR_SHAPE;
  if (!isfinite(scale) || scale < 0.f) return ATTN_ERR_SHAPE;
  // the kernel forms q_offset + (row within the call) + a few tiles in int
  if (q_offset < 0 || q_offset > INT_MAX - Nq - 1024) return ATTN_ERR_SHAPE;
  const long long nqb = (Nq + 255) / 256;
  // work units (pairs of query tiles) are counted in int, with a grid's worth of headroom
  if (static_cast<long long>(B) * Hq * nqb >= (1ll << 31) - 65536) return ATTN_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_ALIGN;
  DeviceState* st = nullptr;
  if (int rc = device_state(&st)) return rc;

  FwdParams p = {};
  if (int rc = encode_3d(&p.tmap_q, q, D, Nq, static_cast<long long>(B) * Hq)) return rc;
  if (int rc = encode_3d(&p.tmap_k, k, D, Nk, static_cast<long long>(B) * Hkv)) return rc;
  if (int rc = encode_3d(&p.tmap_v, v, D, Nk, static_cast<long long>(B) * Hkv)) return rc;
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Nq = Nq;
  p.Nk = Nk;
  p.D = D;
  p.causal = causal ? 1 : 0;
  p.q_offset = causal ? q_offset : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.o_scale = 1.f;
  p.err = st->err_word;
  p.wait_limit_ns = kWaitLimitNs;
  if (launch_fwd(p, stream) != cudaSuccess) return ATTN_ERR_LAUNCH;
  return ATTN_OK;
}

int attn_fwd_fp8(const void* q, const void* k, const void* vt, void* o, float* lse, int B, int Hq,
                 int Hkv, int Nq, int Nk, int D, int causal, float scale, float q_scale,
                 float k_scale, float v_scale, cudaStream_t stream) {
  if (!q || !k || !vt || !o || !lse) return ATTN_ERR_NULL;
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nk < 1 || Hq % Hkv != 0) return ATTN_ERR_SHAPE;
  if (D != 128 || Nk % 16 != 0) return ATTN_ERR_SHAPE;
  for (float x : {scale, q_scale, k_scale, v_scale})
    if (!isfinite(x) || x < 0.f) return ATTN_ERR_SHAPE;
  const float s_qk = scale * q_scale * k_scale;
  if (!isfinite(s_qk)) return ATTN_ERR_SHAPE;
  const long long nqb = (Nq + 255) / 256;
  // work units (pairs of query tiles) are counted in int, with a grid's worth of headroom
  if (static_cast<long long>(B) * Hq * nqb >= (1ll << 31) - 65536) return ATTN_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(vt) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_ALIGN;
  DeviceState* st = nullptr;
  if (int rc = device_state(&st)) return rc;

  FwdParams p = {};
  if (int rc = encode_3d_e4m3(&p.tmap_q, q, D, Nq, static_cast<long long>(B) * Hq)) return rc;
  if (int rc = encode_3d_e4m3(&p.tmap_k, k, D, Nk, static_cast<long long>(B) * Hkv)) return rc;
  if (int rc = encode_3d_e4m3(&p.tmap_v, vt, Nk, D, static_cast<long long>(B) * Hkv)) return rc;
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Nq = Nq;
  p.Nk = Nk;
  p.D = D;
  p.causal = causal ? 1 : 0;
  p.fp8 = 1;
  p.scale_log2 = s_qk * 1.4426950408889634f;
  p.o_scale = v_scale;
  p.err = st->err_word;
  p.wait_limit_ns = kWaitLimitNs;
  if (launch_fwd(p, stream) != cudaSuccess) return ATTN_ERR_LAUNCH;
  return ATTN_OK;
}

// Split + combine with stream-ordered scratch for the partial states.
int attn_decode_splitkv(const void* q, const void* kcache, const void* vcache, void* o, float* lse,
                        int B, int Hq, int Hkv, int Nk, int D, int nsplit, cudaStream_t stream) {
  if (!o) return ATTN_ERR_NULL;
  DecodeParams p;
  if (int rc = decode_prepare(q, kcache, vcache, o, nullptr, lse, B, Hq, Hkv, Nk, D, nsplit, &p))
    return rc;
  return decode_with_cached_scratch(p, stream);
}

int attn_decode_splitkv_states(const void* q, const void* kcache, const void* vcache,
                               float* o_state, float* lse, int B, int Hq, int Hkv, int Nk, int D,
                               int nsplit, cudaStream_t stream) {
  if (!o_state) return ATTN_ERR_NULL;
  DecodeParams p;
  if (int rc =
          decode_prepare(q, kcache, vcache, nullptr, o_state, lse, B, Hq, Hkv, Nk, D, nsplit, &p))
    return rc;
  return decode_with_cached_scratch(p, stream);
}

int attn_combine_states(const float* part_o, const float* part_lse, void* o, float* lse,
                        int rows, int nparts, int D, cudaStream_t stream) {
  if (!part_o || !part_lse || !o || !lse) return ATTN_ERR_NULL;
  if (rows < 1 || nparts < 1 || (D != 64 && D != 128)) return ATTN_ERR_SHAPE;
  if (!aligned16(part_o) || !aligned16(o)) return ATTN_ERR_ALIGN;
  DeviceState* st = nullptr;
  if (int rc = device_state(&st)) return rc;
  DecodeParams p = {};
  p.o = o;
  p.lse = lse;
  p.ws_o = const_cast<float*>(part_o);
  p.ws_lse = const_cast<float*>(part_lse);
  p.B = rows;
  p.Hq = 1;
  p.Hkv = 1;
  p.D = D;
  p.nsplit = nparts;
  p.err = st->err_word;
  p.wait_limit_ns = kWaitLimitNs;
  return launch_decode_combine(p, stream) == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

int attn_selftest_wait_timeout(unsigned int limit_us, cudaStream_t stream) {
  if (limit_us < 1 || limit_us > 1000000) return ATTN_ERR_SHAPE;
  DeviceState* st = nullptr;
  if (int rc = device_state(&st)) return rc;
  selftest_wait_kernel<<<1, 32, 0, stream>>>(st->err_word,
                                             static_cast<uint64_t>(limit_us) * 1000ull);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

int attn_get_device_error(cudaStream_t stream) {
  DeviceState* st = nullptr;
  if (int rc = device_state(&st)) return rc;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpy(&word, st->err_word, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (word && cudaMemset(st->err_word, 0, sizeof word) != cudaSuccess) return ATTN_ERR_CUDA;
  return static_cast<int>(word & 0x7FFFFFFFu);
}

}  // extern "C"
