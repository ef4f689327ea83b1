// attn_decode_splitkv_noalloc: the split-KV decode of attn_decode_splitkv,
// with its partial-state scratch taken from a fixed array in device memory
// instead of the stream-ordered allocator, so that a call allocates nothing.
//
// Who needs it: callers that must not allocate device memory while they
// run -- for example a serving loop whose memory is fully reserved up front
// by its own allocator, or latency-critical code that keeps every allocator
// call (which can take locks or wait on other work) off its hot path.  The
// price is a fixed block of device memory, held by every device that loads
// the library until the process exits, and a cap on the problem size.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "../../include/attn.h"
#include "internal.h"

namespace attn {
namespace {

// Scratch capacity in floats: partial outputs [B, Hq, nsplit, D] followed by
// partial lse [B, Hq, nsplit].  8 MiB holds B*Hq*nsplit*(D+1) <= 2 Mi floats,
// e.g. B=8, Hq=32, nsplit=32, D=128 (4.2 MB).
constexpr size_t kScratchFloats = ATTN_NOALLOC_SCRATCH_BYTES / sizeof(float);

static __device__ __align__(256) float g_decode_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;

// Per-device set-up, done once with that device current: check the compute
// capability and translate the scratch symbol into a device address (host
// code cannot pass the symbol itself to a kernel).
struct ScratchState {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  bool sm103 = false;
  float* ptr = nullptr;
};
ScratchState g_state[kMaxDevices];

int scratch_for_current_device(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_DEVICE;
  ScratchState& st = g_state[dev];
  std::call_once(st.once, [&st, dev] {
    int major = 0, minor = 0;
    st.err = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (st.err == cudaSuccess)
      st.err = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    st.sm103 = (major == 10 && minor == 3);
    if (st.err == cudaSuccess && st.sm103)
      st.err = cudaGetSymbolAddress(reinterpret_cast<void**>(&st.ptr), g_decode_scratch);
  });
  if (st.err != cudaSuccess || (st.sm103 && st.ptr == nullptr)) return ATTN_ERR_CUDA;
  if (!st.sm103) return ATTN_ERR_DEVICE;
  *out = st.ptr;
  return ATTN_OK;
}

}  // namespace
}  // namespace attn

extern "C" int attn_decode_splitkv_noalloc(const void* q, const void* kcache, const void* vcache,
                                           void* o, float* lse, int B, int Hq, int Hkv, int Nk,
                                           int D, int nsplit, cudaStream_t stream) {
  using namespace attn;
  if (!o) return ATTN_ERR_NULL;
  DecodeParams p;
  if (int rc = decode_prepare(q, kcache, vcache, o, nullptr, lse, B, Hq, Hkv, Nk, D, nsplit, &p))
    return rc;
  size_t o_bytes = 0;
  if (decode_scratch_bytes(p, &o_bytes) > ATTN_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_SCRATCH;
  if (int rc = decode_bind_device(&p)) return rc;
  float* scratch = nullptr;
  if (int rc = scratch_for_current_device(&scratch)) return rc;
  // Every partial state is written by the split kernel before the combine
  // kernel reads it, so the scratch needs no clearing between calls.
  p.ws_o = scratch;
  p.ws_lse = scratch + o_bytes / sizeof(float);
  if (launch_decode_split(p, stream) != cudaSuccess ||
      launch_decode_combine(p, stream) != cudaSuccess)
    return ATTN_ERR_LAUNCH;
  return ATTN_OK;
}
