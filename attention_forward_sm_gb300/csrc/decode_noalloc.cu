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

#include <atomic>
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

// Per-device set-up, done with that device current: check the compute
// capability and translate the scratch symbol into a device address (host
// code cannot pass the symbol itself to a kernel).  Under lazy module
// loading the address lookup is also what loads the array onto the device,
// so it can fail for lack of memory; only a completed set-up is kept, and a
// failed one is tried again on the next call.
struct ScratchState {
  std::mutex mu;
  std::atomic<int> ready{0};  // 1: sm_103, ptr valid; 2: not sm_103
  float* ptr = nullptr;
};
ScratchState g_state[kMaxDevices];

int scratch_for_current_device(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_DEVICE;
  ScratchState& st = g_state[dev];
  int ready = st.ready.load(std::memory_order_acquire);
  if (ready == 0) {
    std::lock_guard<std::mutex> lock(st.mu);
    ready = st.ready.load(std::memory_order_relaxed);
    if (ready == 0) {
      int major = 0, minor = 0;
      if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return ATTN_ERR_CUDA;
      if (major == 10 && minor == 3) {
        float* ptr = nullptr;
        if (cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_decode_scratch) !=
                cudaSuccess ||
            ptr == nullptr) {
          cudaGetLastError();  // clear the (non-sticky) error so later calls do not see it
          return ATTN_ERR_CUDA;
        }
        st.ptr = ptr;
        ready = 1;
      } else {
        ready = 2;
      }
      st.ready.store(ready, std::memory_order_release);
    }
  }
  if (ready == 2) return ATTN_ERR_DEVICE;
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
