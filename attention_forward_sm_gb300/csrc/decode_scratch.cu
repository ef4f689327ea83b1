// Partial-state scratch of attn_decode_splitkv / attn_decode_splitkv_states:
// a small per-device cache of device buffers, one per recently used stream,
// so that a decode step allocates nothing once its stream has been seen.
//
// Why: a stream-ordered cudaMallocAsync + cudaFreeAsync pair around the two
// decode kernels costs about 6 us of GPU time per call on GB300 (measured:
// 342 us per call against 336 us with a fixed scratch on the B8 Hq32 Hkv8
// Nk65536 step), about 2 % of a bandwidth-bound step.
//
// Ordering.  A buffer belongs to one stream at a time.  Each use records the
// entry's event after the launches and the next use waits on it, so a buffer
// is never used by two calls at once, even when a destroyed stream's handle
// comes back for a new stream while the old one still has work queued.  A
// buffer that grows, or whose entry is taken over by another stream, is freed
// stream-ordered after that event.  Calls during stream capture take the
// plain stream-ordered allocation path, so a captured graph owns its scratch.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/attn.h"
#include "internal.h"

namespace attn {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kEntries = 8;  // streams remembered per device

struct Entry {
  cudaStream_t stream = nullptr;
  void* ptr = nullptr;
  size_t bytes = 0;
  cudaEvent_t done = nullptr;  // recorded after the entry's last use
  unsigned long long last_use = 0;
  bool live = false;
};

struct Cache {
  std::mutex mu;
  Entry e[kEntries];
  unsigned long long tick = 0;
};
Cache g_cache[kMaxDevices];

int plain_path(DecodeParams& p, size_t bytes, size_t o_bytes, cudaStream_t stream) {
  void* ws = nullptr;
  if (cudaMallocAsync(&ws, bytes, stream) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_ALLOC;
  }
  p.ws_o = static_cast<float*>(ws);
  p.ws_lse = reinterpret_cast<float*>(static_cast<char*>(ws) + o_bytes);
  int rc = ATTN_OK;
  if (launch_decode_split(p, stream) != cudaSuccess ||
      launch_decode_combine(p, stream) != cudaSuccess)
    rc = ATTN_ERR_LAUNCH;
  if (cudaFreeAsync(ws, stream) != cudaSuccess && rc == ATTN_OK) rc = ATTN_ERR_CUDA;
  return rc;
}

}  // namespace

int decode_with_cached_scratch(DecodeParams& p, cudaStream_t stream) {
  if (int rc = decode_bind_device(&p)) return rc;
  size_t o_bytes = 0;
  const size_t bytes = decode_scratch_bytes(p, &o_bytes);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  if (cap != cudaStreamCaptureStatusNone) return plain_path(p, bytes, o_bytes, stream);

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_DEVICE;
  Cache& c = g_cache[dev];
  // held until the launches and the event record are queued, so that no
  // other host thread frees or regrows this buffer in between
  std::lock_guard<std::mutex> lock(c.mu);
  Entry* en = nullptr;
  for (Entry& x : c.e)
    if (x.live && x.stream == stream) en = &x;
  if (!en) {
    // a free entry, else the least recently used one
    for (Entry& x : c.e)
      if (!x.live) {
        en = &x;
        break;
      }
    if (!en) {
      en = &c.e[0];
      for (Entry& x : c.e)
        if (x.last_use < en->last_use) en = &x;
    }
    en->live = true;
    en->stream = stream;
    if (!en->done && cudaEventCreateWithFlags(&en->done, cudaEventDisableTiming) != cudaSuccess) {
      en->live = false;
      return ATTN_ERR_CUDA;
    }
  }
  // after the entry's previous use, whichever stream made it
  if (cudaStreamWaitEvent(stream, en->done, 0) != cudaSuccess) return ATTN_ERR_CUDA;
  if (en->bytes < bytes) {
    if (en->ptr && cudaFreeAsync(en->ptr, stream) != cudaSuccess) {
      en->live = false;
      return ATTN_ERR_CUDA;
    }
    en->ptr = nullptr;
    en->bytes = 0;
    if (cudaMallocAsync(&en->ptr, bytes, stream) != cudaSuccess) {
      cudaGetLastError();
      en->ptr = nullptr;
      en->live = false;
      return ATTN_ERR_ALLOC;
    }
    en->bytes = bytes;
  }
  en->last_use = ++c.tick;
  p.ws_o = static_cast<float*>(en->ptr);
  p.ws_lse = reinterpret_cast<float*>(static_cast<char*>(en->ptr) + o_bytes);
  int rc = ATTN_OK;
  if (launch_decode_split(p, stream) != cudaSuccess ||
      launch_decode_combine(p, stream) != cudaSuccess)
    rc = ATTN_ERR_LAUNCH;
  // recorded even after a failed launch: whatever did get queued is covered
  if (cudaEventRecord(en->done, stream) != cudaSuccess && rc == ATTN_OK) rc = ATTN_ERR_CUDA;
  return rc;
}

}  // namespace attn
