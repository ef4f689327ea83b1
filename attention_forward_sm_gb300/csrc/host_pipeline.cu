// attn_fwd_host: the prefill forward on operands in host memory.  The work is
// cut into units of whole (batch, KV-head block) slices, each large enough to
// fill the GPU several times over; unit u's inputs are copied to the device
// on one stream while unit u-1 computes on the caller's stream and unit u-2's
// outputs are copied back on a third, through two device slots.  The total
// time then approaches the largest of the three (usually the host-to-device
// copy) instead of their sum.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/attn.h"
#include "internal.h"

namespace attn {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kSlots = 2;
constexpr long long kMinCtasPerUnit = 4 * 152;  // about four waves of one CTA per SM

struct CopyStreams {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  cudaStream_t h2d = nullptr, d2h = nullptr;
};
CopyStreams g_streams[kMaxDevices];

int copy_streams(cudaStream_t* h2d, cudaStream_t* d2h) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_DEVICE;
  CopyStreams& cs = g_streams[dev];
  std::call_once(cs.once, [&cs] {
    cs.err = cudaStreamCreateWithFlags(&cs.h2d, cudaStreamNonBlocking);
    if (cs.err == cudaSuccess) cs.err = cudaStreamCreateWithFlags(&cs.d2h, cudaStreamNonBlocking);
  });
  if (cs.err != cudaSuccess) return ATTN_ERR_CUDA;
  *h2d = cs.h2d;
  *d2h = cs.d2h;
  return ATTN_OK;
}

struct Plan {
  int hc;           // KV heads per unit
  int units_per_b;  // ceil(Hkv / hc)
  size_t q_bytes, kv_bytes, lse_bytes, slot_bytes;
};

Plan make_plan(int Hq, int Hkv, int Nq, int Nk, int D) {
  const int G = Hq / Hkv;
  const long long pairs = (Nq + 255) / 256;
  int hc = 1;
  while (hc < Hkv && static_cast<long long>(hc) * G * pairs < kMinCtasPerUnit) ++hc;
  // the same number of blocks, as even as possible
  const int blocks = (Hkv + hc - 1) / hc;
  hc = (Hkv + blocks - 1) / blocks;
  Plan pl;
  pl.hc = hc;
  pl.units_per_b = (Hkv + hc - 1) / hc;
  pl.q_bytes = static_cast<size_t>(hc) * G * Nq * D * 2;
  pl.kv_bytes = static_cast<size_t>(hc) * Nk * D * 2;
  pl.lse_bytes = static_cast<size_t>(hc) * G * Nq * 4;
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  // q, k, v, o, lse of one unit
  pl.slot_bytes = up(pl.q_bytes) * 2 + up(pl.kv_bytes) * 2 + up(pl.lse_bytes);
  return pl;
}

}  // namespace
}  // namespace attn

extern "C" {

long long attn_fwd_host_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nk, int D) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nk < 1 || Hq % Hkv != 0) return 0;
  if (D != 64 && D != 128) return 0;
  return static_cast<long long>(attn::kSlots * attn::make_plan(Hq, Hkv, Nq, Nk, D).slot_bytes);
}

int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                  int Hkv, int Nq, int Nk, int D, int causal, float scale, cudaStream_t stream) {
  using namespace attn;
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_NULL;
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nk < 1 || Hq % Hkv != 0) return ATTN_ERR_SHAPE;
  if (D != 64 && D != 128) return ATTN_ERR_SHAPE;
  if (!isfinite(scale) || scale < 0.f) return ATTN_ERR_SHAPE;
  const Plan pl = make_plan(Hq, Hkv, Nq, Nk, D);
  const int G = Hq / Hkv;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  if (int rc = copy_streams(&h2d, &d2h)) return rc;

  // slot events: inputs on the device, compute done, outputs back on the host
  cudaEvent_t entry = nullptr, in_ready[kSlots] = {}, computed[kSlots] = {}, out_done[kSlots] = {};
  int rc = ATTN_OK;
  auto mk = [&rc](cudaEvent_t* e) {
    if (rc == ATTN_OK && cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess)
      rc = ATTN_ERR_CUDA;
  };
  mk(&entry);
  for (int s = 0; s < kSlots; ++s) {
    mk(&in_ready[s]);
    mk(&computed[s]);
    mk(&out_done[s]);
  }
  char* ws = nullptr;
  if (rc == ATTN_OK &&
      cudaMallocAsync(reinterpret_cast<void**>(&ws), kSlots * pl.slot_bytes, stream) != cudaSuccess)
    rc = ATTN_ERR_ALLOC;
  // the copy streams start after the caller's earlier work (and the
  // workspace allocation) on `stream`
  if (rc == ATTN_OK && (cudaEventRecord(entry, stream) != cudaSuccess ||
                        cudaStreamWaitEvent(h2d, entry, 0) != cudaSuccess ||
                        cudaStreamWaitEvent(d2h, entry, 0) != cudaSuccess))
    rc = ATTN_ERR_CUDA;

  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const char* qh = static_cast<const char*>(q);
  const char* kh = static_cast<const char*>(k);
  const char* vh = static_cast<const char*>(v);
  char* oh = static_cast<char*>(o);
  char* lh = reinterpret_cast<char*>(lse);
  const int units = B * pl.units_per_b;
  for (int u = 0; u < units && rc == ATTN_OK; ++u) {
    const int s = u % kSlots;
    const int b = u / pl.units_per_b, h0 = (u % pl.units_per_b) * pl.hc;
    const int hc = (h0 + pl.hc <= Hkv) ? pl.hc : Hkv - h0;
    char* slot = ws + s * pl.slot_bytes;
    char* dq = slot;
    char* dk = dq + up(pl.q_bytes);
    char* dv = dk + up(pl.kv_bytes);
    char* dout = dv + up(pl.kv_bytes);
    float* dl = reinterpret_cast<float*>(dout + up(pl.q_bytes));
    const size_t q_off = (static_cast<size_t>(b) * Hq + static_cast<size_t>(h0) * G) * Nq * D * 2;
    const size_t kv_off = (static_cast<size_t>(b) * Hkv + h0) * Nk * D * 2;
    const size_t l_off = (static_cast<size_t>(b) * Hq + static_cast<size_t>(h0) * G) * Nq * 4;
    const size_t q_n = static_cast<size_t>(hc) * G * Nq * D * 2;
    const size_t kv_n = static_cast<size_t>(hc) * Nk * D * 2;
    const size_t l_n = static_cast<size_t>(hc) * G * Nq * 4;
    // inputs: the slot's previous unit must have finished reading them
    if (u >= kSlots && cudaStreamWaitEvent(h2d, computed[s], 0) != cudaSuccess) rc = ATTN_ERR_CUDA;
    if (rc == ATTN_OK &&
        (cudaMemcpyAsync(dq, qh + q_off, q_n, cudaMemcpyHostToDevice, h2d) != cudaSuccess ||
         cudaMemcpyAsync(dk, kh + kv_off, kv_n, cudaMemcpyHostToDevice, h2d) != cudaSuccess ||
         cudaMemcpyAsync(dv, vh + kv_off, kv_n, cudaMemcpyHostToDevice, h2d) != cudaSuccess ||
         cudaEventRecord(in_ready[s], h2d) != cudaSuccess))
      rc = ATTN_ERR_CUDA;
    // compute: inputs present, and the slot's previous outputs copied out
    if (rc == ATTN_OK && (cudaStreamWaitEvent(stream, in_ready[s], 0) != cudaSuccess ||
                          (u >= kSlots && cudaStreamWaitEvent(stream, out_done[s], 0) != cudaSuccess)))
      rc = ATTN_ERR_CUDA;
    if (rc == ATTN_OK) {
      rc = attn_fwd(dq, dk, dv, dout, dl, 1, hc * G, hc, Nq, Nk, D, causal, scale, stream);
      if (rc == ATTN_OK && cudaEventRecord(computed[s], stream) != cudaSuccess) rc = ATTN_ERR_CUDA;
    }
    // outputs back
    if (rc == ATTN_OK &&
        (cudaStreamWaitEvent(d2h, computed[s], 0) != cudaSuccess ||
         cudaMemcpyAsync(oh + q_off, dout, q_n, cudaMemcpyDeviceToHost, d2h) != cudaSuccess ||
         cudaMemcpyAsync(lh + l_off, dl, l_n, cudaMemcpyDeviceToHost, d2h) != cudaSuccess ||
         cudaEventRecord(out_done[s], d2h) != cudaSuccess))
      rc = ATTN_ERR_CUDA;
  }
  // `stream` completes only after every copy back; then the workspace goes
  if (ws) {
    for (int s = 0; s < kSlots; ++s)
      if (cudaStreamWaitEvent(stream, out_done[s], 0) != cudaSuccess && rc == ATTN_OK)
        rc = ATTN_ERR_CUDA;
    // also order after the last input copies (a failed unit may have left
    // copies in flight on the h2d stream)
    if (cudaEventRecord(entry, h2d) != cudaSuccess || cudaStreamWaitEvent(stream, entry, 0) != cudaSuccess) {
      if (rc == ATTN_OK) rc = ATTN_ERR_CUDA;
    }
    if (cudaFreeAsync(ws, stream) != cudaSuccess && rc == ATTN_OK) rc = ATTN_ERR_CUDA;
  }
  // events may be destroyed while work that records them is pending
  for (cudaEvent_t e : {entry, in_ready[0], in_ready[1], computed[0], computed[1], out_done[0],
                        out_done[1]})
    if (e) cudaEventDestroy(e);
  if (rc != ATTN_OK) cudaGetLastError();
  return rc;
}

}  // extern "C"
