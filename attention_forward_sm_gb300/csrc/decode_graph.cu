// attn_decode_graph_*: the split-KV decode step (split kernel + combine
// kernel, linked by programmatic dependent launch) captured once into a CUDA
// graph and replayed per step, so a step costs the host one graph launch.
// Source: smzdm digest of Zhihu posts, section 4 (decode fixed costs: CUDA
// Graph + PDL).
#include <cuda_runtime.h>
#include <stdint.h>

#include <new>

#include "../../include/attn.h"
#include "internal.h"

struct attn_decode_graph {
  cudaGraphExec_t exec = nullptr;
  cudaEvent_t done = nullptr;  // recorded after every replay
  void* scratch = nullptr;
};

namespace attn {
namespace {

void release(attn_decode_graph* g) {
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->done) cudaEventDestroy(g->done);
  if (g->scratch) cudaFree(g->scratch);
  delete g;
}

}  // namespace
}  // namespace attn

extern "C" {

int attn_decode_graph_create(const void* q, const void* kcache, const void* vcache, void* o,
                             float* lse, int B, int Hq, int Hkv, int Nk, int D, int nsplit,
                             attn_decode_graph** out) {
  using namespace attn;
  if (!out) return ATTN_ERR_NULL;
  *out = nullptr;
  if (!o) return ATTN_ERR_NULL;
  DecodeParams p;
  if (int rc = decode_prepare(q, kcache, vcache, o, nullptr, lse, B, Hq, Hkv, Nk, D, nsplit, &p))
    return rc;
  if (int rc = decode_bind_device(&p)) return rc;

  attn_decode_graph* g = new (std::nothrow) attn_decode_graph;
  if (!g) return ATTN_ERR_ALLOC;
  size_t o_bytes = 0;
  const size_t bytes = decode_scratch_bytes(p, &o_bytes);
  if (cudaMalloc(&g->scratch, bytes) != cudaSuccess) {
    cudaGetLastError();
    g->scratch = nullptr;
    release(g);
    return ATTN_ERR_ALLOC;
  }
  p.ws_o = static_cast<float*>(g->scratch);
  p.ws_lse = reinterpret_cast<float*>(static_cast<char*>(g->scratch) + o_bytes);
  if (cudaEventCreateWithFlags(&g->done, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    g->done = nullptr;
    release(g);
    return ATTN_ERR_CUDA;
  }

  // Capture on a private stream.  Relaxed mode: the launch helpers may set a
  // kernel attribute on their first use on this device, which is not a
  // stream operation and is harmless during capture.
  cudaStream_t cs = nullptr;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) {
    cudaGetLastError();
    release(g);
    return ATTN_ERR_CUDA;
  }
  int rc = ATTN_OK;
  cudaGraph_t graph = nullptr;
  if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
    rc = ATTN_ERR_CUDA;
  } else {
    if (launch_decode_split(p, cs) != cudaSuccess || launch_decode_combine(p, cs) != cudaSuccess)
      rc = ATTN_ERR_LAUNCH;
    // End the capture in every case, so the stream leaves capture mode.
    if (cudaStreamEndCapture(cs, &graph) != cudaSuccess && rc == ATTN_OK) rc = ATTN_ERR_CUDA;
  }
  if (rc == ATTN_OK && (!graph || cudaGraphInstantiate(&g->exec, graph, 0) != cudaSuccess)) {
    g->exec = nullptr;
    rc = ATTN_ERR_CUDA;
  }
  if (graph) cudaGraphDestroy(graph);
  cudaStreamDestroy(cs);
  if (rc != ATTN_OK) {
    cudaGetLastError();
    release(g);
    return rc;
  }
  *out = g;
  return ATTN_OK;
}

int attn_decode_graph_launch(attn_decode_graph* g, cudaStream_t stream) {
  if (!g || !g->exec) return ATTN_ERR_NULL;
  if (cudaGraphLaunch(g->exec, stream) != cudaSuccess) return ATTN_ERR_LAUNCH;
  if (cudaEventRecord(g->done, stream) != cudaSuccess) return ATTN_ERR_LAUNCH;
  return ATTN_OK;
}

int attn_decode_graph_destroy(attn_decode_graph* g) {
  if (!g) return ATTN_OK;
  int rc = ATTN_OK;
  // The event was recorded after the last replay (or never, when it is
  // trivially complete); the scratch must not be freed under a running replay.
  if (cudaEventSynchronize(g->done) != cudaSuccess) rc = ATTN_ERR_CUDA;
  attn::release(g);
  return rc;
}

}  // extern "C"
