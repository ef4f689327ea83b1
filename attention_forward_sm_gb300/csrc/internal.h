// Host-side interface between the C ABI (api.cu) and the kernel translation
// units (fwd_sm103a.cu, decode_sm103a.cu).  Not part of the public header.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn {

// Bits of the device error word (also listed in include/attn.h).
enum : unsigned int {
  kErrWaitLoad = 1u << 0,     // loader gave up waiting for a free K/V slot
  kErrWaitMma = 1u << 1,      // MMA issuer gave up waiting for data / P / correction
  kErrWaitSoftmax = 1u << 2,  // softmax gave up waiting for S
  kErrWaitCorr = 1u << 3,     // correction / epilogue gave up waiting
  kErrSelfTest = 1u << 4,     // the wait self-test ran out, as intended
};

// Forward (prefill) launch parameters.  Tensor maps are 3-D views with a
// 128-byte swizzle: bf16 [B*H, N, D] with box {64, 128, 1}; for FP8, e4m3
// Q and K [B*H, N, D] with box {128, 128, 1} and V^T [B*Hkv, D, Nk] with box
// {128 keys, 128 rows, 1}.
struct FwdParams {
  CUtensorMap tmap_q, tmap_k, tmap_v;
  void* o;             // [B, Hq, Nq, D] bf16
  float* lse;          // [B, Hq, Nq] fp32
  int B, Hq, Hkv, Nq, Nk, D;
  int causal;
  int q_offset;        // causal: row i of this call is row q_offset + i of the problem
  int fp8;             // e4m3 Q, K, V^T
  int group_heads;     // causal unit order: query heads per group (a multiple of Hq/Hkv)
  float scale_log2;    // scale * log2(e) (FP8: times q_scale * k_scale)
  float o_scale;       // O multiplier (FP8: v_scale; bf16: 1)
  unsigned int* err;   // device error word
  uint64_t wait_limit_ns;
};

// Split-KV decode launch parameters.
struct DecodeParams {
  const void* q;       // [B, Hq, D] bf16
  const void* k;       // [B, Hkv, Nk, D] bf16
  const void* v;       // [B, Hkv, Nk, D] bf16
  void* o;             // [B, Hq, D] bf16 (unless o_state is set)
  float* o_state;      // optional [B, Hq, D] fp32 output instead of o
  float* lse;          // [B, Hq] fp32
  float* ws_o;         // [B, Hq, nsplit, D] fp32 partial outputs (normalised per chunk)
  float* ws_lse;       // [B, Hq, nsplit] fp32 partial lse (natural log)
  int B, Hq, Hkv, Nk, D, nsplit;
  float scale_log2;
  unsigned int* err;   // device error word
  uint64_t wait_limit_ns;
};

// Device error word of the current device (one-time per-device set-up);
// nullptr when the current device is unusable.
unsigned int* device_error_word();
uint64_t wait_limit_ns();

cudaError_t launch_fwd(const FwdParams& p, cudaStream_t stream);
size_t fwd_smem_bytes(int D, bool fp8);

// Checks the arguments of a split-KV decode on the host (exactly one of o /
// o_state is used; the other may be NULL) and fills every field of *p but the
// scratch pointers and the error word.  Returns an ATTN_* status.
int decode_prepare(const void* q, const void* kcache, const void* vcache, void* o, float* o_state,
                   float* lse, int B, int Hq, int Hkv, int Nk, int D, int nsplit,
                   DecodeParams* p);
// Checks the current device (sm_103) and sets p->err to its error word.
int decode_bind_device(DecodeParams* p);
// Bytes of partial-state scratch a decode needs; *o_bytes = the partial
// outputs' share (the partial lse follow them).
size_t decode_scratch_bytes(const DecodeParams& p, size_t* o_bytes);

// Binds the device, takes the partial-state scratch from the per-stream cache
// (or, during stream capture, from the stream-ordered allocator) and queues
// the split and combine kernels.  Returns an ATTN_* status.
int decode_with_cached_scratch(DecodeParams& p, cudaStream_t stream);
cudaError_t launch_decode_split(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_decode_combine(const DecodeParams& p, cudaStream_t stream);
bool decode_supported(int G, int D);

}  // namespace attn
