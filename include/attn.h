/*
 * attn.h -- C ABI of the GB300 (sm_103a) attention library (libattn.so).
 *
 * Two operations, both asynchronous on the caller's CUDA stream:
 *
 *   attn_fwd             tiled, IO-aware attention forward (prefill):
 *                        O = softmax(scale * Q K^T [+ causal mask]) V and the
 *                        per-row log-sum-exp LSE, with grouped KV heads.
 *   attn_decode_splitkv  single-query decode over a contiguous K/V cache, the
 *                        keys cut into nsplit chunks whose partial states are
 *                        recombined through their LSE (split-KV / FlashDecode).
 *
 * Sources for the operations:
 *   - "FlashAttention-3 vs Triton Kernels" (dailyaiworld), introduction:
 *     FlashAttention's IO-aware tiling computes the softmax attention output
 *     without writing the N x N score matrix to HBM; the benchmark listing in
 *     "Benchmarking Triton vs FlashAttention-3" fixes the (batch, heads, seq,
 *     head_dim) tensor layout and the 4*B*H*S^2*D FLOP convention.
 *   - "Warp Specialization in Triton: Design and Roadmap" (PyTorch blog),
 *     "How the compiler does it": the load / MMA / softmax / correction /
 *     epilogue roles of the warp-specialised forward kernel.
 *   - smzdm digest, section 5 ("Attention cannot be split like GEMM"): each
 *     key shard carries an lse_i state with its output and the combine
 *     renormalises through it; summing raw partial outputs is wrong.
 *
 * Numerics (identical for both calls): bf16 inputs; scores, running max,
 * running sum and the output accumulator in fp32; the softmax probabilities
 * are rounded to bf16 before the P*V product; O is rounded to bf16
 * (round-to-nearest-even); LSE is fp32 in natural-log units and includes
 * the scale:  LSE = ln sum_j exp(scale * q . k_j).
 *
 * Ownership: the caller allocates and owns every buffer; the library keeps
 * no pointer after a call returns.  All pointers must be device pointers of
 * the current CUDA device, and the stream must belong to that device.
 *
 * Errors: every call validates its arguments before touching the GPU and
 * returns one of the ATTN_* codes below (0 on success).  A failed check
 * launches nothing and writes nothing.  Faults inside a kernel surface, as
 * for any CUDA call, at the caller's next synchronisation.  Kernels never
 * wait forever: a pipeline wait that exceeds its time limit makes the kernel
 * set a bit in the device error word and exit; read it with
 * attn_get_device_error().
 */
#ifndef ATTN_SM103A_H_
#define ATTN_SM103A_H_

#ifdef __cplusplus
extern "C" {
#endif

/* The runtime's stream handle; declared here so the header does not need the
 * CUDA headers (identical to cuda_runtime_api.h's typedef). */
typedef struct CUstream_st *cudaStream_t;

enum attn_status {
  ATTN_OK = 0,
  ATTN_ERR_NULL = -1,    /* a required pointer is NULL */
  ATTN_ERR_ALIGN = -2,   /* a pointer is not 16-byte aligned (TMA needs 16 B; 128 B recommended) */
  ATTN_ERR_SHAPE = -3,   /* a size is out of range (see each call) */
  ATTN_ERR_DEVICE = -4,  /* current device is not compute capability 10.3 (sm_103) */
  ATTN_ERR_LAUNCH = -5,  /* the kernel launch failed (cudaGetLastError after launch) */
  ATTN_ERR_ALLOC = -6,   /* stream-ordered allocation of the decode scratch failed */
  ATTN_ERR_TMA = -7,     /* cuTensorMapEncodeTiled rejected a tensor view */
  ATTN_ERR_CUDA = -8,    /* another CUDA runtime call failed */
  ATTN_ERR_SCRATCH = -9  /* the problem needs more than the fixed no-allocation scratch */
};

/* Bits of the device error word (attn_get_device_error). */
#define ATTN_DEVERR_WAIT_LOAD 0x1u    /* K/V loader gave up waiting for a free slot */
#define ATTN_DEVERR_WAIT_MMA 0x2u     /* MMA issuer gave up waiting for operands */
#define ATTN_DEVERR_WAIT_SOFTMAX 0x4u /* softmax gave up waiting for scores */
#define ATTN_DEVERR_WAIT_CORR 0x8u    /* correction / epilogue gave up waiting */
#define ATTN_DEVERR_SELFTEST 0x10u    /* attn_selftest_wait_timeout ran out, as intended */

/*
 * attn_fwd -- attention forward (prefill).
 *
 *   q    [B, Hq,  Nq, D] bf16, contiguous (row-major, D fastest)
 *   k, v [B, Hkv, Nk, D] bf16, contiguous
 *   o    [B, Hq,  Nq, D] bf16, written
 *   lse  [B, Hq,  Nq]    fp32, written (natural log, scale included)
 *
 * For query head h the KV head is floor(h / (Hq / Hkv)) (contiguous groups).
 * causal != 0: key j is visible to query row i iff j <= i (mask aligned at
 * row 0, "top-left"); rows i >= Nk then see all keys.  scale multiplies
 * q . k before the softmax (1/sqrt(D) is the usual choice); it must be
 * finite and >= 0 (0 gives uniform weights over the visible keys).
 *
 * Limits: B, Hq, Hkv, Nq, Nk >= 1; Hq % Hkv == 0; D in {64, 128};
 * B*Hq*ceil(Nq/256) < 2^31; every pointer 16-byte aligned; q/k/v/o must not
 * overlap o/lse.  Returns ATTN_OK or an ATTN_ERR_* code.
 */
int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
             int Hkv, int Nq, int Nk, int D, int causal, float scale, cudaStream_t stream);

/*
 * attn_fwd_rows -- attn_fwd on a contiguous block of the query rows of a
 * longer sequence: row i of this call is row q_offset + i of the problem,
 * so with causal != 0 it sees keys j <= q_offset + i (k and v hold keys
 * 0 .. Nk-1 of the whole sequence).  attn_fwd is attn_fwd_rows with
 * q_offset = 0; without causal masking q_offset has no effect.
 *
 * Source: smzdm digest of Zhihu posts, section 5 (SP AllGather attention:
 * each rank keeps its block of the sequence's queries and gathers the keys
 * and values of every rank before attending); the Python helper
 * attention_forward_sm_gb300.sp_prefill does the gather with
 * torch.distributed and calls this with the rank's row offset.
 *
 * Arguments, layouts and limits as attn_fwd, plus 0 <= q_offset <=
 * INT_MAX - Nq - 1024 (ATTN_ERR_SHAPE otherwise).
 */
int attn_fwd_rows(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
                  int Hkv, int Nq, int Nk, int D, int causal, int q_offset, float scale,
                  cudaStream_t stream);

/*
 * attn_fwd_host -- attn_fwd on operands in host memory (pinned memory,
 * e.g. from cudaHostAlloc, lets the copies run asynchronously and at full
 * speed; pageable memory works but the copies then block the host).
 *
 * Same arguments, layouts, numerics and results as attn_fwd, but q, k, v, o
 * and lse are HOST pointers.  The work is cut into units of whole
 * (batch, KV-head block) slices -- the smallest block of KV heads whose
 * query tiles fill the GPU about four times -- and pipelined through two
 * device slots: the inputs of unit u are copied in on one library-owned
 * stream while unit u-1 computes on `stream` and unit u-2's outputs are
 * copied out on another, so a call costs about the largest of the three
 * instead of their sum.  Results are bit-identical to attn_fwd on device
 * copies of the inputs.
 *
 * Asynchronous: returns once everything is enqueued; `stream` completes
 * only after the last output byte has reached o/lse.  The host buffers must
 * stay valid until then, and must not be written (inputs) or read (outputs)
 * before.  The device slots (attn_fwd_host_workspace_bytes) are taken with
 * cudaMallocAsync on `stream` and freed the same way.  Returns the
 * validation errors of attn_fwd (before any copy), ATTN_ERR_ALLOC, or
 * ATTN_ERR_CUDA if a copy, event or stream call fails.
 */
int attn_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
                  int Hkv, int Nq, int Nk, int D, int causal, float scale, cudaStream_t stream);
/* Device bytes attn_fwd_host takes for its two slots (0 for invalid sizes). */
long long attn_fwd_host_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nk, int D);

/*
 * attn_fwd_fp8 -- attention forward on FP8 inputs (the FP8 tensor-core path
 * named on the page "FlashAttention-3 vs Triton Kernels", introduction and
 * pipeline diagram).  The real operands are q_scale*Q, k_scale*K and
 * v_scale*V, where Q, K, V hold E4M3 codes (OCP 8-bit floating point,
 * no infinities):
 *
 *   q  [B, Hq,  Nq, 128] e4m3 codes, contiguous
 *   k  [B, Hkv, Nk, 128] e4m3 codes, contiguous
 *   vt [B, Hkv, 128, Nk] e4m3 codes: V transposed, keys fastest
 *   o  [B, Hq,  Nq, 128] bf16, written
 *   lse [B, Hq, Nq]      fp32, written (natural log of sum_j exp(s_j))
 *
 * with s_j = scale * q_scale * k_scale * <Q_i, K_j> and the mask and head
 * grouping of attn_fwd.  Numerics: S and the softmax statistics are fp32;
 * the softmax weights are rounded to E4M3 (after multiplying by 2^6, which
 * keeps the weights of interest out of the subnormal range) for the
 * FP8 P*V product, accumulated in fp32; the normaliser is summed from the
 * unrounded fp32 weights.  O is rounded to bf16.
 *
 * Limits: D == 128; Nk % 16 == 0 (V^T rows start on 16-byte boundaries);
 * scale, q_scale, k_scale, v_scale finite and >= 0; the other limits and
 * the return codes of attn_fwd.
 */
int attn_fwd_fp8(const void *q, const void *k, const void *vt, void *o, float *lse, int B, int Hq,
                 int Hkv, int Nq, int Nk, int D, int causal, float scale, float q_scale,
                 float k_scale, float v_scale, cudaStream_t stream);

/*
 * attn_decode_splitkv -- split-KV decode of one query row per (batch, head).
 *
 *   q       [B, Hq, D]       bf16, contiguous
 *   kcache  [B, Hkv, Nk, D]  bf16, contiguous (head-major cache)
 *   vcache  [B, Hkv, Nk, D]  bf16, contiguous
 *   o       [B, Hq, D]       bf16, written
 *   lse     [B, Hq]          fp32, written (natural log)
 *
 * All Nk keys are visible; the scale is 1/sqrt(D).  The key axis is cut
 * into nsplit chunks of ceil(Nk/nsplit) keys (the last one shorter, possibly
 * empty); each chunk yields a partial output normalised by its own softmax
 * denominator plus its lse, and a second kernel recombines them:
 *   L = ln sum_c exp(lse_c),   O = sum_c exp(lse_c - L) O_c.
 * The partial states (B*Hq*nsplit*(D+1)*4 bytes) live in a device buffer the
 * library keeps per stream: on each device it remembers the last 8 streams
 * it decoded on, each with one buffer taken from the stream-ordered
 * allocator, grown when a call needs more and otherwise reused, so a
 * repeated decode step allocates nothing.  Each use waits (on the GPU) for
 * the buffer's previous use, so calls never share scratch while running.
 * The buffers stay allocated until the process exits or their entry passes
 * to another stream.  During stream capture a call allocates its scratch on
 * the stream and frees it after the combine instead (the graph owns it).
 *
 * Limits: B, Hq, Hkv, Nk >= 1; Hq % Hkv == 0; D in {64, 128};
 * 1 <= nsplit <= Nk; B <= 65535; pointers 16-byte aligned.
 */
int attn_decode_splitkv(const void *q, const void *kcache, const void *vcache, void *o, float *lse,
                        int B, int Hq, int Hkv, int Nk, int D, int nsplit, cudaStream_t stream);

/*
 * Sequence-parallel decode building blocks (SP FlashDecode, smzdm digest,
 * section 5): each rank holds a contiguous shard of the key axis, computes
 * one state per (batch, q head) -- the shard's normalised output and its lse,
 * [D + 1] numbers -- the ranks exchange the states, and the states are
 * recombined through their lse weights.  Exchanged volume is independent of
 * the cache length.
 *
 * attn_decode_splitkv_states: attn_decode_splitkv over this rank's cache
 * shard, with the output kept in fp32 (o_state [B, Hq, D]) so it can be
 * combined again without an extra rounding; lse [B, Hq] fp32 (natural log).
 * Same arguments, limits and scratch as attn_decode_splitkv.
 */
int attn_decode_splitkv_states(const void *q, const void *kcache, const void *vcache,
                               float *o_state, float *lse, int B, int Hq, int Hkv, int Nk, int D,
                               int nsplit, cudaStream_t stream);

/*
 * attn_combine_states: log-sum-exp combine of nparts partial states per row:
 *   part_o [rows, nparts, D] fp32 (each normalised by its own softmax sum),
 *   part_lse [rows, nparts] fp32 (natural log; -inf marks an empty part),
 *   o [rows, D] bf16 and lse [rows] fp32 written:
 *   L = ln sum_c exp(lse_c),  O = sum_c exp(lse_c - L) O_c.
 * Every row needs at least one non-empty part.  D in {64, 128}.
 */
int attn_combine_states(const float *part_o, const float *part_lse, void *o, float *lse, int rows,
                        int nparts, int D, cudaStream_t stream);

/* Size of the fixed device scratch behind attn_decode_splitkv_noalloc. */
#define ATTN_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)

/*
 * attn_decode_splitkv_noalloc -- attn_decode_splitkv without any allocation.
 * (No counterpart on the method's pages: this is a deployment variant.)
 *
 * For callers that cannot allocate device memory at call time, e.g. a
 * serving loop whose device memory is reserved in full by its own allocator
 * before it starts, or latency-critical code that keeps allocator calls
 * (which may take locks or wait on other work) off its path.  Arguments,
 * layouts, numerics and results are those of attn_decode_splitkv; the
 * partial states live in a fixed array in device memory defined by this
 * library instead of in stream-ordered allocations.
 *
 *   - The array holds ATTN_NOALLOC_SCRATCH_BYTES of device memory on every
 *     device where the library's code is loaded, until the process exits.
 *     Under CUDA's default lazy module loading that happens during the
 *     first call on each device, so that first call itself commits the
 *     8 MiB: make it before reserving the rest of the device's memory.
 *   - A call needs B*Hq*nsplit*(D+1)*4 bytes of it (the decode workload
 *     B8 Hq32 D128 nsplit32 needs 4.2 MB); a larger problem returns
 *     ATTN_ERR_SCRATCH and launches nothing.
 *   - All calls on a device share the one array and it keeps the previous
 *     call's contents (every element a call reads is first written by that
 *     same call, so nothing needs clearing).  Two calls whose kernels overlap
 *     on the GPU -- e.g. on different streams without ordering between them
 *     -- race on the array and may both return wrong results: order them.
 *   - The first call on each device does a one-time set-up on the host (it
 *     loads the array and looks up its device address for the current
 *     device); make that first call before any stream capture on that
 *     device.  If the set-up fails (ATTN_ERR_CUDA, e.g. no memory left for
 *     the array) nothing is cached and the next call tries again.
 *   - Calls nothing that allocates or frees memory.
 */
int attn_decode_splitkv_noalloc(const void *q, const void *kcache, const void *vcache, void *o,
                                float *lse, int B, int Hq, int Hkv, int Nk, int D, int nsplit,
                                cudaStream_t stream);

/*
 * Decode step as a replayable CUDA graph.  Source: smzdm digest of Zhihu
 * posts, section 4: a decode step is two short kernels, so its fixed
 * per-step costs (host launch work, the gap between the split kernel and the
 * combine) matter; the remedy named there is a CUDA Graph around the step
 * with programmatic dependent launch (PDL) between the kernels.
 *
 * attn_decode_graph_create captures attn_decode_splitkv's two kernels (the
 * combine linked to the split by PDL) for the given buffers and sizes once,
 * and instantiates the graph; attn_decode_graph_launch replays it on any
 * stream of the same device: one graph launch per step, no argument checks,
 * no allocation.  Arguments, layouts, numerics and results of a replay are
 * those of attn_decode_splitkv on the buffers' contents at replay time.
 *
 *   - The handle owns its partial-state scratch (B*Hq*nsplit*(D+1)*4 bytes,
 *     cudaMalloc'ed at create; ATTN_ERR_ALLOC if that fails) and an event.
 *   - q, kcache, vcache, o and lse are bound by address: they must stay
 *     allocated, at the same addresses, until the handle is destroyed;
 *     their contents may change between replays (e.g. the next token's q).
 *   - Replays of one handle share its scratch: order them (one stream, or
 *     events), as for any kernel that writes the same buffer.
 *   - create returns the same validation errors as attn_decode_splitkv, plus
 *     ATTN_ERR_NULL for out == NULL and ATTN_ERR_CUDA if capture or
 *     instantiation fails; nothing is left allocated on failure.  It must be
 *     called with the target device current and no capture running on the
 *     calling thread.
 *   - destroy waits for the handle's last replay to finish, then frees
 *     everything; destroy(NULL) is a no-op returning ATTN_OK.
 */
typedef struct attn_decode_graph attn_decode_graph;
int attn_decode_graph_create(const void *q, const void *kcache, const void *vcache, void *o,
                             float *lse, int B, int Hq, int Hkv, int Nk, int D, int nsplit,
                             attn_decode_graph **out);
/* Replays the step on `stream`; ATTN_ERR_NULL for a NULL handle,
 * ATTN_ERR_LAUNCH if the graph launch fails. */
int attn_decode_graph_launch(attn_decode_graph *graph, cudaStream_t stream);
int attn_decode_graph_destroy(attn_decode_graph *graph);

/* Human-readable name of an ATTN_* status code (static string). */
const char *attn_status_string(int status);

/* Synchronises `stream`, then returns the device error word of the current
 * device (ATTN_DEVERR_* bits, 0 when no kernel gave up a wait) and clears
 * it.  Returns a negative ATTN_ERR_* code if a CUDA call fails. */
int attn_get_device_error(cudaStream_t stream);

/* Failure-detection self-test: launches one CTA that waits, through the same
 * bounded mbarrier wait the kernels use, on a barrier nothing arrives at.
 * The wait gives up after limit_us microseconds (1 .. 1e6), sets
 * ATTN_DEVERR_SELFTEST in the device error word and the kernel exits
 * normally, leaving the context usable; read the word with
 * attn_get_device_error().  Returns ATTN_OK once launched. */
int attn_selftest_wait_timeout(unsigned int limit_us, cudaStream_t stream);

/* Bytes of decode scratch one attn_decode_splitkv call takes. */
long long attn_decode_workspace_bytes(int B, int Hq, int D, int nsplit);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_SM103A_H_ */
