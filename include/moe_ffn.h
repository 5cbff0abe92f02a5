/*
 * moe_ffn.h -- C ABI of the fused mixture-of-experts FFN layer for GB300
 * (sm_103a), one GPU.
 *
 * The layer is the one named in "ggml-cuda: overlap the MoE shared expert on
 * a separate stream" (ROCm/llama.cpp PR #36, "What this changes"): a router,
 * top-k routed SwiGLU experts and a gated shared expert forked from the same
 * FFN input and joined by add(ffn_moe_out, ffn_shexp), in the small-batch
 * (decode) mat-vec regime.  Here the two branches are one fused operator;
 * nothing is overlapped across CUDA streams.
 *
 * Per token t (x_t is one row of x):
 *   logit[e] = sum_h router_w[e,h] x_t[h]                        (fp32)
 *   ids      = the top_k largest logits, larger first, equal logits ordered
 *              by the lower expert index
 *   p_j      = exp(logit[ids_j] - logit[ids_0]) / sum_i exp(logit[ids_i] - logit[ids_0])
 *              (softmax over all experts followed by renormalisation of the
 *              kept top_k: the same numbers)
 *   s        = sigmoid(sum_h shexp_gate_w[h] x_t[h])
 *   FFN(x)   = down( silu(gate x) * (up x) ),  silu(z) = z / (1 + exp(-z))
 *   out_t    = sum_{j=0..top_k-1} p_j FFN_{ids_j}(x_t)  +  s FFN_shared(x_t)
 * The routed sum runs in rank order and the shared term is added last.  GPU
 * results are bitwise reproducible run to run (no floating-point atomics).
 *
 * The lifecycle follows the prepare / execute / destroy contract of the
 * "ggml operator extensions" page (stable-diffusion.cpp docs/ggml_extensions.md,
 * sections "Kernel selection" and "CUDA kernels can opt into device replay"):
 *   - prepare is host-only: it validates shapes, builds an immutable plan and
 *     reports the workspace size.  It launches nothing and allocates no
 *     device memory.
 *   - execute enqueues device work on the caller's stream only.  It makes no
 *     host decision based on tensor contents and never synchronises, so it
 *     can be captured in a CUDA graph and replayed.  Every counter and flag
 *     in the workspace is initialised by the recorded device work of each
 *     call; workspace contents are not preserved between calls.  An error is
 *     returned, never retried.
 *   - destroy frees the host plan only.
 *
 * Ownership: the caller owns every tensor and the workspace.  The library
 * keeps no pointer beyond a call.  One plan may be executed concurrently on
 * several streams when each call has its own workspace.
 *
 * All functions return MOE_FFN_OK (0) or a negative moe_ffn_status.
 */
#ifndef MOE_FFN_H
#define MOE_FFN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st* moe_ffn_stream_t;
/* Same type as cudaEvent_t. */
typedef struct CUevent_st* moe_ffn_event_t;

typedef enum {
  MOE_FFN_OK = 0,
  MOE_FFN_ERR_INVALID_ARG = -1, /* null required pointer, null plan, bad enum */
  MOE_FFN_ERR_UNSUPPORTED = -2, /* shapes or dtype outside the supported set (see moe_ffn_prepare) */
  MOE_FFN_ERR_WORKSPACE = -3,   /* workspace_bytes smaller than prepare reported */
  MOE_FFN_ERR_MISALIGNED = -4,  /* a pointer is not 16-byte aligned (workspace: 256-byte) */
  MOE_FFN_ERR_CUDA = -5,        /* a CUDA runtime call or launch failed */
  MOE_FFN_ERR_TIMEOUT = -6,     /* device status only: a bounded in-kernel wait gave up */
  MOE_FFN_ERR_DEVICE = -7       /* the current device is not sm_103 (GB300) or lacks a needed feature */
} moe_ffn_status;

/* T tokens, hidden size H, E experts, top_k kept per token, expert
 * intermediate size I, shared-expert intermediate size Is. */
typedef struct {
  int32_t T, H, E, top_k, I, Is;
} moe_ffn_shapes;

typedef enum { MOE_FFN_ACT_F32 = 0, MOE_FFN_ACT_BF16 = 1 } moe_ffn_act_dtype;

/* Weight format of the routed experts and of the shared expert.  The router
 * and the shared-gate vector are bf16 in both formats. */
typedef enum {
  MOE_FFN_W_BF16 = 0,
  /* 4-bit blocks of 32 along each stored row (H elements for every matrix,
   * see expert_w): one fp16 scale d per block and 4-bit codes n in 0..15
   * with weight = d * (n - 8).
   * Row layout: C/2 bytes of codes (element 2j in the low nibble of byte j,
   * element 2j+1 in the high nibble), then C/32 little-endian fp16 scales;
   * 9*C/16 bytes per row of C elements. */
  MOE_FFN_W_Q4B32 = 1,
  /* int8 rows with one fp32 scale per stored row (the int8 linear,
   * sd.linear_i8.v1, of "ggml operator extensions", section "sd.cpp
   * integration"): weight = s * q, q in -127..127.  Row layout: C int8 codes, the
   * little-endian fp32 scale s, 12 zero bytes; C + 16 bytes per row of C
   * elements.  The activation is quantised per token to int8 in fp32
   * (x_scale = max|x| / 127, q = round-half-away(x / x_scale) clamped to
   * +-127; x_scale = 0 gives q = 0), the gate and up projections are exact
   * int32 dot products, g = float(int32_dot) * x_scale * s in fp32 in that
   * order (likewise u), then SwiGLU; the down projection takes the
   * dequantised rows s * q of the transposed down matrix.  Decode path only
   * (T <= 8), H a multiple of 16. */
  MOE_FFN_W_I8 = 2
} moe_ffn_weight_format;

typedef struct {
  int32_t act;  /* moe_ffn_act_dtype: dtype of x */
  int32_t wfmt; /* moe_ffn_weight_format */
} moe_ffn_dtype;

typedef struct moe_ffn_plan* moe_ffn_plan_t;

/*
 * Validate `shapes` and `dtype`, build a plan and report the workspace size.
 * Host only: no device call, no launch, no device allocation.
 * Supported:
 *   decode path, 1 <= T <= 8: 1 <= E <= 1024, 1 <= top_k <= min(E, 32),
 *     H <= 4096 and a multiple of 8 (bf16 weights), of 256 (4-bit
 *     weights) or of 16 (int8 weights), I, Is >= 1; x fp32 or bf16;
 *   batched path, 9 <= T <= 1024 (routing, expert-sorted gather, grouped
 *     GEMMs on the tcgen05 tensor cores, fixed-order combine): bf16 or 4-bit
 *     weights and bf16 x, E <= 256, top_k <= 32, H a multiple of 256, I and
 *     Is multiples of 128.  With 4-bit weights the GEMM operands are fp16:
 *     each weight is d (code - 8) rounded once to fp16, x and the SwiGLU
 *     output h are carried in fp16 (accumulation fp32), so x and h must lie
 *     within fp16's range (|v| < 65504); the decode path keeps the exact
 *     weights.
 * moe_ffn_query(MOE_FFN_QUERY_PATH) reports the path taken.
 * Returns MOE_FFN_ERR_UNSUPPORTED otherwise, MOE_FFN_ERR_INVALID_ARG for null
 * pointers.  On success *plan is owned by the caller (moe_ffn_destroy).
 */
int moe_ffn_prepare(const moe_ffn_shapes* shapes, moe_ffn_dtype dtype, moe_ffn_plan_t* plan,
                    size_t* workspace_bytes);

/*
 * Enqueue the layer on `stream` (the current device must be a GB300).
 * Device pointers, all caller-owned:
 *   workspace     >= workspace_bytes from prepare, 256-byte aligned, scratch
 *   x             [T,H] fp32 or bf16 (plan dtype), row-major
 *   router_w      bf16 [E,H]
 *   expert_w      E consecutive blocks, block e = gate[I,H] | up[I,H] | downT[I,H]
 *                 in the plan's weight format, each matrix row-major with
 *                 H-element rows: gate and up are [out,in]; downT is the down
 *                 projection stored transposed (row i holds the weights from
 *                 intermediate unit i to all H outputs)
 *                 A caller holding the usual down[H,I] matrix passes its
 *                 transpose; with 4-bit weights it quantises that transpose
 *                 row by row, so down's blocks of 32 run along H.
 *   shexp_w       gate[Is,H] | up[Is,H] | downT[Is,H]
 *   shexp_gate_w  bf16 [H]
 *   out           fp32 [T,H]; may alias x exactly (the layer reads all of x
 *                 before it writes out); any other overlap is undefined.
 * Every pointer must be 16-byte aligned.  Returns without synchronising.
 */
int moe_ffn_execute(moe_ffn_plan_t plan, moe_ffn_stream_t stream, void* workspace, size_t workspace_bytes,
                    const void* x, const void* router_w, const void* expert_w, const void* shexp_w,
                    const void* shexp_gate_w, float* out);

/*
 * moe_ffn_execute, and also write the routing: topk_ids int32 [T,top_k] and
 * topk_w fp32 [T,top_k] in rank order (either may be NULL).
 */
int moe_ffn_execute_ex(moe_ffn_plan_t plan, moe_ffn_stream_t stream, void* workspace, size_t workspace_bytes,
                       const void* x, const void* router_w, const void* expert_w, const void* shexp_w,
                       const void* shexp_gate_w, float* out, int32_t* topk_ids, float* topk_w);

/*
 * Pre-norm transformer-block form (one layer of a decode stack):
 *   xn = bf16( x_res / sqrt(mean(x_res^2) + eps) )      (RMSNorm, weight 1)
 *   x_res <- x_res + layer(xn)
 * with the layer output and the residual add rounded to fp32 separately.
 * x_res is fp32 [T,H], read and updated in place.  The plan must have been
 * prepared with act = MOE_FFN_ACT_BF16 (the layer sees the bf16 xn) and
 * T <= 8.  topk_ids / topk_w as in moe_ffn_execute_ex (may be NULL).  Other
 * arguments as moe_ffn_execute; eps >= 0 or MOE_FFN_ERR_INVALID_ARG.
 */
int moe_ffn_execute_block(moe_ffn_plan_t plan, moe_ffn_stream_t stream, void* workspace, size_t workspace_bytes,
                          float* x_res, const void* router_w, const void* expert_w, const void* shexp_w,
                          const void* shexp_gate_w, float eps, int32_t* topk_ids, float* topk_w);

/*
 * Test/debug: synchronise `stream`, then copy the device status word of the
 * last execute that used `workspace` (MOE_FFN_OK or MOE_FFN_ERR_TIMEOUT) to
 * *device_status.  Returns a host-side status.
 */
int moe_ffn_read_status(moe_ffn_plan_t plan, const void* workspace, moe_ffn_stream_t stream,
                        int32_t* device_status);

/*
 * Test/debug: synchronise `stream`, then copy the token -> expert bucketing
 * of the last execute that used `workspace` to host arrays:
 *   counts [E]      tokens routed to each expert
 *   offsets [E+1]   exclusive prefix sum of counts
 *   perm [T*top_k]  flat (t*top_k + j) indices grouped by ascending expert,
 *                   token-major inside a group (a stable counting sort)
 *   active [E]      experts with counts > 0, ascending; *num_active of them
 */
int moe_ffn_read_routing(moe_ffn_plan_t plan, const void* workspace, moe_ffn_stream_t stream, int32_t* counts,
                         int32_t* offsets, int32_t* perm, int32_t* active, int32_t* num_active);

/*
 * Allocation-free variant of moe_ffn_execute, for callers that cannot
 * allocate device memory: for example a library embedded in a runtime that
 * has already handed all free device memory to its own pool (an inference
 * server that reserves the memory for its caches at start-up), or a plugin
 * given no allocator and no workspace.  This entry point has no counterpart
 * on the pages the layer is built from; it is an addition of this library.
 *
 * The scratch lives in one file-scope __device__ array of
 * MOE_FFN_STATIC_SCRATCH_BYTES bytes inside the library, which every GPU that
 * loads the library holds until the process exits.  The caller still passes
 * inputs and output exactly as for moe_ffn_execute.  Plans whose workspace is
 * larger than the array are rejected with MOE_FFN_ERR_WORKSPACE (the decode
 * shapes of one token batch, e.g. T <= 8, H = 2048, E = 128, top_k = 8,
 * I = 768, fit).  No cudaMalloc, cudaFree or other allocating call is made.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it; make that
 * first call before any stream capture.  Every call on a device shares the
 * one array and the kernels re-initialise what they read in each call, but
 * calls whose work overlaps on the GPU (other streams, or graphs replayed
 * concurrently) race on the array and give undefined results: serialise them.
 */
#define MOE_FFN_STATIC_SCRATCH_BYTES (1 << 24)
int moe_ffn_execute_static_scratch(moe_ffn_plan_t plan, moe_ffn_stream_t stream, const void* x, const void* router_w,
                                   const void* expert_w, const void* shexp_w, const void* shexp_gate_w, float* out);

/*
 * Test: the in-kernel failure path, without a fault.  Enqueues on `stream` one
 * small kernel that waits, with the bounded waits the layer's kernels use, on
 * a condition that nothing ever satisfies: which = 0 an mbarrier phase that
 * never completes (the wait of a shared-memory copy that never lands), which
 * = 1 a workspace flag that never receives the value waited for (the decode
 * kernel's grid-wide barriers), which = 2 a tagged workspace word that never
 * carries the tag waited for (the decode kernel's poll of the partial
 * outputs, T = 1).  The wait gives up after its iteration cap, records
 * MOE_FFN_ERR_TIMEOUT in the workspace status word (read it with
 * moe_ffn_read_status) and the kernel returns; the CUDA context stays usable
 * and the next execute on the workspace clears the word.  Returns a host-side
 * status (MOE_FFN_ERR_INVALID_ARG for a bad `which` or null pointers,
 * MOE_FFN_ERR_WORKSPACE if workspace_bytes is below the plan's size).
 */
int moe_ffn_probe_timeout(moe_ffn_plan_t plan, moe_ffn_stream_t stream, void* workspace, size_t workspace_bytes,
                          int32_t which);

/*
 * The layer in the form of "ggml-cuda: overlap the MoE shared expert on a
 * separate stream" (ROCm/llama.cpp PR #36, "What this changes"): the routed
 * branch (router, top-k, routed experts: ffn_moe_out) runs on `stream`, the
 * gated shared expert (ffn_shexp) on `aux_stream`, forked after everything
 * enqueued on `stream` before this call (fork_event recorded on `stream`,
 * waited by `aux_stream`) and joined back (join_event recorded on
 * `aux_stream`, waited by `stream`); then out = ffn_moe_out + ffn_shexp on
 * `stream`, the add of the page's diamond.  Decode plans (T <= 8) only, like
 * the page's batch gate; MOE_FFN_ERR_UNSUPPORTED otherwise.  The two
 * branches split the SMs in proportion to the bytes they stream.  When
 * aux_stream equals `stream` or an event is NULL, the same kernels run one
 * after the other on `stream` (the sequential form); both forms give
 * bit-identical results.  The fused moe_ffn_execute overlaps the shared
 * expert inside one kernel instead; its results agree with these within
 * the layer's tolerance (the sums are formed in another order).
 * Arguments as moe_ffn_execute, except that the workspace must hold
 * moe_ffn_query(MOE_FFN_QUERY_TWO_STREAM_WORKSPACE) bytes.  The events are
 * caller-owned (cudaEventCreateWithFlags with cudaEventDisableTiming is
 * enough); the call records and waits on them and keeps no reference.
 */
int moe_ffn_execute_two_stream(moe_ffn_plan_t plan, moe_ffn_stream_t stream, moe_ffn_stream_t aux_stream,
                               moe_ffn_event_t fork_event, moe_ffn_event_t join_event, void* workspace,
                               size_t workspace_bytes, const void* x, const void* router_w, const void* expert_w,
                               const void* shexp_w, const void* shexp_gate_w, float* out);

/* Queries on a plan. */
typedef enum {
  MOE_FFN_QUERY_PATH = 0,                 /* 0 = decode, 1 = grouped GEMM */
  MOE_FFN_QUERY_LAUNCHES_PER_EXECUTE = 1, /* kernels one execute launches */
  MOE_FFN_QUERY_TWO_STREAM_WORKSPACE = 2  /* workspace bytes of moe_ffn_execute_two_stream (decode plans) */
} moe_ffn_query_t;
int moe_ffn_query(moe_ffn_plan_t plan, int32_t what, int64_t* value);

/* Free a plan (host memory only).  NULL is ignored. */
void moe_ffn_destroy(moe_ffn_plan_t plan);

/* Static text for a status code. */
const char* moe_ffn_strerror(int status);

/* Text of the CUDA runtime error behind the last MOE_FFN_ERR_CUDA returned to
 * the calling host thread ("" if none).  The pointer stays valid until that
 * thread's next call into the library. */
const char* moe_ffn_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FFN_H */
