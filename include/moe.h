/*
 * moe.h -- C ABI of the Mixtral sparse mixture-of-experts feed-forward layer
 *          on B300 (sm_103a).  Library: sparse_mixture_experts_54_b300/libmoe_b300.so
 *
 * The layer (Mixtral of Experts, section 2.1; restated in "从Mistral 7B到MoE模型
 * Mixtral 8x7B的全面解析" (aiqianji) section 2.1.1 and in the xyznot summary,
 * "Method"):
 *
 *     y = sum_{i=0}^{n-1} Softmax(TopK(x . W_g))_i * SwiGLU_i(x),
 *     SwiGLU_i(x) = W2_i ( SiLU(W1_i x) * (W3_i x) ),   SiLU(z) = z / (1 + e^-z)
 *
 * with TopK keeping the K largest router logits and setting the rest to -inf,
 * so only K experts per token are evaluated.  Mixtral: d = 4096, d_ff = 14336,
 * n = 8, K = 2.
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - Layouts are row-major, nn.Linear style ([out][in]), as in the router
 *    `nn.Linear(hidden_dim, num_experts, bias=False)` (aiqianji 2.1.4) and the
 *    expert's w1/w3/w2 linears (aiqianji 3.2.4, code block D):
 *        x   [T][d]            element type = context dtype
 *        W_g [n][d]            fp32 always
 *        W1  [n][d_ff][d]      element type = context dtype
 *        W3  [n][d_ff][d]
 *        W2  [n][d][d_ff]
 *        y   [T][d]            element type = context dtype
 *  - Pointers named "device" must point to device memory of the current CUDA
 *    device and be 16-byte aligned.  The caller owns every pointer and the
 *    stream; the library never frees caller memory.
 *  - All compute entry points are asynchronous on `stream` and do not
 *    synchronise the host.  Argument errors are returned synchronously
 *    (moe_status_t).  Failures inside kernels (a bounded wait that ran out, an
 *    index check of the routing and dispatch kernels that failed: an expert id
 *    outside [0, n) or a dispatch position outside [0, k*T), which is then
 *    never used as an address) are recorded in a sticky status word that
 *    moe_status() reads without synchronising.
 *  - Each forward call is one NVTX range on the calling host thread ("moe_forward"
 *    or "moe_forward_fp8") holding one nested range per stage, named as the
 *    stages of moe_stage_times; a profiler that records NVTX shows them.
 *  - A context must not be used from two host threads at once; calls on
 *    different streams with the same context share its workspace and must be
 *    ordered by the caller.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_ctx moe_ctx;
/* Same object as cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st* moe_stream_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID = -1,      /* bad argument (NULL pointer, T < 0, misaligned pointer, ...) */
    MOE_ERR_CUDA = -2,         /* a CUDA runtime call or kernel launch failed */
    MOE_ERR_OOM = -3,          /* workspace allocation failed */
    MOE_ERR_TIMEOUT = -4,      /* a kernel's bounded wait ran out (sticky, via moe_status) */
    MOE_ERR_UNSUPPORTED = -5,  /* shape/dtype the kernels cannot tile */
    MOE_ERR_BOUNDS = -6,       /* a kernel-side index check failed (sticky, via moe_status) */
    MOE_ERR_SCRATCH_LIMIT = -7 /* moe_forward_noalloc: the call needs more than its fixed scratch */
} moe_status_t;

typedef enum { MOE_BF16 = 0, MOE_F32 = 1 } moe_dtype_t;

/* Options for moe_set_option. */
typedef enum {
    MOE_OPT_DECODE_MAX_T = 1,  /* forward uses the weight-streaming decode kernels when T <= value (default 128) */
    MOE_OPT_WAIT_LIMIT_US = 2, /* wall-time limit of every bounded wait inside a kernel (default 2,000,000 us) */
    MOE_OPT_FORCE_PATH = 3,    /* 0 = choose by T, 1 = always grouped GEMM, 2 = always decode kernels */
    MOE_OPT_STAGE_TIMING = 4,  /* 1 = record CUDA events around every kernel of moe_forward (see moe_stage_times) */
    MOE_OPT_GEMM_PAIR = 5,     /* grouped GEMMs: 0 = default (both on CTA pairs -- tcgen05 cta_group::2,
                                  256/128-row tiles -- when the device can co-schedule them, else both on
                                  single CTAs with 128-row tiles), 1 = both single-CTA, 2 = both on CTA
                                  pairs or MOE_ERR_UNSUPPORTED */
    MOE_OPT_HOST_OUTPUT = 6,   /* moe_forward_host: 1 = when y_host is pinned, the layer's last kernel writes y
                                  into it directly over the bus (default; measured 0.19 ms faster per call at
                                  T=4096), 0 = always copy y back on the stream */
    MOE_OPT_FP8_WIDEN = 7,     /* moe_forward_fp8: 0 = e4m3 weights into the 8-bit MMA against split token rows
                                  (default), 1 = weights widened to bf16 on chip (bitwise equal to the bf16
                                  path with MOE_OPT_DECODE_STREAMK 0 on the dequantised weights; slower) */
    MOE_OPT_DECODE_STREAMK = 8 /* bf16 weight-streaming path, T >= 2: 1 = every CTA streams an equal,
                                  contiguous share of all touched experts' k-blocks (default), 0 = K split
                                  uniformly into items (always so at T = 1); the partial sums are grouped
                                  differently, so results differ in rounding */
} moe_option_t;

/*
 * Create a layer context for hidden size d, expert hidden size d_ff, n_experts
 * experts and top-k routing (Mixtral: 4096, 14336, 8, 2; the K/n trade-off is
 * aiqianji 2.1.1).  Requires 1 <= k <= n_experts <= 32, d % 8 == 0, d_ff >= 1.
 * Context dtype defaults to MOE_BF16.  Allocates only the host-mapped status
 * word; the workspace grows on first use (or moe_reserve).  Returns NULL on bad
 * arguments or when no CUDA device is usable.
 */
moe_ctx* moe_create(int d, int d_ff, int n_experts, int k);

/* Element type of x, W1, W3, W2 and y: MOE_BF16 (default) or MOE_F32.
 * bf16 additionally requires d % 256 == 0 and d_ff % 128 == 0 (tensor-core tiling);
 * MOE_F32 runs CUDA-core FMA kernels (no TF32) for any shape. */
int moe_set_dtype(moe_ctx* ctx, int dtype);

/* Optional router bias b_g [n] fp32, device pointer, added to the logits before
 * top-k and softmax; NULL removes it.  Mixtral's router has no bias
 * (aiqianji 2.1.4); this exists for skewed-load workloads.  The pointer is
 * kept, not copied: it must stay valid while the context uses it. */
int moe_set_router_bias(moe_ctx* ctx, const float* b_g);

int moe_set_option(moe_ctx* ctx, int option, long long value);

/* Grow the workspace now for up to T_max tokens (no allocation happens later
 * for T <= T_max, e.g. while a stream is being captured into a CUDA graph). */
int moe_reserve(moe_ctx* ctx, int T_max);

/* Device workspace bytes a call with T tokens needs. */
size_t moe_workspace_bytes(const moe_ctx* ctx, int T);

/*
 * Routing and dispatch only (router logits, top-k gate, expert-contiguous order).
 *   x [T][d] (device, context dtype), W_g [n][d] (device, fp32).
 * Outputs (device; each may be NULL):
 *   topk_idx [T][k] int32   experts by descending logit, equal logits -> lower index first
 *   topk_w   [T][k] fp32    Softmax over the kept logits (aiqianji 2.1.1; equal to the
 *                           renormalised top-k of the full softmax, aiqianji 3.1.1 steps 4-6)
 *   counts   [n]    int32   assignments per expert
 *   offsets  [n+1]  int32   exclusive scan of counts, offsets[n] = k*T
 *   perm     [k*T]  int32   flat assignment number t*k+slot at each expert-contiguous
 *                           position; stable (ascending t*k+slot within an expert), which
 *                           lists each expert's tokens as the one_hot/where walk of
 *                           aiqianji 3.1.2 and code blocks B/C does.
 * T == 0 is valid and writes nothing but counts/offsets (all zero).
 */
int moe_route(moe_ctx* ctx, const void* x, const float* W_g, int T,
              int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
              int32_t* perm, moe_stream_t stream);

/* Router logits only: logits [T][n] fp32 (device) = x . W_g^T (+ bias), with the
 * same fp32 arithmetic moe_route and moe_forward use. */
int moe_router_logits(moe_ctx* ctx, const void* x, const float* W_g, int T, float* logits,
                      moe_stream_t stream);

/*
 * The whole layer: y [T][d] = MoE(x).  All pointers device.  Steps (all CUDA
 * kernels): router + top-k gate; dispatch (histogram, scan, stable scatter,
 * row gather); expert W1/W3 GEMM with the SiLU(a)*b product fused; expert W2
 * GEMM with the gate weight applied to each row (the gate multiplies the W2
 * output inside the expert, aiqianji 3.2.4 code block D); and a combine that
 * adds each token's k expert rows in slot order (replacing index_add_,
 * aiqianji 3.1.2) with no atomics, so results are bitwise reproducible.
 * bf16: fp32 accumulation, the SwiGLU product rounded once to bf16, y rounded
 * once.  Small T (<= MOE_OPT_DECODE_MAX_T) uses weight-streaming kernels.
 * x and y must not overlap.  T == 0 is a no-op.
 */
int moe_forward(moe_ctx* ctx, const void* x, const float* W_g, const void* W1, const void* W3,
                const void* W2, void* y, int T, moe_stream_t stream);

/*
 * moe_forward with x and y in host memory (pinned memory gives asynchronous
 * copies; pageable memory works but the copies then synchronise).  Copies x
 * to one of two context-owned device buffers on a stream of the context's own
 * (so that, with pinned memory, the copy overlaps the previous call's
 * kernels), runs the layer on `stream` once the copy is done, and -- when
 * y_host is pinned -- lets the layer's last kernel write y straight into it
 * (else y is copied back on `stream`; see MOE_OPT_HOST_OUTPUT).  Weights stay
 * device pointers.  When `stream` reaches this
 * point, y_host holds the result; x_host must stay valid and unchanged until
 * then.  While `stream` is being captured into a graph, all of it runs on
 * `stream`.
 */
int moe_forward_host(moe_ctx* ctx, const void* x_host, const float* W_g, const void* W1,
                     const void* W3, const void* W2, void* y_host, int T, moe_stream_t stream);

/*
 * One residual block of a layer stack, in place:
 *     h <- h + MoE(RMSNorm(h)),   RMSNorm(h) = h / sqrt(mean_j h_j^2 + eps)  (unit gain)
 * The pages' block diagram has, per layer, RMSNorm -> attention -> RMSNorm ->
 * MoE with residual connections (the DL reading-group slides, "Architecture -
 * 全体"; 32 layers, xyznot "Method"); this is the MoE half of it (attention
 * is outside this library).  h [T][d] (device, context dtype) is read and
 * overwritten.  The normalised row is rounded to the element type once and
 * feeds both the router and the experts; h + MoE(...) is summed in fp32 and
 * rounded once.  eps >= 0 (Mixtral-style models use 1e-5).  Other arguments,
 * errors and asynchrony as moe_forward.
 */
int moe_block_forward(moe_ctx* ctx, void* h, float eps, const float* W_g, const void* W1,
                      const void* W3, const void* W2, int T, moe_stream_t stream);

/*
 * n_layers residual blocks in order (layer l uses W_g[l], W1[l], W3[l], W2[l]):
 * for l in 0..n_layers-1: h <- h + MoE_l(RMSNorm(h)).  The four arguments are
 * host arrays of n_layers device pointers (each layout as moe_forward).  The
 * context's router bias, if set, applies to every layer.  Launches 3 kernels
 * per layer for T above the decode threshold (5 at or below it); nothing is
 * synchronised.  Returns the first error; the layers before it have run.
 */
int moe_stack_forward(moe_ctx* ctx, void* h, float eps, int n_layers, const float* const* W_g,
                      const void* const* W1, const void* const* W3, const void* const* W2, int T,
                      moe_stream_t stream);

/*
 * moe_forward with fp8 expert weights, for decode-sized batches: y [T][d] =
 * MoE(x) with
 *     W1_i[f][j] = W1_scale[i][f] * W1q[i][f][j]     (same for W3; W2 per d row)
 * where W1q, W3q, W2q hold OCP e4m3 bytes (1 sign, 4 exponent bits with bias
 * 7, 3 mantissa bits; 0x7F/0xFF (NaN) are not accepted and give unspecified
 * results) in the layouts of W1, W3, W2 above, and the scales are fp32, one
 * per weight row: W1_scale, W3_scale [n][d_ff], W2_scale [n][d].  Fp8 weights
 * are not part of the method as the pages give it; they halve the bytes a
 * weight-streaming layer reads (the layer's decode time is the time to read
 * the touched experts' weights).
 *
 * Computation: the weight-streaming kernels of moe_forward's small-T path with
 * the row scale applied to the fp32 accumulator, in one of two ways
 * (MOE_OPT_FP8_WIDEN):
 *  - 0 (default): the weight bytes go straight into the 8-bit tensor-core MMA.
 *    Each bf16 token row v (the gathered input rows for W1/W3, the SwiGLU rows
 *    for W2) is first written as two e4m3 rows hi, lo with s*v = hi + lo for
 *    a power-of-two s per row that maps max|v| into (224, 448]; this is exact
 *    for every element with |s*v| >= 1/4 and rounds the bits below 2^-9/s of
 *    the smaller ones.  The tensor core sums the exact e4m3 products in fp32.
 *    The result agrees with moe_forward on the bf16 weights scale * q to
 *    within the layer's bf16 tolerance, not bitwise.
 *  - 1: the weight tiles are widened exactly to bf16 on chip and multiplied by
 *    the bf16 token rows.  When every scale is a power of two (including 1)
 *    the result is bitwise identical to moe_forward on the bf16 weights
 *    scale * q (which are exact in bf16); other scales are exact to the fp32
 *    rounding of one product per partial sum.  Slower: the widening runs on
 *    the integer pipes.
 *
 * Requirements: bf16 context; d a multiple of 256 and d_ff of 128 (as
 * moe_forward's bf16 path); n <= 31.  x, y, W_g device as moe_forward; W1q,
 * W3q, W2q device, 16-byte aligned; the scales device, 4-byte aligned.
 * Batches of more than 256 tokens run as consecutive 256-token chunks on
 * `stream` (each chunk reads every touched expert's weights once).  Errors
 * and asynchrony as moe_forward; per-kernel times through moe_stage_times
 * with the same four stages.
 */
int moe_forward_fp8(moe_ctx* ctx, const void* x, const float* W_g, const uint8_t* W1q,
                    const float* W1_scale, const uint8_t* W3q, const float* W3_scale,
                    const uint8_t* W2q, const float* W2_scale, void* y, int T, moe_stream_t stream);

/* Sticky kernel-side status (MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_BOUNDS) of every
 * call so far; reads host-mapped memory, synchronises nothing.  Results written
 * by kernels still running are not yet visible. */
int moe_status(moe_ctx* ctx);
/* Reset the sticky status to MOE_OK. */
int moe_clear_status(moe_ctx* ctx);

/* Self-test of the bounded-wait machinery: launches one kernel whose wait can
 * never complete (nothing arrives on its barrier); it gives up after
 * wait_limit_us microseconds, records MOE_ERR_TIMEOUT and returns normally. */
int moe_selftest_wait_timeout(moe_ctx* ctx, long long wait_limit_us, moe_stream_t stream);

/*
 * Per-kernel device time of the moe_forward calls made since the last read,
 * while MOE_OPT_STAGE_TIMING is on.  Events are recorded on the call's stream
 * around each kernel, so they measure exactly the launches of that stream.
 * Synchronises on the last recorded event, writes the mean milliseconds per
 * call of each stage into ms[0..max_stages) (stage names: moe_stage_name) and
 * the number of calls into *calls, then forgets the recorded calls.  Returns
 * the number of stages (>= 0) or a negative moe_status_t.  Stages: "route",
 * "expert_w1w3_swiglu" (with the decode path's SwiGLU kernel), "expert_w2_gate"
 * and "combine" (zero-length on the grouped path, whose W2 epilogue combines).
 */
int moe_stage_times(moe_ctx* ctx, float* ms, int max_stages, int* calls);
/* Name of stage i of moe_stage_times, or NULL past the last stage. */
const char* moe_stage_name(int i);

/*
 * moe_forward_noalloc -- the same layer as moe_forward, for callers that
 * cannot call cudaMalloc: it allocates nothing, on the device or the host, and
 * needs no context (creating one allocates).  The pages have no counterpart to
 * this entry point; it exists for processes whose device memory is owned and
 * budgeted by another allocator, or that must not allocate once they are
 * serving.
 *
 *  - Scratch: one fixed 32 MiB __device__ array inside this library.  Every GPU
 *    that loads the library holds it until the process exits.  A call needs
 *    256-byte-rounded regions of 4*k*T bytes (four of them), (3n+2)*4 bytes,
 *    k*T*d*es, k*T*d_ff*es and k*T*d*4 bytes (es = 2 for bf16, 4 for fp32);
 *    if their sum exceeds 32 MiB it returns MOE_ERR_SCRATCH_LIMIT and launches
 *    nothing.  At the Mixtral shape (bf16, d=4096, d_ff=14336, k=2) that allows
 *    T <= 314.
 *  - Every call uses the same array, and each call overwrites the parts it
 *    uses before reading them (nothing has to start at zero).  Calls that can
 *    overlap on the GPU (different streams, different host threads, several
 *    layers in flight) race on it: order them on one stream.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and caches it; make that
 *    first call before any stream capture.  The cached address belongs to the
 *    device's primary context as it was then: after cudaDeviceReset (or any
 *    other teardown of that context) it is stale, so this entry point must not
 *    be used across a device reset.
 *  - Arguments: as moe_forward, plus the shape (d, d_ff, n_experts, k), the
 *    element type (moe_dtype_t) and an optional router bias b_g [n] (device,
 *    fp32, NULL for none).  status, if not NULL, is a caller-owned device int
 *    into which kernels OR their failure bits (1 = a bounded wait ran out,
 *    2 = an index check failed); bounded waits give up after 2 s.  Returns
 *    MOE_OK, MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_SCRATCH_LIMIT or
 *    MOE_ERR_CUDA; asynchronous like moe_forward.
 */
int moe_forward_noalloc(const void* x, const float* W_g, const float* b_g, const void* W1,
                        const void* W3, const void* W2, void* y, int T, int d, int d_ff,
                        int n_experts, int k, int dtype, int* status, moe_stream_t stream);

/* Human-readable name of a moe_status_t value. */
const char* moe_error_string(int code);

/* Release the context and its workspace.  NULL-safe.  The caller must have
 * synchronised every stream that used the context. */
void moe_destroy(moe_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif /* MOE_B300_H */
