/*
 * wsf.h — C ABI of libwsfwd: forward and backward (vector-Jacobian product)
 * kernels of memory-bound row operators on one GPU (sm_103a).
 *
 *   weighted sum   y[i] = Σ_d x[i,d]·w[d]           x [N,D], w [D], y [N]
 *   scaled SiLU    y    = w·x·sigmoid(x)            x [n], scalar w
 *   row softmax, RMSNorm and LayerNorm over the rows of x [N,D]
 *
 * Sources (web pages, cited by title and section):
 *   [WS]   "Writing Triton Kernels with Autograd: A Minimal End-to-End
 *          Example": §1 Problem Setup, §2 Triton Forward Kernel, §3 Backward:
 *          Deriving Gradients First, §4 Triton Backward Kernel, §5 Wrapping
 *          with torch.autograd.Function.
 *   [SILU] "Backward in Triton — autograd.Function and the backward grid":
 *          § A complete minimal example — fused scaled-SiLU; § The backward
 *          grid is not the forward grid; § fp32 accumulation, and why
 *          gradients use +=.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.  Every pointer argument is DEVICE memory owned by the caller.  The
 * library allocates nothing, keeps no state between calls, and never frees
 * caller memory.  A pointer may be NULL only when the buffer it addresses
 * has no elements.  Outputs must not overlap any input or each other
 * (checked on the host; WSF_ERR_OVERLAP).
 *
 * Types.  `dtype` is the storage type of x, dy, y and dx: WSF_F32, WSF_F16
 * (IEEE binary16) or WSF_BF16 (bfloat16).  w, grad_w and dw are always
 * binary32.  All arithmetic is binary32 (16-bit inputs are widened exactly);
 * each 16-bit output is rounded once, to nearest-even.
 *
 * Layout.  x and dx are row-major with unit inner stride; row i starts at
 * element i·ld (ld >= D).  Any alignment of the element type is accepted:
 * 16-byte-aligned pointers and strides take 128-bit vector paths, others a
 * scalar path.
 *
 * Streams and errors.  Work is enqueued on `stream` (a cudaStream_t; NULL is
 * the legacy default stream) and the call returns without waiting.
 * Arguments are validated on the host before anything is enqueued; a
 * rejected call enqueues nothing and returns a negative status.  A launch
 * failure reported by the CUDA runtime returns WSF_ERR_CUDA.  Faults inside
 * a kernel surface at the caller's next synchronisation.  No entry point
 * throws or aborts.
 *
 * Determinism.  The parameter gradients (grad_w, dw) are reduced in two
 * stages — per-tile partial sums into the caller's workspace, then a sum
 * over tiles in a fixed order — with no atomic operations, so repeating a
 * call with the same arguments gives the same bits.  The tiling depends only
 * on the sizes, the storage type and block_n, never on the device.
 */
#ifndef WSF_H
#define WSF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* wsf_stream_t;

/* storage types */
#define WSF_F32 0
#define WSF_F16 1
#define WSF_BF16 2

/* status codes */
#define WSF_OK 0
#define WSF_ERR_NULL_PTR (-1)   /* a required pointer is NULL */
#define WSF_ERR_BAD_SHAPE (-2)  /* negative extent, or a size that overflows int64 */
#define WSF_ERR_BAD_DTYPE (-3)  /* dtype is not WSF_F32 / WSF_F16 / WSF_BF16 */
#define WSF_ERR_BAD_STRIDE (-4) /* a row stride smaller than D */
#define WSF_ERR_WORKSPACE (-5)  /* workspace NULL or smaller than the query says */
#define WSF_ERR_OVERLAP (-6)    /* an output overlaps an input or another output */
#define WSF_ERR_MISALIGNED (-7) /* a pointer not aligned to its element type */
#define WSF_ERR_BAD_ARG (-8)    /* another invalid argument (block_n < 0, accumulate not 0/1) */
#define WSF_ERR_CUDA (-9)       /* the CUDA runtime rejected a launch */

/* Human-readable text for a status code (static storage, never NULL). */
const char* wsf_status_string(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int wsf_version(void);

/*
 * wsf_cluster_wait_timeouts — health counter of the cluster paths.
 * Rows too wide for one CTA (softmax rows of more than 2048 16-byte chunks,
 * RMSNorm/LayerNorm rows of 8193..65536 elements) are split over a
 * thread-block cluster whose CTAs exchange their partial row sums through
 * distributed shared memory.  Each wait for the
 * other CTAs' sums gives up after about a second; the launch then finishes
 * with invalid results and adds one to this counter per thread that gave up,
 * instead of hanging the GPU.  The counter is zero in correct operation.
 * count: host pointer receiving the value for the current device.  reset = 1
 * zeroes it after reading.  Synchronises the current device.
 * Returns WSF_OK, WSF_ERR_NULL_PTR or WSF_ERR_CUDA.
 */
int wsf_cluster_wait_timeouts(unsigned* count, int reset);

/*
 * wsf_selftest_exchange_timeout — runs the bounded wait of the cluster
 * exchange where nothing completes it: one cluster of two CTAs posts the
 * bytes an exchange turn expects and waits, but no CTA pushes any.  Every
 * waiting warp gives up after limit_ms milliseconds and adds one to *count;
 * the kernel then returns and the context stays usable.  count: device
 * memory, one unsigned (4-byte aligned), owned by the caller, added to (zero
 * it first); after the stream completes it holds wsf_selftest_waiting_warps()
 * more than before.  limit_ms: 1..1000.  The counter that
 * wsf_cluster_wait_timeouts reads is not touched.  Stream-ordered.
 * Returns WSF_OK, WSF_ERR_NULL_PTR, WSF_ERR_MISALIGNED, WSF_ERR_BAD_ARG or
 * WSF_ERR_CUDA.
 */
int wsf_selftest_exchange_timeout(unsigned* count, unsigned limit_ms, wsf_stream_t stream);

/* Number of warps that wait in wsf_selftest_exchange_timeout (one timeout each). */
int wsf_selftest_waiting_warps(void);

/*
 * ws_fwd — weighted-sum forward  [WS §1, §2]
 *   y[i] = Σ_{d<D} x[i,d] · w[d]   for 0 <= i < N
 * x: [N, D] dtype, row stride ldx; w: [D] binary32; y: [N] dtype.
 * Products and the sum are binary32; y is rounded once to dtype.  D == 0
 * writes y = 0; N == 0 does nothing.
 */
int ws_fwd(const void* x, int64_t ldx, const float* w, void* y, int64_t N, int64_t D, int dtype,
           wsf_stream_t stream);

/*
 * ws_bwd_workspace_bytes — size in bytes of the partial buffer that ws_bwd
 * needs for these sizes: two binary32 planes (high and low parts of the
 * compensated partial sums) of P·D values, each rounded up to 256 bytes,
 * where P is the number of row tiles.  block_n > 0 forces tiles of block_n consecutive rows
 * (P = ceil(N / block_n)), as in [WS §3]'s BLOCK_N; block_n == 0 lets the
 * library choose.  Returns 0 when no workspace is needed, and SIZE_MAX for
 * invalid arguments.  Host-only; touches no device.
 */
size_t ws_bwd_workspace_bytes(int64_t N, int64_t D, int dtype, int64_t block_n);

/*
 * ws_bwd — weighted-sum backward  [WS §3, §4]
 *   dx[i,d]   = dy[i] · w[d]                       (elementwise, written)
 *   grad_w[d] = Σ_{i<N} x[i,d] · dy[i]             (reduction over rows)
 * Inputs: x [N, D] dtype (row stride ldx), w [D] binary32, dy [N] dtype.
 * Outputs: dx [N, D] dtype (row stride lddx), grad_w [D] binary32.
 * Stage 1 writes dx and, for each row tile p, partial[p, d] = Σ over the
 * tile's rows of x[i,d]·dy[i] into `workspace` as a compensated binary32
 * pair (high and low planes, [P, D] each).  Stage 2 sums partial[0..P-1, d]
 * in a fixed order, again as a pair, and rounds it once: grad_w is as
 * accurate as a sum in twice binary32's precision.  With accumulate == 1 the
 * result is added to the existing grad_w[d] (old + sum, one binary32 add),
 * with accumulate == 0 it replaces it ([SILU] § fp32 accumulation ...: a
 * gradient accumulates with += across micro-batches).  N == 0 gives
 * grad_w = 0 (or leaves it when accumulating).  The workspace contents are
 * scratch: nothing needs to be initialised and nothing is kept.
 */
int ws_bwd(const void* x, int64_t ldx, const float* w, const void* dy, void* dx, int64_t lddx,
           float* grad_w, int accumulate, void* workspace, size_t workspace_bytes,
           int64_t block_n, int64_t N, int64_t D, int dtype, wsf_stream_t stream);

/*
 * ws_bwd_noalloc — ws_bwd for callers that cannot allocate device memory.
 * The pages have no counterpart of this entry point; it exists for callers
 * that are handed only their input and output buffers, such as a plugin in a
 * host program that owns all device memory through its own pool, or a
 * latency-critical loop that cannot afford cudaMalloc's implicit device-wide
 * synchronisation.  Same arguments, results and errors as ws_bwd, minus the
 * workspace: the per-tile partials go to a scratch array of
 * WSF_NOALLOC_SCRATCH_BYTES (8 MiB) that lives in the library's own device
 * memory, one copy per device that loads the library, held until the
 * process exits.  The call allocates nothing.
 *   - Sizes whose ws_bwd_workspace_bytes(N, D, dtype, block_n) exceeds
 *     WSF_NOALLOC_SCRATCH_BYTES are rejected with WSF_ERR_WORKSPACE before
 *     anything is enqueued (the five benchmark workloads need at most 7.2 MiB).
 *   - The first call on a device looks up that device's copy of the array
 *     (cudaGetSymbolAddress, with the device current); make that first call
 *     before any stream capture.
 *   - Every call shares the array and it keeps the last call's contents;
 *     nothing in it needs clearing, but calls whose kernels overlap on the
 *     GPU (e.g. issued on two streams) race on it: serialise them.
 */
#define WSF_NOALLOC_SCRATCH_BYTES (8u << 20)
int ws_bwd_noalloc(const void* x, int64_t ldx, const float* w, const void* dy, void* dx,
                   int64_t lddx, float* grad_w, int accumulate, int64_t block_n, int64_t N,
                   int64_t D, int dtype, wsf_stream_t stream);

/*
 * silu_fwd — scaled-SiLU forward  [SILU, forward kernel]
 *   s = 1 / (1 + exp(-x)),  y = w · x · s       elementwise over n elements
 * x, y: [n] dtype (contiguous); w: one binary32 value in device memory.
 */
int silu_fwd(const void* x, const float* w, void* y, int64_t n, int dtype, wsf_stream_t stream);

/*
 * silu_bwd_workspace_bytes — bytes of the per-block partial buffer for
 * silu_bwd (two binary32 planes of P values, high and low parts, each rounded
 * up to 256 bytes); 0 when none is needed, SIZE_MAX for invalid arguments.
 * Host-only.
 */
size_t silu_bwd_workspace_bytes(int64_t n, int dtype);

/*
 * silu_bwd — scaled-SiLU backward  [SILU, backward kernel; § The backward
 * grid is not the forward grid]
 *   dx = dy · w · (s + x·s·(1 - s))             elementwise (written)
 *   dw = Σ_k dy_k · x_k · s_k                    scalar reduction over all n
 * s is recomputed from x (nothing from the forward is needed but x and w).
 * Stage 1 writes dx and one compensated binary32 pair, the partial of dw, per
 * block into `workspace`; stage 2 reduces the pairs in a fixed tree order,
 * rounds once and writes *dw (added to the existing value when
 * accumulate == 1).  n == 0 gives dw = 0
 * (or leaves it when accumulating).
 */
int silu_bwd(const void* dy, const void* x, const float* w, void* dx, float* dw, int accumulate,
             void* workspace, size_t workspace_bytes, int64_t n, int dtype, wsf_stream_t stream);

/*
 * softmax_fwd / softmax_bwd — row softmax and its vector-Jacobian product
 * ["Backprop for kernel writers", §04 The duality: the backward collapses the
 * dense Jacobian diag(y) − y·yᵀ to one row scalar and needs the output y, not
 * x; the forward's max shift contributes nothing to it]:
 *   y[i,j]  = exp(x[i,j] − m_i) / Σ_k exp(x[i,k] − m_i),  m_i = max_k x[i,k]
 *   dx[i,j] = y[i,j] · (dy[i,j] − s_i),   s_i = Σ_k dy[i,k]·y[i,k]
 * x, y, dy, dx: [N, D] in dtype, row strides ldx, ldy, lddy, lddx (>= D).
 * fp32 arithmetic (for binary32 storage the row sums are compensated and
 * x − max is split exactly before the exponential), each output rounded once.
 * Rows of up to 32 KB are read once and written once; wider or unaligned rows
 * read their inputs two or three times.  N == 0 or D == 0 does nothing.
 * Errors as for ws_fwd.
 */
int softmax_fwd(const void* x, int64_t ldx, void* y, int64_t ldy, int64_t N, int64_t D, int dtype,
                wsf_stream_t stream);
int softmax_bwd(const void* y, int64_t ldy, const void* dy, int64_t lddy, void* dx, int64_t lddx,
                int64_t N, int64_t D, int dtype, wsf_stream_t stream);

/*
 * Atomic comparison variants  [SILU, backward kernel: per-block sums added
 * into one fp32 cell with an atomic add; § The backward grid is not the
 * forward grid: "atomics (small, non-critical)" versus the two-pass partials
 * buffer; VJP §02 The kernel consequence: "atomicAdd, split-K, or a separate
 * reduction pass"; §06: atomic adds are nondeterministic by default].
 *
 * Same results as ws_bwd / silu_bwd up to fp32 rounding, but the parameter
 * gradient is summed with atomic additions in whatever order the blocks
 * finish, so its bits may differ from run to run; they exist to measure what
 * the deterministic two-pass form costs.  No workspace: grad_w / dw is
 * zeroed first (unless accumulate == 1) and every row tile adds its partial
 * into it.  ws_bwd_atomic supports only the 16-byte-aligned layout of the
 * staged path (x, dx, w, dy, grad_w 16-byte aligned; D, ldx, lddx multiples
 * of 16 bytes) and returns WSF_ERR_MISALIGNED otherwise.  Other arguments and
 * errors as for ws_bwd / silu_bwd.
 */
int ws_bwd_atomic(const void* x, int64_t ldx, const float* w, const void* dy, void* dx,
                  int64_t lddx, float* grad_w, int accumulate, int64_t N, int64_t D, int dtype,
                  wsf_stream_t stream);
int silu_bwd_atomic(const void* dy, const void* x, const float* w, void* dx, float* dw,
                    int accumulate, int64_t n, int dtype, wsf_stream_t stream);

/*
 * RMSNorm and LayerNorm over the rows of x, forward and vector-Jacobian
 * product  ["Backward in Triton — autograd.Function and the backward grid",
 * § Save vs recompute (the row statistic rstd is recomputed from x in the
 * backward rather than stored) and § The backward grid is not the forward
 * grid (RMSNorm's dw sums a length-D partial from every row: a map for dx and
 * a separate reduce, the two-pass partials buffer being the deterministic
 * choice); "Backprop for kernel writers", §04 (LayerNorm's backward collapses
 * to two row scalars plus the batch-axis reductions of its parameters)].
 * The pages give no formulas; these are the standard definitions:
 *   RMSNorm:   r_i = 1/sqrt(mean_j x[i,j]² + eps),  x̂ = x·r_i,
 *              y = x̂·w,                dx = r_i·(g − x̂·mean_j(g·x̂))
 *   LayerNorm: μ_i = mean_j x[i,j],  r_i = 1/sqrt(mean_j (x[i,j]−μ_i)² + eps),
 *              x̂ = (x−μ_i)·r_i,  y = x̂·w + b,
 *              dx = r_i·(g − mean_j g − x̂·mean_j(g·x̂))
 *   with g = dy·w;  grad_w[j] = Σ_i dy[i,j]·x̂[i,j],  grad_b[j] = Σ_i dy[i,j].
 * x, dy, y, dx: [N, D] in dtype with row strides ldx, lddy, ldy, lddx (>= D);
 * w, b, grad_w, grad_b: [D] binary32.  eps: binary32, finite and >= 0
 * (WSF_ERR_BAD_ARG otherwise).  Nothing from the forward is needed by the
 * backward but x: the row statistics are recomputed.  All arithmetic is
 * binary32 (for binary32 storage the row sums are compensated); each output
 * is rounded once to dtype.  Rows of up to 8192 elements with 16-byte
 * aligned pointers and strides are read once and written once; other layouts
 * take a multi-pass element-wise path.
 * The backward writes dx and, per row tile p, the partial sums of dy·x̂ (and,
 * LayerNorm, dy) into `workspace` (binary32 [P, D], twice for LayerNorm);
 * then sums the tiles in a fixed order into grad_w (and grad_b), added to the
 * existing values when accumulate == 1.  N == 0 gives zero gradients (or
 * leaves them when accumulating); D == 0 does nothing.  The workspace size
 * comes from the *_workspace_bytes query (0 when none is needed, SIZE_MAX for
 * invalid sizes; host-only).  Other errors as for ws_bwd.
 */
int rmsnorm_fwd(const void* x, int64_t ldx, const float* w, float eps, void* y, int64_t ldy,
                int64_t N, int64_t D, int dtype, wsf_stream_t stream);
size_t rmsnorm_bwd_workspace_bytes(int64_t N, int64_t D, int dtype);
int rmsnorm_bwd(const void* x, int64_t ldx, const float* w, const void* dy, int64_t lddy,
                float eps, void* dx, int64_t lddx, float* grad_w, int accumulate, void* workspace,
                size_t workspace_bytes, int64_t N, int64_t D, int dtype, wsf_stream_t stream);
int layernorm_fwd(const void* x, int64_t ldx, const float* w, const float* b, float eps, void* y,
                  int64_t ldy, int64_t N, int64_t D, int dtype, wsf_stream_t stream);
size_t layernorm_bwd_workspace_bytes(int64_t N, int64_t D, int dtype);
int layernorm_bwd(const void* x, int64_t ldx, const float* w, const void* dy, int64_t lddy,
                  float eps, void* dx, int64_t lddx, float* grad_w, float* grad_b, int accumulate,
                  void* workspace, size_t workspace_bytes, int64_t N, int64_t D, int dtype,
                  wsf_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* WSF_H */
