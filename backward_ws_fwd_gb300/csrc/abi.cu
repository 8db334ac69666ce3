// abi.cu — the extern "C" entry points declared in include/wsf.h.
//
// Every entry point validates its arguments on the host, before anything is
// enqueued, and maps them to a launcher in ws.cu, silu.cu, softmax.cu or
// norm.cu.  Host-only work
// here never touches the device, so argument errors can be checked without
// a GPU.
#include <limits.h>
#include <stdint.h>

#include "wsf.h"
#include "wsf_internal.h"

namespace {

using wsf::elt_bytes;

bool valid_dtype(int dtype) { return dtype == WSF_F32 || dtype == WSF_F16 || dtype == WSF_BF16; }

// a * b without overflow of int64 (both non-negative)
bool mul_ok(int64_t a, int64_t b, int64_t* out) {
    if (a == 0 || b == 0) {
        *out = 0;
        return true;
    }
    if (a > INT64_MAX / b) return false;
    *out = a * b;
    return true;
}

// Byte extent of a [rows, cols] matrix with row stride ld (elements): the
// span from the first to one past the last element; 0 if empty; -1 on
// overflow.
int64_t extent_bytes(int64_t rows, int64_t cols, int64_t ld, int esize) {
    if (rows == 0 || cols == 0) return 0;
    int64_t a;
    if (!mul_ok(rows - 1, ld, &a)) return -1;
    if (a > INT64_MAX - cols) return -1;
    int64_t b;
    if (!mul_ok(a + cols, esize, &b)) return -1;
    return b;
}

bool aligned_to(const void* p, int a) { return ((uintptr_t)p % (uintptr_t)a) == 0; }

struct Span {
    uintptr_t lo, hi;  // [lo, hi)
};

Span span(const void* p, int64_t bytes) {
    return Span{(uintptr_t)p, (uintptr_t)p + (uintptr_t)(bytes > 0 ? bytes : 0)};
}

bool overlap(Span a, Span b) {
    if (a.lo == a.hi || b.lo == b.hi) return false;
    return a.lo < b.hi && b.lo < a.hi;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? WSF_OK : WSF_ERR_CUDA; }

}  // namespace

extern "C" {

const char* wsf_status_string(int status) {
    switch (status) {
        case WSF_OK: return "ok";
        case WSF_ERR_NULL_PTR: return "a required pointer is NULL";
        case WSF_ERR_BAD_SHAPE: return "negative extent or size overflow";
        case WSF_ERR_BAD_DTYPE: return "unknown storage type";
        case WSF_ERR_BAD_STRIDE: return "row stride smaller than the row length";
        case WSF_ERR_WORKSPACE: return "workspace missing or too small";
        case WSF_ERR_OVERLAP: return "an output overlaps an input or another output";
        case WSF_ERR_MISALIGNED: return "pointer not aligned to its element type";
        case WSF_ERR_BAD_ARG: return "invalid argument";
        case WSF_ERR_CUDA: return "CUDA launch failed";
        default: return "unknown status";
    }
}

int wsf_version(void) { return 100; }

int wsf_selftest_exchange_timeout(unsigned* count, unsigned limit_ms, wsf_stream_t stream) {
    if (!count) return WSF_ERR_NULL_PTR;
    if (!aligned_to(count, 4)) return WSF_ERR_MISALIGNED;
    if (limit_ms < 1 || limit_ms > 1000) return WSF_ERR_BAD_ARG;
    return cuda_status(wsf::launch_exchange_timeout(count, (uint64_t)limit_ms * 1000000ull,
                                                    (cudaStream_t)stream));
}

int wsf_selftest_waiting_warps(void) { return wsf::selftest_waiting_warps(); }

int wsf_cluster_wait_timeouts(unsigned* count, int reset) {
    if (!count) return WSF_ERR_NULL_PTR;
    if (reset != 0 && reset != 1) return WSF_ERR_BAD_ARG;
    unsigned a = 0, b = 0;
    cudaError_t e = wsf::norm_wait_timeouts(&a, reset != 0);
    if (e == cudaSuccess) e = wsf::softmax_wait_timeouts(&b, reset != 0);
    if (e != cudaSuccess) return WSF_ERR_CUDA;
    *count = a + b;
    return WSF_OK;
}

int ws_fwd(const void* x, int64_t ldx, const float* w, void* y, int64_t N, int64_t D, int dtype,
           wsf_stream_t stream) {
    if (!valid_dtype(dtype)) return WSF_ERR_BAD_DTYPE;
    if (N < 0 || D < 0) return WSF_ERR_BAD_SHAPE;
    const int es = elt_bytes(dtype);
    const bool xin = N > 0 && D > 0;
    if (xin && ldx < D) return WSF_ERR_BAD_STRIDE;
    const int64_t xb = xin ? extent_bytes(N, D, ldx, es) : 0;
    int64_t yb, wb;
    if (xb < 0 || !mul_ok(N, es, &yb) || !mul_ok(D, 4, &wb)) return WSF_ERR_BAD_SHAPE;
    if ((xin && (!x || !w)) || (N > 0 && !y)) return WSF_ERR_NULL_PTR;
    if (!aligned_to(x, es) || !aligned_to(w, 4) || !aligned_to(y, es)) return WSF_ERR_MISALIGNED;
    if (N == 0) return WSF_OK;
    const Span sy = span(y, yb);
    if (overlap(sy, span(x, xb)) || overlap(sy, span(w, xin ? wb : 0))) return WSF_ERR_OVERLAP;
    return cuda_status(wsf::launch_ws_fwd(x, ldx, w, y, N, D, dtype, (cudaStream_t)stream));
}

size_t ws_bwd_workspace_bytes(int64_t N, int64_t D, int dtype, int64_t block_n) {
    if (!valid_dtype(dtype) || N < 0 || D < 0 || block_n < 0) return SIZE_MAX;
    const int64_t P = wsf::ws_tiles(N, D, dtype, block_n);
    int64_t b;
    if (!mul_ok(P, D, &b) || b > INT64_MAX / 16) return SIZE_MAX;
    return (size_t)(wsf::gradient_plane(P, D) * 4 * 2);  // high and low planes
}

}  // extern "C"

// Validation of ws_bwd's arguments, shared with ws_bwd_noalloc (which has no
// caller workspace: check_ws = false skips the workspace's alignment, size
// and overlap checks).  *need receives ws_bwd_workspace_bytes for the sizes.
int wsf::ws_bwd_check(const void* x, int64_t ldx, const float* w, const void* dy, void* dx,
                      int64_t lddx, float* grad_w, int accumulate, const void* workspace,
                      size_t workspace_bytes, bool check_ws, int64_t block_n, int64_t N,
                      int64_t D, int dtype, size_t* need) {
    if (!valid_dtype(dtype)) return WSF_ERR_BAD_DTYPE;
    if (N < 0 || D < 0) return WSF_ERR_BAD_SHAPE;
    if (block_n < 0 || (accumulate != 0 && accumulate != 1)) return WSF_ERR_BAD_ARG;
    const int es = elt_bytes(dtype);
    const bool mat = N > 0 && D > 0;
    if (mat && (ldx < D || lddx < D)) return WSF_ERR_BAD_STRIDE;
    const int64_t xb = mat ? extent_bytes(N, D, ldx, es) : 0;
    const int64_t dxb = mat ? extent_bytes(N, D, lddx, es) : 0;
    int64_t dyb, wb;
    if (xb < 0 || dxb < 0 || !mul_ok(N, es, &dyb) || !mul_ok(D, 4, &wb)) return WSF_ERR_BAD_SHAPE;
    if ((mat && (!x || !dy || !dx || !w)) || (D > 0 && !grad_w)) return WSF_ERR_NULL_PTR;
    if (!aligned_to(x, es) || !aligned_to(dy, es) || !aligned_to(dx, es) || !aligned_to(w, 4) ||
        !aligned_to(grad_w, 4) || (check_ws && !aligned_to(workspace, 4)))
        return WSF_ERR_MISALIGNED;
    *need = ws_bwd_workspace_bytes(N, D, dtype, block_n);
    if (*need == SIZE_MAX) return WSF_ERR_BAD_SHAPE;
    if (check_ws && *need > 0 && (!workspace || workspace_bytes < *need)) return WSF_ERR_WORKSPACE;
    if (D == 0) return WSF_OK;
    const Span sdx = span(dx, dxb), sg = span(grad_w, wb);
    const Span sws = span(check_ws ? workspace : nullptr, check_ws ? (int64_t)*need : 0);
    const Span sx = span(x, xb), sdy = span(dy, mat ? dyb : 0), sw = span(w, mat ? wb : 0);
    if (overlap(sdx, sx) || overlap(sdx, sdy) || overlap(sdx, sw) || overlap(sg, sx) ||
        overlap(sg, sdy) || overlap(sg, sw) || overlap(sws, sx) || overlap(sws, sdy) ||
        overlap(sws, sw) || overlap(sdx, sg) || overlap(sdx, sws) || overlap(sg, sws))
        return WSF_ERR_OVERLAP;
    return WSF_OK;
}

extern "C" {

int ws_bwd(const void* x, int64_t ldx, const float* w, const void* dy, void* dx, int64_t lddx,
           float* grad_w, int accumulate, void* workspace, size_t workspace_bytes, int64_t block_n,
           int64_t N, int64_t D, int dtype, wsf_stream_t stream) {
    size_t need = 0;
    const int rc = wsf::ws_bwd_check(x, ldx, w, dy, dx, lddx, grad_w, accumulate, workspace,
                                     workspace_bytes, true, block_n, N, D, dtype, &need);
    if (rc != WSF_OK || D == 0) return rc;
    return cuda_status(wsf::launch_ws_bwd(x, ldx, w, dy, dx, lddx, grad_w, accumulate,
                                          (float*)workspace, block_n, N, D, dtype,
                                          (cudaStream_t)stream));
}

int silu_fwd(const void* x, const float* w, void* y, int64_t n, int dtype, wsf_stream_t stream) {
    if (!valid_dtype(dtype)) return WSF_ERR_BAD_DTYPE;
    if (n < 0) return WSF_ERR_BAD_SHAPE;
    const int es = elt_bytes(dtype);
    int64_t b;
    if (!mul_ok(n, es, &b)) return WSF_ERR_BAD_SHAPE;
    if (n > 0 && (!x || !y || !w)) return WSF_ERR_NULL_PTR;
    if (!aligned_to(x, es) || !aligned_to(y, es) || !aligned_to(w, 4)) return WSF_ERR_MISALIGNED;
    if (n == 0) return WSF_OK;
    const Span sy = span(y, b);
    if (overlap(sy, span(x, b)) || overlap(sy, span(w, 4))) return WSF_ERR_OVERLAP;
    return cuda_status(wsf::launch_silu_fwd(x, w, y, n, dtype, (cudaStream_t)stream));
}

size_t silu_bwd_workspace_bytes(int64_t n, int dtype) {
    if (!valid_dtype(dtype) || n < 0) return SIZE_MAX;
    const int64_t P = wsf::silu_tiles(n);
    return (size_t)(wsf::gradient_plane(P, 1) * 4 * 2);  // high and low planes
}

int silu_bwd(const void* dy, const void* x, const float* w, void* dx, float* dw, int accumulate,
             void* workspace, size_t workspace_bytes, int64_t n, int dtype, wsf_stream_t stream) {
    if (!valid_dtype(dtype)) return WSF_ERR_BAD_DTYPE;
    if (n < 0) return WSF_ERR_BAD_SHAPE;
    if (accumulate != 0 && accumulate != 1) return WSF_ERR_BAD_ARG;
    const int es = elt_bytes(dtype);
    int64_t b;
    if (!mul_ok(n, es, &b)) return WSF_ERR_BAD_SHAPE;
    if (!dw || (n > 0 && (!x || !dy || !dx || !w))) return WSF_ERR_NULL_PTR;
    if (!aligned_to(x, es) || !aligned_to(dy, es) || !aligned_to(dx, es) || !aligned_to(w, 4) ||
        !aligned_to(dw, 4) || !aligned_to(workspace, 4))
        return WSF_ERR_MISALIGNED;
    const size_t need = silu_bwd_workspace_bytes(n, dtype);
    if (need > 0 && (!workspace || workspace_bytes < need)) return WSF_ERR_WORKSPACE;
    const Span sdx = span(dx, b), sdw = span(dw, 4), sws = span(workspace, (int64_t)need);
    const Span sx = span(x, b), sdy = span(dy, b), sw = span(w, n > 0 ? 4 : 0);
    if (overlap(sdx, sx) || overlap(sdx, sdy) || overlap(sdx, sw) || overlap(sdw, sx) ||
        overlap(sdw, sdy) || overlap(sdw, sw) || overlap(sws, sx) || overlap(sws, sdy) ||
        overlap(sws, sw) || overlap(sdx, sdw) || overlap(sdx, sws) || overlap(sdw, sws))
        return WSF_ERR_OVERLAP;
    return cuda_status(wsf::launch_silu_bwd(dy, x, w, dx, dw, accumulate, (float*)workspace, n,
                                            dtype, (cudaStream_t)stream));
}

int ws_bwd_atomic(const void* x, int64_t ldx, const float* w, const void* dy, void* dx,
                  int64_t lddx, float* grad_w, int accumulate, int64_t N, int64_t D, int dtype,
                  wsf_stream_t stream) {
    if (!valid_dtype(dtype)) return WSF_ERR_BAD_DTYPE;
    if (N < 0 || D < 0) return WSF_ERR_BAD_SHAPE;
    if (accumulate != 0 && accumulate != 1) return WSF_ERR_BAD_ARG;
    const int es = elt_bytes(dtype);
    const bool mat = N > 0 && D > 0;
    if (mat && (ldx < D || lddx < D)) return WSF_ERR_BAD_STRIDE;
    const int64_t xb = mat ? extent_bytes(N, D, ldx, es) : 0;
    const int64_t dxb = mat ? extent_bytes(N, D, lddx, es) : 0;
    int64_t dyb, wb;
    if (xb < 0 || dxb < 0 || !mul_ok(N, es, &dyb) || !mul_ok(D, 4, &wb)) return WSF_ERR_BAD_SHAPE;
    if ((mat && (!x || !dy || !dx || !w)) || (D > 0 && !grad_w)) return WSF_ERR_NULL_PTR;
    if (D == 0) return WSF_OK;
    if (mat && !wsf::ws_bwd_atomic_supported(x, ldx, w, dy, dx, lddx, grad_w, D, dtype))
        return WSF_ERR_MISALIGNED;
    const Span sdx = span(dx, dxb), sg = span(grad_w, wb);
    const Span sx = span(x, xb), sdy = span(dy, mat ? dyb : 0), sw = span(w, mat ? wb : 0);
    if (overlap(sdx, sx) || overlap(sdx, sdy) || overlap(sdx, sw) || overlap(sg, sx) ||
        overlap(sg, sdy) || overlap(sg, sw) || overlap(sdx, sg))
        return WSF_ERR_OVERLAP;
    return cuda_status(wsf::launch_ws_bwd_atomic(x, ldx, w, dy, dx, lddx, grad_w, accumulate, N, D,
                                                 dtype, (cudaStream_t)stream));
}

int silu_bwd_atomic(const void* dy, const void* x, const float* w, void* dx, float* dw,
                    int accumulate, int64_t n, int dtype, wsf_stream_t stream) {
    if (!valid_dtype(dtype)) return WSF_ERR_BAD_DTYPE;
    if (n < 0) return WSF_ERR_BAD_SHAPE;
    if (accumulate != 0 && accumulate != 1) return WSF_ERR_BAD_ARG;
    const int es = elt_bytes(dtype);
    int64_t b;
    if (!mul_ok(n, es, &b)) return WSF_ERR_BAD_SHAPE;
    if (!dw || (n > 0 && (!x || !dy || !dx || !w))) return WSF_ERR_NULL_PTR;
    if (!aligned_to(x, es) || !aligned_to(dy, es) || !aligned_to(dx, es) || !aligned_to(w, 4) ||
        !aligned_to(dw, 4))
        return WSF_ERR_MISALIGNED;
    const Span sdx = span(dx, b), sdw = span(dw, 4);
    const Span sx = span(x, b), sdy = span(dy, b), sw = span(w, n > 0 ? 4 : 0);
    if (overlap(sdx, sx) || overlap(sdx, sdy) || overlap(sdx, sw) || overlap(sdw, sx) ||
        overlap(sdw, sdy) || overlap(sdw, sw) || overlap(sdx, sdw))
        return WSF_ERR_OVERLAP;
    return cuda_status(wsf::launch_silu_bwd_atomic(dy, x, w, dx, dw, accumulate, n, dtype,
                                                   (cudaStream_t)stream));
}

int softmax_fwd(const void* x, int64_t ldx, void* y, int64_t ldy, int64_t N, int64_t D, int dtype,
                wsf_stream_t stream) {
    if (!valid_dtype(dtype)) return WSF_ERR_BAD_DTYPE;
    if (N < 0 || D < 0) return WSF_ERR_BAD_SHAPE;
    const int es = elt_bytes(dtype);
    const bool mat = N > 0 && D > 0;
    if (mat && (ldx < D || ldy < D)) return WSF_ERR_BAD_STRIDE;
    const int64_t xb = mat ? extent_bytes(N, D, ldx, es) : 0;
    const int64_t yb = mat ? extent_bytes(N, D, ldy, es) : 0;
    if (xb < 0 || yb < 0) return WSF_ERR_BAD_SHAPE;
    if (mat && (!x || !y)) return WSF_ERR_NULL_PTR;
    if (!aligned_to(x, es) || !aligned_to(y, es)) return WSF_ERR_MISALIGNED;
    if (!mat) return WSF_OK;
    if (overlap(span(y, yb), span(x, xb))) return WSF_ERR_OVERLAP;
    return cuda_status(wsf::launch_softmax_fwd(x, ldx, y, ldy, N, D, dtype, (cudaStream_t)stream));
}

int softmax_bwd(const void* y, int64_t ldy, const void* dy, int64_t lddy, void* dx, int64_t lddx,
                int64_t N, int64_t D, int dtype, wsf_stream_t stream) {
    if (!valid_dtype(dtype)) return WSF_ERR_BAD_DTYPE;
    if (N < 0 || D < 0) return WSF_ERR_BAD_SHAPE;
    const int es = elt_bytes(dtype);
    const bool mat = N > 0 && D > 0;
    if (mat && (ldy < D || lddy < D || lddx < D)) return WSF_ERR_BAD_STRIDE;
    const int64_t yb = mat ? extent_bytes(N, D, ldy, es) : 0;
    const int64_t gb = mat ? extent_bytes(N, D, lddy, es) : 0;
    const int64_t xb = mat ? extent_bytes(N, D, lddx, es) : 0;
    if (yb < 0 || gb < 0 || xb < 0) return WSF_ERR_BAD_SHAPE;
    if (mat && (!y || !dy || !dx)) return WSF_ERR_NULL_PTR;
    if (!aligned_to(y, es) || !aligned_to(dy, es) || !aligned_to(dx, es)) return WSF_ERR_MISALIGNED;
    if (!mat) return WSF_OK;
    const Span sdx = span(dx, xb);
    if (overlap(sdx, span(y, yb)) || overlap(sdx, span(dy, gb))) return WSF_ERR_OVERLAP;
    return cuda_status(wsf::launch_softmax_bwd(y, ldy, dy, lddy, dx, lddx, N, D, dtype,
                                               (cudaStream_t)stream));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// RMSNorm / LayerNorm
namespace {

bool valid_eps(float eps) { return eps >= 0.0f && eps <= 3.0e38f; }  // finite, not negative

size_t norm_ws_bytes(int64_t N, int64_t D, int dtype, int nout) {
    if (!valid_dtype(dtype) || N < 0 || D < 0) return SIZE_MAX;
    const int64_t P = wsf::norm_tiles(N, D);
    int64_t b;
    if (!mul_ok(P, D, &b) || !mul_ok(b, 4 * nout, &b) || b > INT64_MAX - 255) return SIZE_MAX;
    return (size_t)((b + 255) / 256 * 256);
}

int norm_fwd_entry(const void* x, int64_t ldx, const float* w, const float* b, float eps, void* y,
                   int64_t ldy, int64_t N, int64_t D, int dtype, int layer, wsf_stream_t stream) {
    if (!valid_dtype(dtype)) return WSF_ERR_BAD_DTYPE;
    if (N < 0 || D < 0) return WSF_ERR_BAD_SHAPE;
    if (!valid_eps(eps)) return WSF_ERR_BAD_ARG;
    const int es = elt_bytes(dtype);
    const bool mat = N > 0 && D > 0;
    if (mat && (ldx < D || ldy < D)) return WSF_ERR_BAD_STRIDE;
    const int64_t xb = mat ? extent_bytes(N, D, ldx, es) : 0;
    const int64_t yb = mat ? extent_bytes(N, D, ldy, es) : 0;
    int64_t wb;
    if (xb < 0 || yb < 0 || !mul_ok(D, 4, &wb)) return WSF_ERR_BAD_SHAPE;
    if (mat && (!x || !y || !w || (layer && !b))) return WSF_ERR_NULL_PTR;
    if (!aligned_to(x, es) || !aligned_to(y, es) || !aligned_to(w, 4) || !aligned_to(b, 4))
        return WSF_ERR_MISALIGNED;
    if (!mat) return WSF_OK;
    const Span sy = span(y, yb);
    if (overlap(sy, span(x, xb)) || overlap(sy, span(w, wb)) ||
        (layer && overlap(sy, span(b, wb))))
        return WSF_ERR_OVERLAP;
    return cuda_status(wsf::launch_norm_fwd(x, ldx, w, layer ? b : nullptr, eps, y, ldy, N, D,
                                            dtype, layer, (cudaStream_t)stream));
}

int norm_bwd_entry(const void* x, int64_t ldx, const float* w, const void* dy, int64_t lddy,
                   float eps, void* dx, int64_t lddx, float* grad_w, float* grad_b, int accumulate,
                   void* workspace, size_t workspace_bytes, int64_t N, int64_t D, int dtype,
                   int layer, wsf_stream_t stream) {
    if (!valid_dtype(dtype)) return WSF_ERR_BAD_DTYPE;
    if (N < 0 || D < 0) return WSF_ERR_BAD_SHAPE;
    if (!valid_eps(eps) || (accumulate != 0 && accumulate != 1)) return WSF_ERR_BAD_ARG;
    const int es = elt_bytes(dtype);
    const bool mat = N > 0 && D > 0;
    if (mat && (ldx < D || lddy < D || lddx < D)) return WSF_ERR_BAD_STRIDE;
    const int64_t xb = mat ? extent_bytes(N, D, ldx, es) : 0;
    const int64_t gb = mat ? extent_bytes(N, D, lddy, es) : 0;
    const int64_t dxb = mat ? extent_bytes(N, D, lddx, es) : 0;
    int64_t wb;
    if (xb < 0 || gb < 0 || dxb < 0 || !mul_ok(D, 4, &wb)) return WSF_ERR_BAD_SHAPE;
    if ((mat && (!x || !dy || !dx || !w)) || (D > 0 && (!grad_w || (layer && !grad_b))))
        return WSF_ERR_NULL_PTR;
    if (!aligned_to(x, es) || !aligned_to(dy, es) || !aligned_to(dx, es) || !aligned_to(w, 4) ||
        !aligned_to(grad_w, 4) || !aligned_to(grad_b, 4) || !aligned_to(workspace, 4))
        return WSF_ERR_MISALIGNED;
    const size_t need = norm_ws_bytes(N, D, dtype, layer ? 2 : 1);
    if (need == SIZE_MAX) return WSF_ERR_BAD_SHAPE;
    if (need > 0 && (!workspace || workspace_bytes < need)) return WSF_ERR_WORKSPACE;
    if (D == 0) return WSF_OK;
    const Span ins[3] = {span(x, xb), span(dy, gb), span(w, mat ? wb : 0)};
    const Span outs[4] = {span(dx, dxb), span(grad_w, wb), span(grad_b, layer ? wb : 0),
                          span(workspace, (int64_t)need)};
    for (int i = 0; i < 4; i++) {
        for (int j = 0; j < 3; j++)
            if (overlap(outs[i], ins[j])) return WSF_ERR_OVERLAP;
        for (int j = i + 1; j < 4; j++)
            if (overlap(outs[i], outs[j])) return WSF_ERR_OVERLAP;
    }
    return cuda_status(wsf::launch_norm_bwd(x, ldx, w, dy, lddy, eps, dx, lddx, grad_w,
                                            layer ? grad_b : nullptr, accumulate,
                                            (float*)workspace, N, D, dtype, layer,
                                            (cudaStream_t)stream));
}

}  // namespace

extern "C" {

int rmsnorm_fwd(const void* x, int64_t ldx, const float* w, float eps, void* y, int64_t ldy,
                int64_t N, int64_t D, int dtype, wsf_stream_t stream) {
    return norm_fwd_entry(x, ldx, w, nullptr, eps, y, ldy, N, D, dtype, 0, stream);
}

size_t rmsnorm_bwd_workspace_bytes(int64_t N, int64_t D, int dtype) {
    return norm_ws_bytes(N, D, dtype, 1);
}

int rmsnorm_bwd(const void* x, int64_t ldx, const float* w, const void* dy, int64_t lddy,
                float eps, void* dx, int64_t lddx, float* grad_w, int accumulate, void* workspace,
                size_t workspace_bytes, int64_t N, int64_t D, int dtype, wsf_stream_t stream) {
    return norm_bwd_entry(x, ldx, w, dy, lddy, eps, dx, lddx, grad_w, nullptr, accumulate,
                          workspace, workspace_bytes, N, D, dtype, 0, stream);
}

int layernorm_fwd(const void* x, int64_t ldx, const float* w, const float* b, float eps, void* y,
                  int64_t ldy, int64_t N, int64_t D, int dtype, wsf_stream_t stream) {
    return norm_fwd_entry(x, ldx, w, b, eps, y, ldy, N, D, dtype, 1, stream);
}

size_t layernorm_bwd_workspace_bytes(int64_t N, int64_t D, int dtype) {
    return norm_ws_bytes(N, D, dtype, 2);
}

int layernorm_bwd(const void* x, int64_t ldx, const float* w, const void* dy, int64_t lddy,
                  float eps, void* dx, int64_t lddx, float* grad_w, float* grad_b, int accumulate,
                  void* workspace, size_t workspace_bytes, int64_t N, int64_t D, int dtype,
                  wsf_stream_t stream) {
    return norm_bwd_entry(x, ldx, w, dy, lddy, eps, dx, lddx, grad_w, grad_b, accumulate,
                          workspace, workspace_bytes, N, D, dtype, 1, stream);
}

}  // extern "C"
