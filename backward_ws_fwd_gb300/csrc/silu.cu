// silu.cu — scaled-SiLU forward and backward kernels for sm_103a.
//
// Operator ("Backward in Triton — autograd.Function and the backward grid",
// § A complete minimal example — fused scaled-SiLU): s = sigmoid(x),
// y = w·x·s with one learnable scalar w.  Backward: dx = dy·w·(s + x·s·(1−s))
// is elementwise; dw = Σ dy·x·s reduces over every element.  The page's
// atomic add of per-block sums is replaced by the two-pass partials buffer
// that its § The backward grid is not the forward grid names as the
// deterministic choice: per-block fp32 partials, then one block sums them in
// a fixed tree order.  s is recomputed from x in the backward (§ Save vs
// recompute).
//
// Evaluation in fp32.  With a = |x| and t = exp(−a) (never overflows),
// r = 1/(1+t):
//   x >= 0:  s = r,    silu'(x) = r²·(1 + t·(1+x))
//   x <  0:  s = t·r,  silu'(x) = t·r²·((1+x) + t)
// Both are algebraically s + x·s·(1−s).  The second form keeps the
// cancellation near the minimum of silu (x ≈ −1.2785, where silu' = 0) down
// to the error of exp: (1+x) is exact for x in [−2, −1/2] and (1+x) + t is
// an exact difference there.
//
// 16-bit storage takes a shorter form, because the 2^-11 half-unit of a
// 16-bit result leaves room: with u = e^(−x) from the hardware ex2.approx
// (of −x·log2 e; relative error ~|x|·6e-8) and s = 1/(1+u) from rcp.approx,
//   silu = x·s,   silu'(x) = s + x·u·s²          (as s·(1−s) = u·s²)
// — no branch on the sign of x.  u = +inf (x < −88) gives s = +0 in the
// forward; the backward caps −x·log2 e at 126 so that u·s stays finite.
// Near the zero of silu' (x ≈ −1.2785) the sum cancels, but its two terms
// carry ~3e-7 relative error, ~1e-7 of the terms' size against a 16-bit
// tolerance of 2^-10.  The full-precision functions made these kernels
// instruction-bound.  binary32 storage keeps expf, an IEEE division and the
// two-branch form above.
#include <algorithm>
#include <type_traits>

#include "wsf_device.cuh"
#include "wsf_internal.h"

namespace wsf {

constexpr int64_t kSiluTilesMax = 8 * kDesignSMs;   // 1216 partials at most
constexpr int64_t kSiluElemsPerTileMin = 8192;

int64_t silu_tiles(int64_t n) {
    if (n <= 0) return 0;
    const int64_t p = (n + kSiluElemsPerTileMin - 1) / kSiluElemsPerTileMin;
    return p < kSiluTilesMax ? p : kSiluTilesMax;
}

struct SiluTerms {
    float silu;   // x·s
    float dsilu;  // d(x·s)/dx
};

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2_approx(float v) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ float rcp_approx(float v) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// exp(-a) for a >= 0 and 1/d for d in [1, 2], full precision (binary32 storage)
__device__ __forceinline__ float exp_neg(float a) { return expf(-a); }
__device__ __forceinline__ float recip(float d) { return 1.0f / d; }

template <typename T>
constexpr bool kFastMath = !std::is_same<T, float>::value;

template <bool Fast>
__device__ __forceinline__ float silu_only(float x) {
    if constexpr (Fast) {
        const float u = ex2_approx(x * -kLog2e);
        return x * rcp_approx(1.0f + u);
    }
    const float t = exp_neg(fabsf(x));
    const float r = recip(1.0f + t);
    const float s = (x >= 0.f) ? r : t * r;
    return x * s;
}

template <bool Fast>
__device__ __forceinline__ SiluTerms silu_terms(float x) {
    SiluTerms o;
    if constexpr (Fast) {
        const float u = ex2_approx(fminf(x * -kLog2e, 126.0f));
        const float s = rcp_approx(1.0f + u);
        o.silu = x * s;
        o.dsilu = fmaf(x, (u * s) * s, s);
        return o;
    }
    const float t = exp_neg(fabsf(x));
    const float r = recip(1.0f + t);
    if (x >= 0.f) {
        o.silu = x * r;
        o.dsilu = (r * r) * fmaf(t, 1.0f + x, 1.0f);
    } else {
        const float s = t * r;
        o.silu = x * s;
        o.dsilu = (s * r) * ((1.0f + x) + t);
    }
    return o;
}

// ---------------------------------------------------------------------------
// Forward: 16-byte vectors, U per thread in flight, grid-stride.
template <typename T, int U, int NT>
__global__ void __launch_bounds__(NT)
    silu_fwd_vec(const T* __restrict__ x, const float* __restrict__ w, T* __restrict__ y,
                 int64_t n) {
    using E = Elt<T>;
    constexpr int V = E::V;
    pdl_wait();
    const float wv = __ldg(w);
    const int64_t nv = n / V;
    for (int64_t base = (int64_t)blockIdx.x * NT * U; base < nv; base += (int64_t)gridDim.x * NT * U) {
        Raw16 xr[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int64_t i = base + (int64_t)u * NT + threadIdx.x;
            xr[u] = (i < nv) ? ld_stream(x + i * V) : raw_zero();
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int64_t i = base + (int64_t)u * NT + threadIdx.x;
            if (i < nv) {
                float f[V];
                E::widen(xr[u], f);
#pragma unroll
                for (int v = 0; v < V; v++) f[v] = wv * silu_only<kFastMath<T>>(f[v]);
                st_stream(y + i * V, E::narrow(f));
            }
        }
    }
    if (blockIdx.x == 0) {
        const int64_t k = nv * V + threadIdx.x;
        if (k < n) E::store1(y + k, wv * silu_only<kFastMath<T>>(E::load1(x + k)));
    }
    pdl_trigger();
}

template <typename T, int NT>
__global__ void __launch_bounds__(NT)
    silu_fwd_scalar(const T* __restrict__ x, const float* __restrict__ w, T* __restrict__ y,
                    int64_t n) {
    using E = Elt<T>;
    pdl_wait();
    const float wv = __ldg(w);
    for (int64_t k = (int64_t)blockIdx.x * NT + threadIdx.x; k < n; k += (int64_t)gridDim.x * NT)
        E::store1(y + k, wv * silu_only<kFastMath<T>>(E::load1(x + k)));
    pdl_trigger();
}

// ---------------------------------------------------------------------------
// Backward, stage 1.  Block p owns the 16-byte vectors p·NT·U + k·P·NT·U +
// [0, NT·U) for k = 0, 1, ... (grid-stride, so that the whole grid sweeps
// memory in order — contiguous per-block ranges measured ~10% slower at the
// c2 size), and the last block the n mod V tail elements; each thread
// accumulates dy·silu(x) over its elements in order, then the block combines:
// xor butterfly inside each warp, warps added in index order.  The ownership
// depends only on n, so the partials, and dw, are the same bits every run.
// Sums are compensated pairs (hi, lo): a thread adds the V terms of each
// 16-byte vector in binary32 and that vector's sum into its pair with
// TwoSum; warps, the block and the second stage add pairs.  The binary32
// vector sums err by a few units of their own last place, random in sign,
// below the error of the terms themselves (the 16-bit path's approximate
// exponential and reciprocal).  A block's partial is stored as its high part
// at part[p] and its low part at part[plane + p].  With ATOMIC the block's
// sum is added into *out with one atomic addition (the page's own scheme,
// kept as a measured comparison: the order of the blocks' additions, and so
// the bits of dw, depend on scheduling).
template <int NT>
__device__ __forceinline__ Acc2 block_sum2(Acc2 acc) {  // the result is thread 0's
    constexpr int NW = NT / 32;
    __shared__ Acc2 red[NW];
    acc = group_sum2<32>(acc);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    Acc2 t = red[0];
    if (threadIdx.x == 0) {
#pragma unroll
        for (int q = 1; q < NW; q++) t = acc2_add(t, red[q]);
    }
    return t;
}

template <int NT, bool ATOMIC = false>
__device__ __forceinline__ void block_sum_store(Acc2 acc, float* out, int64_t plane) {
    const Acc2 t = block_sum2<NT>(acc);
    if (threadIdx.x == 0) {
        if constexpr (ATOMIC) {
            atomicAdd(out, acc2_value(t));
        } else {
            out[0] = t.hi;
            out[plane] = t.lo;
        }
    }
}

template <typename T, int U, int NT, bool ATOMIC = false>
__global__ void __launch_bounds__(NT)
    silu_bwd_vec(const T* __restrict__ dy, const T* __restrict__ x, const float* __restrict__ w,
                 T* __restrict__ dx, float* __restrict__ part, int64_t plane, int64_t n,
                 int64_t P) {
    using E = Elt<T>;
    constexpr int V = E::V;
    pdl_wait();
    const float wv = __ldg(w);
    const int64_t nv = n / V;
    const int64_t p = blockIdx.x;
    const int64_t ve = nv;
    Acc2 acc = acc2_zero();
    for (int64_t base = p * NT * U; base < ve; base += P * NT * U) {
        Raw16 xr[U], gr[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int64_t i = base + (int64_t)u * NT + threadIdx.x;
            const bool ok = i < ve;
            xr[u] = ok ? ld_stream(x + i * V) : raw_zero();
            gr[u] = ok ? ld_stream(dy + i * V) : raw_zero();
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int64_t i = base + (int64_t)u * NT + threadIdx.x;
            float xf[V], gf[V];
            E::widen(xr[u], xf);
            E::widen(gr[u], gf);
            float vs = 0.f;
#pragma unroll
            for (int v = 0; v < V; v++) {
                const SiluTerms st = silu_terms<kFastMath<T>>(xf[v]);
                vs = fmaf(gf[v], st.silu, vs);
                xf[v] = (gf[v] * wv) * st.dsilu;
            }
            acc2_add1(acc, vs);
            if (i < ve) st_stream(dx + i * V, E::narrow(xf));
        }
    }
    if (p == P - 1) {
        const int64_t k = nv * V + threadIdx.x;
        if (k < n) {
            const float xv = E::load1(x + k), gv = E::load1(dy + k);
            const SiluTerms st = silu_terms<kFastMath<T>>(xv);
            acc2_add1(acc, __fmul_rn(gv, st.silu));
            E::store1(dx + k, (gv * wv) * st.dsilu);
        }
    }
    pdl_trigger();
    block_sum_store<NT, ATOMIC>(acc, ATOMIC ? part : part + p, plane);
}

template <typename T, int NT, bool ATOMIC = false>
__global__ void __launch_bounds__(NT)
    silu_bwd_scalar(const T* __restrict__ dy, const T* __restrict__ x, const float* __restrict__ w,
                    T* __restrict__ dx, float* __restrict__ part, int64_t plane, int64_t n,
                    int64_t P) {
    using E = Elt<T>;
    pdl_wait();
    const float wv = __ldg(w);
    const int64_t p = blockIdx.x;
    const int64_t kb = (p * n) / P, ke = ((p + 1) * n) / P;
    Acc2 acc = acc2_zero();
    for (int64_t k = kb + threadIdx.x; k < ke; k += NT) {
        const float xv = E::load1(x + k), gv = E::load1(dy + k);
        const SiluTerms st = silu_terms<kFastMath<T>>(xv);
        acc2_add1(acc, __fmul_rn(gv, st.silu));
        E::store1(dx + k, (gv * wv) * st.dsilu);
    }
    pdl_trigger();
    block_sum_store<NT, ATOMIC>(acc, ATOMIC ? part : part + p, plane);
}

// Backward, stage 2: one block; thread t sums the pairs part[t], part[t + NT],
// ... in order, then the block combines as above; the pair is rounded once to
// binary32.  dw = (accumulate ? dw : 0) + sum, one binary32 addition.
template <int NT>
__global__ void __launch_bounds__(NT)
    silu_bwd_reduce(const float* __restrict__ part, int64_t plane, int64_t P,
                    float* __restrict__ dw, int accumulate) {
    pdl_wait();
    Acc2 s = acc2_zero();
    for (int64_t i = threadIdx.x; i < P; i += NT) s = acc2_add(s, Acc2{part[i], part[plane + i]});
    const Acc2 t = block_sum2<NT>(s);
    if (threadIdx.x == 0) {
        const float total = acc2_value(t);
        *dw = accumulate ? *dw + total : total;
    }
    pdl_trigger();
}

// ---------------------------------------------------------------------------
static inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
static inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

template <typename T>
static cudaError_t silu_fwd_t(const T* x, const float* w, T* y, int64_t n, cudaStream_t s) {
    constexpr int V = Elt<T>::V;
    if (aligned16(x) && aligned16(y)) {
        constexpr int NT = 256, U = 8;
        const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(cdiv(n / V, NT * U), 8 * kDesignSMs));
        return launch(silu_fwd_vec<T, U, NT>, dim3((unsigned)grid), dim3(NT), 0, s, true, x, w, y,
                      n);
    }
    constexpr int NT = 256;
    const int64_t grid = std::min<int64_t>(cdiv(n, NT), 8 * kDesignSMs);
    return launch(silu_fwd_scalar<T, NT>, dim3((unsigned)grid), dim3(NT), 0, s, true, x, w, y, n);
}

cudaError_t launch_silu_fwd(const void* x, const float* w, void* y, int64_t n, int dtype,
                            cudaStream_t s) {
    switch (dtype) {
        case 0: return silu_fwd_t((const float*)x, w, (float*)y, n, s);
        case 1: return silu_fwd_t((const __half*)x, w, (__half*)y, n, s);
        default: return silu_fwd_t((const __nv_bfloat16*)x, w, (__nv_bfloat16*)y, n, s);
    }
}

template <typename T>
static cudaError_t silu_bwd_t(const T* dy, const T* x, const float* w, T* dx, float* dw,
                              int accumulate, float* part, int64_t n, cudaStream_t s) {
    const int64_t P = silu_tiles(n);
    const int64_t plane = gradient_plane(P, 1);
    cudaError_t e = cudaSuccess;
    if (P > 0) {
        if (aligned16(dy) && aligned16(x) && aligned16(dx)) {
            constexpr int NT = 256, U = 2;
            e = launch(silu_bwd_vec<T, U, NT>, dim3((unsigned)P), dim3(NT), 0, s, true, dy, x, w,
                       dx, part, plane, n, P);
        } else {
            constexpr int NT = 256;
            e = launch(silu_bwd_scalar<T, NT>, dim3((unsigned)P), dim3(NT), 0, s, true, dy, x, w,
                       dx, part, plane, n, P);
        }
        if (e != cudaSuccess) return e;
    }
    constexpr int NT = 1024;
    return launch(silu_bwd_reduce<NT>, dim3(1), dim3(NT), 0, s, true, (const float*)part, plane,
                  P, dw, accumulate);
}

__global__ void __launch_bounds__(32) zero_one_f32(float* __restrict__ p) {
    pdl_wait();
    if (threadIdx.x == 0) *p = 0.f;
    pdl_trigger();
}

template <typename T>
static cudaError_t silu_bwd_atomic_t(const T* dy, const T* x, const float* w, T* dx, float* dw,
                                     int accumulate, int64_t n, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    if (!accumulate) {
        e = launch(zero_one_f32, dim3(1), dim3(32), 0, s, true, dw);
        if (e != cudaSuccess) return e;
    }
    const int64_t P = silu_tiles(n);
    if (P == 0) return e;
    constexpr int NT = 256;
    if (aligned16(dy) && aligned16(x) && aligned16(dx))
        return launch(silu_bwd_vec<T, 2, NT, true>, dim3((unsigned)P), dim3(NT), 0, s, true, dy, x,
                      w, dx, dw, (int64_t)0, n, P);
    return launch(silu_bwd_scalar<T, NT, true>, dim3((unsigned)P), dim3(NT), 0, s, true, dy, x, w,
                  dx, dw, (int64_t)0, n, P);
}

cudaError_t launch_silu_bwd_atomic(const void* dy, const void* x, const float* w, void* dx,
                                   float* dw, int accumulate, int64_t n, int dtype,
                                   cudaStream_t s) {
    switch (dtype) {
        case 0:
            return silu_bwd_atomic_t((const float*)dy, (const float*)x, w, (float*)dx, dw,
                                     accumulate, n, s);
        case 1:
            return silu_bwd_atomic_t((const __half*)dy, (const __half*)x, w, (__half*)dx, dw,
                                     accumulate, n, s);
        default:
            return silu_bwd_atomic_t((const __nv_bfloat16*)dy, (const __nv_bfloat16*)x, w,
                                     (__nv_bfloat16*)dx, dw, accumulate, n, s);
    }
}

cudaError_t launch_silu_bwd(const void* dy, const void* x, const float* w, void* dx, float* dw,
                            int accumulate, float* part, int64_t n, int dtype, cudaStream_t s) {
    switch (dtype) {
        case 0:
            return silu_bwd_t((const float*)dy, (const float*)x, w, (float*)dx, dw, accumulate,
                              part, n, s);
        case 1:
            return silu_bwd_t((const __half*)dy, (const __half*)x, w, (__half*)dx, dw, accumulate,
                              part, n, s);
        default:
            return silu_bwd_t((const __nv_bfloat16*)dy, (const __nv_bfloat16*)x, w,
                              (__nv_bfloat16*)dx, dw, accumulate, part, n, s);
    }
}

}  // namespace wsf
