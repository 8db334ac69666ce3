// softmax.cu — row softmax forward and backward for sm_103a.
//
// "Backprop for kernel writers", §04 The duality: the softmax backward is a
// row-scalar collapse, dx = y ⊙ (dy − Σ_j dy_j·y_j), computed from the saved
// output y ("you need y, not x"), so the dense Jacobian is never formed; the
// stability shift of the forward (x − max x) adds nothing to the backward.
//
// Forward:  y[i,j] = exp(x[i,j] − m_i) / Σ_k exp(x[i,k] − m_i),  m_i = max_k x[i,k]
// Backward: dx[i,j] = y[i,j] · (dy[i,j] − s_i),  s_i = Σ_k dy[i,k]·y[i,k]
//
// Row path (rows of up to 2048 16-byte chunks): a row is held in registers
// by a group of TPR threads (CPT chunks each); the row max and the row sums
// are combined with xor butterflies inside a warp and, for groups wider than
// a warp, through shared memory in warp order.  x (or y and dy) is read once
// and y (dx) written once.  Rows of up to 32,768 chunks are split over a
// thread-block cluster (below), wider rows over a cluster that streams them
// twice (two-pass).  Rows that do not start on 16 bytes, or whose width is
// not a whole number of chunks, are read as the chunks that cover them, with
// the edges masked (Win), when every array of the call has the same offset in
// each row; other rows take a multi-pass element-wise path with one CTA per
// row.  Sums of binary32 rows are compensated and their
// exponentials taken of exactly split differences.
#include <algorithm>
#include <type_traits>

#include "wsf_device.cuh"
#include "wsf_internal.h"

namespace wsf {

template <typename T>
constexpr bool kSoftmaxFast = !std::is_same<T, float>::value;

// ---------------------------------------------------------------------------
// exp(a − b) for binary32 rows, within a few units of 2^-24 relative, built
// on the hardware base-2 exponential:
//  1. d = a − b exactly, as dh + dl (Knuth's TwoSum), so the rounding of the
//     difference (up to |d|·2^-24 in the exponent) never reaches the result;
//  2. t = d·log2(e) as th + tl, with log2(e) carried as L1 + L2 (L1 = log2 e
//     rounded to binary32, L2 = the remainder rounded to binary32): th is
//     dh·L1 rounded, its rounding error is recovered exactly with an FMA
//     (Dekker's exact product), and dl·L1 + dh·L2 are added to that error;
//  3. exp(d) = 2^th · 2^tl: 2^th from ex2.approx (subnormal results kept),
//     2^tl = 1 + tl·ln 2 to first order (|tl| < 2^-15 wherever 2^th does
//     not underflow, so the neglected term is below 2^-31 of the result).
// A masked logit (a = −inf) is first raised to −2^100, whose exponential
// underflows to +0 as exp(−inf) does, without the NaN that −inf − (−inf)
// would leave in the split.
constexpr float kLog2eHi = 1.44269502162933349609375f;  // 0x3FB8AA3B
constexpr float kLog2eLo = 1.925963033500011e-08f;      // log2(e) − kLog2eHi, rounded
constexpr float kLn2f = 0.693147182464599609375f;       // ln 2 rounded to binary32
constexpr float kMaskFloor = 0x1p100f;

__device__ __forceinline__ float ex2_keep_subnormal(float v) {
    float r;
    asm("ex2.approx.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ float exp_diff_f32(float a, float b) {
    float dh, dl;
    two_sum(fmaxf(a, -kMaskFloor), -b, dh, dl);
    const float nth = __fmul_rn(dh, -kLog2eHi);  // −th
    const float tl = fmaf(dh, kLog2eLo, fmaf(dl, kLog2eHi, fmaf(dh, kLog2eHi, nth)));
    const float r = ex2_keep_subnormal(-nth);
    return fmaf(r, __fmul_rn(tl, kLn2f), r);
}

// exp_diff_f32 on two lanes at once (packed f32x2 arithmetic; the same
// operations in the same order, so each lane gets the scalar function's
// bits).  a2: two values of a; nb2 = (−b, −b).
__device__ __forceinline__ uint64_t exp_diff_f32x2(uint64_t a2, uint64_t nb2) {
    float a0, a1;
    f2_unpack(a2, a0, a1);
    a2 = f2_pack(fmaxf(a0, -kMaskFloor), fmaxf(a1, -kMaskFloor));
    // TwoSum(a, −b)
    const uint64_t dh = f2_add(a2, nb2);
    const uint64_t bp = f2_sub(dh, a2);
    const uint64_t dl = f2_add(f2_sub(a2, f2_sub(dh, bp)), f2_sub(nb2, bp));
    const uint64_t L1 = f2_pack(kLog2eHi, kLog2eHi), L2 = f2_pack(kLog2eLo, kLog2eLo);
    const uint64_t nth = f2_mul(dh, f2_pack(-kLog2eHi, -kLog2eHi));
    const uint64_t tl = f2_fma(dh, L2, f2_fma(dl, L1, f2_fma(dh, L1, nth)));
    float n0, n1;
    f2_unpack(nth, n0, n1);
    const uint64_t r = f2_pack(ex2_keep_subnormal(-n0), ex2_keep_subnormal(-n1));
    return f2_fma(r, f2_mul(tl, f2_pack(kLn2f, kLn2f)), r);
}

// exp(a − b) for the terms of the first pass's sum only (two lanes; a ≤ b,
// b finite): the rounded difference scaled by log2(e) in one rounding, then
// ex2.approx.  The two roundings put a term off by up to about
// 2·|a − b|·2^-24 of itself, ex2.approx adds its own few units; the signs
// follow each term's own roundings.  The sum is dominated by the terms
// nearest the maximum, where the error is smallest, and the outputs take
// their exponentials from exp_diff_f32x2.
__device__ __forceinline__ uint64_t exp_sum_f32x2(uint64_t a2, uint64_t nb2) {
    const uint64_t t = f2_mul(f2_add(a2, nb2), f2_pack(kLog2eHi, kLog2eHi));
    float t0, t1;
    f2_unpack(t, t0, t1);
    return f2_pack(ex2_keep_subnormal(t0), ex2_keep_subnormal(t1));
}

// exp(a − b).  Binary32 storage: exp_diff_f32 above.  16-bit storage: the
// hardware exponential of the rounded difference (its error is far below a
// 16-bit unit).
template <bool Fast>
__device__ __forceinline__ float exp_diff(float a, float b) {
    if constexpr (Fast)
        return __expf(a - b);
    else
        return exp_diff_f32(a, b);
}

// Reductions over a group of TPR threads (aligned, consecutive).  Groups of
// more than 32 threads combine per-warp results through `red` (NT/32 floats)
// in warp order; every thread of the CTA must call these together.
template <int TPR>
__device__ __forceinline__ float group_max(float v, float* red) {
    constexpr int W = TPR < 32 ? TPR : 32;
#pragma unroll
    for (int off = W / 2; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL_MASK, v, off));
    if constexpr (TPR > 32) {
        const int wid = threadIdx.x >> 5, first = (threadIdx.x / TPR) * (TPR / 32);
        if ((threadIdx.x & 31) == 0) red[wid] = v;
        __syncthreads();
        v = red[first];
#pragma unroll
        for (int q = 1; q < TPR / 32; q++) v = fmaxf(v, red[first + q]);
        __syncthreads();
    }
    return v;
}

// Plain fp32 group sum with the same combination order as group_sum_acc2
// (xor butterfly in each warp, warps in index order), for 16-bit storage.
template <int TPR>
__device__ __forceinline__ float group_sum_plain(float v, float* red) {
    constexpr int W = TPR < 32 ? TPR : 32;
    v = group_sum<W>(v);
    if constexpr (TPR > 32) {
        const int wid = threadIdx.x >> 5, first = (threadIdx.x / TPR) * (TPR / 32);
        if ((threadIdx.x & 31) == 0) red[wid] = v;
        __syncthreads();
        v = red[first];
#pragma unroll
        for (int q = 1; q < TPR / 32; q++) v += red[first + q];
        __syncthreads();
    }
    return v;
}

template <int TPR>
__device__ __forceinline__ Acc2 group_sum_acc2(Acc2 v, Acc2* red) {
    constexpr int W = TPR < 32 ? TPR : 32;
    v = group_sum2<W>(v);
    if constexpr (TPR > 32) {
        const int wid = threadIdx.x >> 5, first = (threadIdx.x / TPR) * (TPR / 32);
        if ((threadIdx.x & 31) == 0) red[wid] = v;
        __syncthreads();
        v = red[first];
#pragma unroll
        for (int q = 1; q < TPR / 32; q++) v = acc2_add(v, red[first + q]);
        __syncthreads();
    }
    return v;
}


// 16-bit rows: the maximum of a 16-byte chunk taken on packed pairs (exact),
// and e^(x − m) as 2^(x·log2(e) − m·log2(e)) with the argument formed by one
// FMA and the hardware base-2 exponential.
template <typename T>
__device__ __forceinline__ float chunk_max16(const Raw16& r) {
    if constexpr (std::is_same<T, __half>::value) {
        __half2 m;
        memcpy(&m, &r.u[0], 4);
#pragma unroll
        for (int i = 1; i < 4; i++) {
            __half2 h;
            memcpy(&h, &r.u[i], 4);
            m = __hmax2(m, h);
        }
        return fmaxf(__low2float(m), __high2float(m));
    } else {
        __nv_bfloat162 m;
        memcpy(&m, &r.u[0], 4);
#pragma unroll
        for (int i = 1; i < 4; i++) {
            __nv_bfloat162 h;
            memcpy(&h, &r.u[i], 4);
            m = __hmax2(m, h);
        }
        return fmaxf(__low2float(m), __high2float(m));
    }
}

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float exp2_approx(float v) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// Compensated (binary32) or plain (16-bit) running sum.
template <bool Comp>
__device__ __forceinline__ void add_to(Acc2& a, float v) {
    if constexpr (Comp) {
        float s, e;
        two_sum(a.hi, v, s, e);
        a.hi = s;
        a.lo += e;
    } else {
        a.hi += v;
    }
}

// ---------------------------------------------------------------------------
// Row path.  Each CTA takes R = NT / TPR rows per iteration (grid-stride
// over iterations k = 0, 1, ...).  Every thread copies its own chunks of the
// rows of iteration k + S - 1 into private shared-memory slots with cp.async
// while it computes iteration k, so S - 1 iterations' loads are in flight
// without holding registers; only the row reductions synchronise threads.
template <int TPR, int CPT, int NT, int S>
struct RowStage {
    static constexpr size_t bytes(int arrays) { return (size_t)arrays * S * CPT * NT * 16; }
};

// A row of D elements as 16-byte chunks.  Aligned rows (U = false) start at
// their first element.  Otherwise (U) the chunks start at the row's first
// element rounded down to 16 bytes, off = that element's place in chunk 0:
// chunk c holds the row's elements c·V − off … c·V − off + V − 1, and those
// outside [0, D) are masked (reads of the masked elements stay inside the
// 16-byte blocks that hold the row's own elements).  Every array of a call
// has the same offset in each row (checked by the launcher).
template <typename T, bool U>
__device__ __forceinline__ int win_off(const T* row_start) {
    if constexpr (U)
        return (int)(((uintptr_t)row_start & 15u) / sizeof(T));
    else
        return 0;
}

// Row window of a thread's chunk cc (= chunk index in the row): any element
// of the row, only elements of the row, element v of the row.
template <typename T, bool U>
struct Win {
    static constexpr int V = Elt<T>::V;
    int off, D;
    __device__ __forceinline__ bool has(int cc) const {
        return U ? cc * V < off + D : cc * V < D;
    }
    __device__ __forceinline__ bool full(int cc) const {
        return !U || (cc * V >= off && (cc + 1) * V <= off + D);
    }
    __device__ __forceinline__ bool elt(int cc, int v) const {
        const int j = cc * V + v - off;
        return !U || (j >= 0 && j < D);
    }
    // first element of chunk cc, relative to the row's first element
    __device__ __forceinline__ int64_t at(int cc) const { return (int64_t)cc * V - off; }
};

template <typename T, int TPR, int CPT, int NT, bool U>
__device__ __forceinline__ void stage_row(Raw16* slots, const T* __restrict__ p, int64_t ld,
                                          int64_t row, int64_t N, int D, int l) {
    constexpr int V = Elt<T>::V;
    const bool rok = row < N;
    const T* rp = p + (rok ? row : 0) * ld;
    const int off = win_off<T, U>(rp);
    const T* base = rp - off;
    const int nc = (off + D + V - 1) / V;  // D / V for aligned rows
#pragma unroll
    for (int k = 0; k < CPT; k++) {
        const int c = l + k * TPR;
        const bool ok = rok && c < nc;
        cp_async16(&slots[k * NT + threadIdx.x],
                   ok ? (const void*)(base + (int64_t)c * V) : (const void*)p, ok ? 16 : 0);
    }
}

// The 16-bit lanes of a chunk outside [lo, hi) set to −inf (for the packed
// maximum).
template <typename T>
__device__ __forceinline__ Raw16 mask_ninf(Raw16 r, int lo, int hi) {
    constexpr uint32_t ninf = std::is_same<T, __half>::value ? 0xFC00u : 0xFF80u;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        if (2 * i < lo || 2 * i >= hi) r.u[i] = (r.u[i] & 0xFFFF0000u) | ninf;
        if (2 * i + 1 < lo || 2 * i + 1 >= hi) r.u[i] = (r.u[i] & 0x0000FFFFu) | (ninf << 16);
    }
    return r;
}

// Store chunk cc of a row: one 16-byte store for a full chunk, else the
// row's elements one by one.
template <typename T, bool U>
__device__ __forceinline__ void store_chunk(T* row_start, const Win<T, U>& w, int cc,
                                            const float (&o)[Elt<T>::V]) {
    using E = Elt<T>;
    if (w.full(cc)) {
        st_stream(row_start + w.at(cc), E::narrow(o));
    } else {
#pragma unroll
        for (int v = 0; v < E::V; v++)
            if (w.elt(cc, v)) E::store1(row_start + w.at(cc) + v, o[v]);
    }
}

template <typename T, int TPR, int CPT, int NT, int S, bool U>
__global__ void __launch_bounds__(NT)
    softmax_fwd_rows(const T* __restrict__ x, int64_t ldx, T* __restrict__ y, int64_t ldy,
                     int64_t N, int D) {
    using E = Elt<T>;
    constexpr int V = E::V;
    constexpr int R = NT / TPR;
    constexpr bool kComp = std::is_same<T, float>::value;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Raw16* slots = reinterpret_cast<Raw16*>(smem_raw);  // [S][CPT][NT]
    __shared__ float redm[NT / 32];
    __shared__ Acc2 reds[NT / 32];
    const int g = threadIdx.x / TPR, l = threadIdx.x % TPR;
    pdl_wait();
    const int64_t first = (int64_t)blockIdx.x * R + g, stride = (int64_t)gridDim.x * R;
    const int64_t iters = ((int64_t)blockIdx.x * R < N) ? (N - (int64_t)blockIdx.x * R + stride - 1) / stride : 0;
#pragma unroll
    for (int k = 0; k < S - 1; k++) {
        if (k < iters) stage_row<T, TPR, CPT, NT, U>(slots + k * CPT * NT, x, ldx, first + k * stride, N, D, l);
        cp_async_commit();
    }
    for (int64_t k = 0; k < iters; k++) {
        cp_async_wait<S - 2>();
        const int64_t nk = k + S - 1;
        if (nk < iters)
            stage_row<T, TPR, CPT, NT, U>(slots + (nk % S) * CPT * NT, x, ldx, first + nk * stride, N, D, l);
        cp_async_commit();
        const int64_t row = first + k * stride;
        const bool rok = row < N;
        Raw16* cur = slots + (k % S) * CPT * NT;
        const Win<T, U> win{rok ? win_off<T, U>(x + row * ldx) : 0, D};
        T* yrow = y + (rok ? row : 0) * ldy;
        if constexpr (!kComp) {
            // 16-bit storage: packed max, one FMA + ex2 per element, plain
            // sums; an edge chunk of a windowed row gets −inf outside the row
            // (in the thread's own slot), whose exponential is 0
            float m = -INFINITY;
#pragma unroll
            for (int c = 0; c < CPT; c++) {
                const int cc = l + c * TPR;
                if (rok && win.has(cc)) {
                    Raw16 r = cur[c * NT + threadIdx.x];
                    if (!win.full(cc)) {
                        r = mask_ninf<T>(r, win.off - cc * V, win.off + D - cc * V);
                        cur[c * NT + threadIdx.x] = r;
                    }
                    m = fmaxf(m, chunk_max16<T>(r));
                }
            }
            m = group_max<TPR>(m, redm);
            const float ms = m * kLog2e;
            float f[CPT][V];
            float st = 0.f;
#pragma unroll
            for (int c = 0; c < CPT; c++) {
                E::widen(cur[c * NT + threadIdx.x], f[c]);
                const bool ok = rok && win.has(l + c * TPR);
#pragma unroll
                for (int v = 0; v < V; v++) {
                    f[c][v] = ok ? exp2_approx(fmaf(f[c][v], kLog2e, -ms)) : 0.f;
                    st += f[c][v];
                }
            }
            const float inv = 1.0f / group_sum_plain<TPR>(st, redm);
#pragma unroll
            for (int c = 0; c < CPT; c++) {
                const int cc = l + c * TPR;
                if (rok && win.has(cc)) {
                    float o[V];
#pragma unroll
                    for (int v = 0; v < V; v++) o[v] = f[c][v] * inv;
                    store_chunk<T, U>(yrow, win, cc, o);
                }
            }
        } else {
            // binary32 storage: exactly split exponentials, compensated sum
            float f[CPT][V];
            bool cok[CPT];
#pragma unroll
            for (int c = 0; c < CPT; c++) {
                cok[c] = rok && win.has(l + c * TPR);
                E::widen(cur[c * NT + threadIdx.x], f[c]);
            }
            float m = -INFINITY;
#pragma unroll
            for (int c = 0; c < CPT; c++) {
                if (cok[c] && !win.full(l + c * TPR))  // edge chunk: −inf outside the row
#pragma unroll
                    for (int v = 0; v < V; v++)
                        if (!win.elt(l + c * TPR, v)) f[c][v] = -INFINITY;
                if (cok[c])
#pragma unroll
                    for (int v = 0; v < V; v++) m = fmaxf(m, f[c][v]);
            }
            m = group_max<TPR>(m, redm);
            Acc2 s = acc2_zero();
#pragma unroll
            for (int c = 0; c < CPT; c++) {
#pragma unroll
                for (int v = 0; v < V; v++) {
                    // exp(−inf − m) = 0 outside the row
                    f[c][v] = cok[c] ? exp_diff<kSoftmaxFast<T>>(f[c][v], m) : 0.f;
                    add_to<kComp>(s, f[c][v]);
                }
            }
            s = group_sum_acc2<TPR>(s, reds);
            const float inv = 1.0f / (s.hi + s.lo);
#pragma unroll
            for (int c = 0; c < CPT; c++) {
                if (cok[c]) {
                    float o[V];
#pragma unroll
                    for (int v = 0; v < V; v++) o[v] = f[c][v] * inv;
                    store_chunk<T, U>(yrow, win, l + c * TPR, o);
                }
            }
        }
    }
    cp_async_wait<0>();
    pdl_trigger();
}

template <typename T, int TPR, int CPT, int NT, int S, bool U>
__global__ void __launch_bounds__(NT)
    softmax_bwd_rows(const T* __restrict__ y, int64_t ldy, const T* __restrict__ dy, int64_t lddy,
                     T* __restrict__ dx, int64_t lddx, int64_t N, int D) {
    using E = Elt<T>;
    constexpr int V = E::V;
    constexpr int R = NT / TPR;
    constexpr bool kComp = std::is_same<T, float>::value;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Raw16* ys = reinterpret_cast<Raw16*>(smem_raw);  // [S][CPT][NT]
    Raw16* gs = ys + S * CPT * NT;                    // [S][CPT][NT]
    __shared__ Acc2 reds[NT / 32];
    __shared__ float redf[NT / 32];
    const int g = threadIdx.x / TPR, l = threadIdx.x % TPR;
    pdl_wait();
    const int64_t first = (int64_t)blockIdx.x * R + g, stride = (int64_t)gridDim.x * R;
    const int64_t iters = ((int64_t)blockIdx.x * R < N) ? (N - (int64_t)blockIdx.x * R + stride - 1) / stride : 0;
#pragma unroll
    for (int k = 0; k < S - 1; k++) {
        if (k < iters) {
            stage_row<T, TPR, CPT, NT, U>(ys + k * CPT * NT, y, ldy, first + k * stride, N, D, l);
            stage_row<T, TPR, CPT, NT, U>(gs + k * CPT * NT, dy, lddy, first + k * stride, N, D, l);
        }
        cp_async_commit();
    }
    for (int64_t k = 0; k < iters; k++) {
        cp_async_wait<S - 2>();
        const int64_t nk = k + S - 1;
        if (nk < iters) {
            stage_row<T, TPR, CPT, NT, U>(ys + (nk % S) * CPT * NT, y, ldy, first + nk * stride, N, D, l);
            stage_row<T, TPR, CPT, NT, U>(gs + (nk % S) * CPT * NT, dy, lddy, first + nk * stride, N, D, l);
        }
        cp_async_commit();
        const int64_t row = first + k * stride;
        const bool rok = row < N;
        const Raw16* cy = ys + (k % S) * CPT * NT;
        const Raw16* cg = gs + (k % S) * CPT * NT;
        const Win<T, U> win{rok ? win_off<T, U>(y + row * ldy) : 0, D};
        float fy[CPT][V], fg[CPT][V];
        bool cok[CPT];
#pragma unroll
        for (int c = 0; c < CPT; c++) {
            cok[c] = rok && win.has(l + c * TPR);
            E::widen(cy[c * NT + threadIdx.x], fy[c]);
            E::widen(cg[c * NT + threadIdx.x], fg[c]);
            if (U && !win.full(l + c * TPR))
#pragma unroll
                for (int v = 0; v < V; v++)
                    if (!win.elt(l + c * TPR, v)) fy[c][v] = fg[c][v] = 0.f;
        }
        Acc2 s = acc2_zero();
#pragma unroll
        for (int c = 0; c < CPT; c++)
#pragma unroll
            for (int v = 0; v < V; v++) {
                const float a = cok[c] ? fg[c][v] : 0.f, b = cok[c] ? fy[c][v] : 0.f;
                if constexpr (kComp)
                    acc2_fma(s, a, b);
                else
                    s.hi = fmaf(a, b, s.hi);
            }
        float sv;
        if constexpr (kComp) {
            s = group_sum_acc2<TPR>(s, reds);
            sv = s.hi + s.lo;
        } else {
            sv = group_sum_plain<TPR>(s.hi, redf);
        }
        T* dxrow = dx + (rok ? row : 0) * lddx;
#pragma unroll
        for (int c = 0; c < CPT; c++) {
            if (cok[c]) {
                float o[V];
#pragma unroll
                for (int v = 0; v < V; v++) o[v] = fy[c][v] * (fg[c][v] - sv);
                store_chunk<T, U>(dxrow, win, l + c * TPR, o);
            }
        }
    }
    cp_async_wait<0>();
    pdl_trigger();
}

// Wide path: one CTA per row (grid-stride), element-wise loads, three passes
// over the row (max, sum of exponentials, write), each reduction combining the
// threads in a fixed order.
template <typename T, int NT>
__global__ void __launch_bounds__(NT)
    softmax_fwd_wide(const T* __restrict__ x, int64_t ldx, T* __restrict__ y, int64_t ldy,
                     int64_t N, int64_t D) {
    using E = Elt<T>;
    constexpr bool kComp = std::is_same<T, float>::value;
    __shared__ float redm[NT / 32];
    __shared__ Acc2 reds[NT / 32];
    pdl_wait();
    for (int64_t row = blockIdx.x; row < N; row += gridDim.x) {
        const T* xr = x + row * ldx;
        float m = -INFINITY;
        for (int64_t j = threadIdx.x; j < D; j += NT) m = fmaxf(m, E::load1(xr + j));
        m = group_max<NT>(m, redm);
        Acc2 s = acc2_zero();
        for (int64_t j = threadIdx.x; j < D; j += NT)
            add_to<kComp>(s, exp_diff<kSoftmaxFast<T>>(E::load1(xr + j), m));
        s = group_sum_acc2<NT>(s, reds);
        const float inv = 1.0f / (s.hi + s.lo);
        for (int64_t j = threadIdx.x; j < D; j += NT)
            E::store1(y + row * ldy + j, exp_diff<kSoftmaxFast<T>>(E::load1(xr + j), m) * inv);
    }
    pdl_trigger();
}

template <typename T, int NT>
__global__ void __launch_bounds__(NT)
    softmax_bwd_wide(const T* __restrict__ y, int64_t ldy, const T* __restrict__ dy, int64_t lddy,
                     T* __restrict__ dx, int64_t lddx, int64_t N, int64_t D) {
    using E = Elt<T>;
    constexpr bool kComp = std::is_same<T, float>::value;
    __shared__ Acc2 red[NT / 32];
    pdl_wait();
    for (int64_t row = blockIdx.x; row < N; row += gridDim.x) {
        Acc2 s = acc2_zero();
        for (int64_t j = threadIdx.x; j < D; j += NT) {
            const float a = E::load1(dy + row * lddy + j), b = E::load1(y + row * ldy + j);
            if constexpr (kComp)
                acc2_fma(s, a, b);
            else
                s.hi = fmaf(a, b, s.hi);
        }
        s = group_sum_acc2<NT>(s, red);
        const float sv = s.hi + s.lo;
        for (int64_t j = threadIdx.x; j < D; j += NT) {
            const float yv = E::load1(y + row * ldy + j);
            E::store1(dx + row * lddx + j, yv * (E::load1(dy + row * lddy + j) - sv));
        }
    }
    pdl_trigger();
}

// ---------------------------------------------------------------------------
// Cluster path (16-byte aligned rows wider than the row path holds): one
// thread-block cluster of CS CTAs takes one row per iteration (grid-stride
// over rows by cluster).  The CTA of rank r owns the row's chunks
// [r·NT·CPT, (r+1)·NT·CPT), CPT = 4 chunks a thread, staged S rows ahead into
// the thread's private shared-memory slots with cp.async, so each CTA reads
// its slice of x (y, dy) once and writes y (dx) once.
//
// One exchange a row.  Each warp reduces its own part of the slice (xor
// butterfly) and pushes the warp's entry into every CTA of the cluster
// (WarpPush: st.async completing on the receiver's mbarrier, no cluster
// barrier in the loop); warp 0 of every CTA then combines all CS·NT/32
// entries from its own shared memory, lane ℓ taking entries ℓ, ℓ+32, …, in
// that order and then across lanes (xor butterfly), and hands the result to
// the other warps through shared memory and a CTA barrier, so every CTA
// derives the same bits of the row statistic.  The forward publishes (m_w, s_w): the
// warp's maximum and its sum of exp(x − m_w); the row sum is
// Σ_w s_w·exp(m_w − M), M = max_w m_w, and y = exp(x − m_w)·(exp(m_w − M)/sum)
// (the combination of partial softmax sums by rescaling, as in online
// softmax).  The backward publishes the warp's part of Σ dy·y.  Every CTA of
// a cluster runs the same number of rows (it depends only on the cluster's
// index), hence the same exchanges.
constexpr int kClusterCPT = 4;
constexpr int kClusterCPT5 = 5;  // the forward's wider CTAs (see softmax_fwd_cluster_t)

// Waits of the cluster exchanges that ran out (see WarpPush); zero unless
// the exchange protocol failed.
__device__ unsigned g_softmax_wait_timeouts;

template <int NT>
using SoftmaxPush = WarpPush<NT / 32, kClusterMaxCS*(NT / 32), 1>;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL_MASK, v, off));
    return v;
}

// exp(a − b) for the combination of partial sums: the binary32 form of the
// elements (exactly split difference) or the base-2 form of 16-bit rows.
template <bool Comp>
__device__ __forceinline__ float rescale(float a, float b) {
    if constexpr (Comp) return exp_diff<false>(a, b);
    else return exp2_approx(fmaf(a, kLog2e, -b * kLog2e));
}

template <typename T, int NT, int S, bool U, int CPT>
__global__ void __launch_bounds__(NT, (CPT > kClusterCPT ? 768 : 1024) / NT)
    softmax_fwd_cluster(const T* __restrict__ x, int64_t ldx, T* __restrict__ y, int64_t ldy,
                        int64_t N, int D) {
    using E = Elt<T>;
    constexpr int V = E::V, W = NT / 32;
    constexpr bool kComp = std::is_same<T, float>::value;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Raw16* slots = reinterpret_cast<Raw16*>(smem_raw);  // [S][CPT][NT]
    __shared__ __align__(16) float4 xbuf[2][kClusterMaxCS * W][1];
    __shared__ __align__(8) uint64_t xbar[2];
    __shared__ float2 res[2];  // (row maximum, 1/sum), by turn parity
    SoftmaxPush<NT> xp{xbuf, xbar, &g_softmax_wait_timeouts, 0u, true};
    xp.init();
    cluster_sync();
    const int l = (int)cluster_ctarank() * NT * CPT + (int)threadIdx.x;  // chunk l + c·NT
    const int lane = threadIdx.x & 31;
    const int total = (int)cluster_nctarank() * W;
    const int64_t cid = cluster_id_x(), ncl = cluster_count_x();
    const int64_t iters = cid < N ? (N - 1 - cid) / ncl + 1 : 0;
    pdl_wait();
#pragma unroll
    for (int k = 0; k < S - 1; k++) {
        if (k < iters) stage_row<T, NT, CPT, NT, U>(slots + k * CPT * NT, x, ldx, cid + k * ncl, N, D, l);
        cp_async_commit();
    }
    for (int64_t k = 0; k < iters; k++) {
        cp_async_wait<S - 2>();
        const int64_t nk = k + S - 1;
        if (nk < iters)
            stage_row<T, NT, CPT, NT, U>(slots + (nk % S) * CPT * NT, x, ldx, cid + nk * ncl, N, D, l);
        cp_async_commit();
        const int64_t row = cid + k * ncl;
        Raw16* cur = slots + (k % S) * CPT * NT;
        const Win<T, U> win{win_off<T, U>(x + row * ldx), D};
        // the warp's maximum and its sum of exp(x − m_w)
        float f[CPT][V];
        float m = -INFINITY;
#pragma unroll
        for (int c = 0; c < CPT; c++) {
            const int cc = l + c * NT;
            if (win.has(cc)) {
                if constexpr (!kComp) {
                    // an edge chunk gets −inf outside the row (in the
                    // thread's own slot), whose exponential is 0
                    Raw16 r = cur[c * NT + threadIdx.x];
                    if (!win.full(cc)) {
                        r = mask_ninf<T>(r, win.off - cc * V, win.off + D - cc * V);
                        cur[c * NT + threadIdx.x] = r;
                    }
                    m = fmaxf(m, chunk_max16<T>(r));
                } else {
                    E::widen(cur[c * NT + threadIdx.x], f[c]);
                    if (!win.full(cc))  // edge chunk: −inf outside the row
#pragma unroll
                        for (int v = 0; v < V; v++)
                            if (!win.elt(cc, v)) f[c][v] = -INFINITY;
#pragma unroll
                    for (int v = 0; v < V; v++) m = fmaxf(m, f[c][v]);
                }
            }
        }
        m = warp_max(m);
        // a warp whose elements are all −inf (masked) shifts by 0: its
        // exponentials and its sum are then 0, and its entry is skipped
        if (m == -INFINITY) m = 0.f;
        Acc2 s = acc2_zero();
        if constexpr (!kComp) {
            const float ms = m * kLog2e;
#pragma unroll
            for (int c = 0; c < CPT; c++) {
                E::widen(cur[c * NT + threadIdx.x], f[c]);
                const bool ok = win.has(l + c * NT);
#pragma unroll
                for (int v = 0; v < V; v++) {
                    f[c][v] = ok ? exp2_approx(fmaf(f[c][v], kLog2e, -ms)) : 0.f;
                    s.hi += f[c][v];
                }
            }
            s.hi = group_sum<32>(s.hi);
        } else {
#pragma unroll
            for (int c = 0; c < CPT; c++) {
                const bool ok = win.has(l + c * NT);
#pragma unroll
                for (int v = 0; v < V; v++) {
                    // exp(−inf − m) = 0 outside the row
                    f[c][v] = ok ? exp_diff<false>(f[c][v], m) : 0.f;
                    add_to<true>(s, f[c][v]);
                }
            }
            s = group_sum2<32>(s);
        }
        const float4 mine[1] = {make_float4(m, s.hi, s.lo, 0.f)};
        const unsigned turn = xp.template push<1>(mine);
        float2* out = &res[turn & 1u];
        if (threadIdx.x < 32) {  // warp 0 combines the turn's entries
            const float4(*buf)[1] = xp.wait(turn);
            // every (rank, warp) entry j = rank·W + warp, from this CTA's buffer
            float M = -INFINITY;
            for (int j = lane; j < total; j += 32) M = fmaxf(M, buf[j][0].x);
            M = warp_max(M);
            Acc2 t = acc2_zero();
            for (int j = lane; j < total; j += 32) {
                const float4 en = buf[j][0];
                if (en.y > 0.f) {  // skip warps without a finite element
                    const float g = rescale<kComp>(en.x, M);
                    if constexpr (kComp)
                        acc2_fma(t, __fadd_rn(en.y, en.z), g);
                    else
                        t.hi = fmaf(en.y, g, t.hi);
                }
            }
            float inv;
            if constexpr (kComp) {
                t = group_sum2<32>(t);
                inv = 1.0f / (t.hi + t.lo);
            } else {
                inv = 1.0f / group_sum<32>(t.hi);
            }
            if (lane == 0) *out = make_float2(M, inv);
        }
        __syncthreads();
        const float2 Mi = *out;
        const float sc = rescale<kComp>(m, Mi.x) * Mi.y;
        T* yrow = y + row * ldy;
#pragma unroll
        for (int c = 0; c < CPT; c++) {
            const int cc = l + c * NT;
            if (win.has(cc)) {
                float o[V];
#pragma unroll
                for (int v = 0; v < V; v++) o[v] = f[c][v] * sc;
                store_chunk<T, U>(yrow, win, cc, o);
            }
        }
    }
    cp_async_wait<0>();
    cluster_sync();
    pdl_trigger();
}

template <typename T, int NT, int S, bool U>
__global__ void __launch_bounds__(NT)
    softmax_bwd_cluster(const T* __restrict__ y, int64_t ldy, const T* __restrict__ dy,
                        int64_t lddy, T* __restrict__ dx, int64_t lddx, int64_t N, int D) {
    using E = Elt<T>;
    constexpr int V = E::V, CPT = kClusterCPT, W = NT / 32;
    constexpr bool kComp = std::is_same<T, float>::value;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Raw16* ys = reinterpret_cast<Raw16*>(smem_raw);  // [S][CPT][NT]
    Raw16* gs = ys + S * CPT * NT;                    // [S][CPT][NT]
    __shared__ __align__(16) float4 xbuf[2][kClusterMaxCS * W][1];
    __shared__ __align__(8) uint64_t xbar[2];
    __shared__ float res[2];  // Σ dy·y, by turn parity
    SoftmaxPush<NT> xp{xbuf, xbar, &g_softmax_wait_timeouts, 0u, true};
    xp.init();
    cluster_sync();
    const int l = (int)cluster_ctarank() * NT * CPT + (int)threadIdx.x;
    const int lane = threadIdx.x & 31;
    const int total = (int)cluster_nctarank() * W;
    const int64_t cid = cluster_id_x(), ncl = cluster_count_x();
    const int64_t iters = cid < N ? (N - 1 - cid) / ncl + 1 : 0;
    pdl_wait();
#pragma unroll
    for (int k = 0; k < S - 1; k++) {
        if (k < iters) {
            stage_row<T, NT, CPT, NT, U>(ys + k * CPT * NT, y, ldy, cid + k * ncl, N, D, l);
            stage_row<T, NT, CPT, NT, U>(gs + k * CPT * NT, dy, lddy, cid + k * ncl, N, D, l);
        }
        cp_async_commit();
    }
    for (int64_t k = 0; k < iters; k++) {
        cp_async_wait<S - 2>();
        const int64_t nk = k + S - 1;
        if (nk < iters) {
            stage_row<T, NT, CPT, NT, U>(ys + (nk % S) * CPT * NT, y, ldy, cid + nk * ncl, N, D, l);
            stage_row<T, NT, CPT, NT, U>(gs + (nk % S) * CPT * NT, dy, lddy, cid + nk * ncl, N, D, l);
        }
        cp_async_commit();
        const int64_t row = cid + k * ncl;
        const Raw16* cy = ys + (k % S) * CPT * NT;
        const Raw16* cg = gs + (k % S) * CPT * NT;
        const Win<T, U> win{win_off<T, U>(y + row * ldy), D};
        // y and dy of chunk cc, zero outside the row
        auto load = [&](int c, int cc, float (&fy)[V], float (&fg)[V]) {
            E::widen(cy[c * NT + threadIdx.x], fy);
            E::widen(cg[c * NT + threadIdx.x], fg);
            if (!win.full(cc))
#pragma unroll
                for (int v = 0; v < V; v++)
                    if (!win.elt(cc, v)) fy[v] = fg[v] = 0.f;
        };
        Acc2 s = acc2_zero();
#pragma unroll
        for (int c = 0; c < CPT; c++) {
            const int cc = l + c * NT;
            if (win.has(cc)) {
                float fy[V], fg[V];
                load(c, cc, fy, fg);
#pragma unroll
                for (int v = 0; v < V; v++) {
                    if constexpr (kComp)
                        acc2_fma(s, fg[v], fy[v]);
                    else
                        s.hi = fmaf(fg[v], fy[v], s.hi);
                }
            }
        }
        if constexpr (kComp)
            s = group_sum2<32>(s);
        else
            s.hi = group_sum<32>(s.hi);
        const float4 mine[1] = {make_float4(s.hi, s.lo, 0.f, 0.f)};
        const unsigned turn = xp.template push<1>(mine);
        float* out = &res[turn & 1u];
        if (threadIdx.x < 32) {  // warp 0 combines the turn's entries
            const float4(*buf)[1] = xp.wait(turn);
            Acc2 t = acc2_zero();
            for (int j = lane; j < total; j += 32) {
                const float4 o = buf[j][0];
                if constexpr (kComp)
                    t = acc2_add(t, Acc2{o.x, o.y});
                else
                    t.hi += o.x;
            }
            float r;
            if constexpr (kComp) {
                t = group_sum2<32>(t);
                r = t.hi + t.lo;
            } else {
                r = group_sum<32>(t.hi);
            }
            if (lane == 0) *out = r;
        }
        __syncthreads();
        const float sv = *out;
        T* dxrow = dx + row * lddx;
#pragma unroll
        for (int c = 0; c < CPT; c++) {
            const int cc = l + c * NT;
            if (win.has(cc)) {
                float fy[V], fg[V], o[V];
                load(c, cc, fy, fg);
#pragma unroll
                for (int v = 0; v < V; v++) o[v] = fy[v] * (fg[v] - sv);
                store_chunk<T, U>(dxrow, win, cc, o);
            }
        }
    }
    cp_async_wait<0>();
    cluster_sync();
    pdl_trigger();
}

// ---------------------------------------------------------------------------
// Two-pass cluster path (rows wider than the cluster path holds: more than
// 32,768 chunks).  A cluster of CS CTAs takes a row; the CTA of rank r owns
// the chunks [r·SL, (r+1)·SL), SL = ⌈Dc/CS⌉, which its threads stream from
// memory twice, a few chunks a thread a batch: the first pass forms each
// thread's maximum and its sum of exp(x − m) (rescaled when the maximum
// grows; forward) or its part of Σ dy·y (backward), the warps exchange these
// as on the cluster path, and the second pass reads the slice again and
// writes y (dx).  Only the clusters' rows in flight (tens of MB) are read
// between the passes, so the second read is served by L2; x (y, dy) is read
// from HBM once.  Bulk L2 prefetches of the cluster's next row measured slower
// once clusters were small and many (bf16 [1024, 524288]: 3957 GB/s with,
// 5461 without; the backward's likewise, earlier).  Elements outside the row
// (windowed edges, the tail of the last slice) enter as −inf (forward) or 0
// (backward).
constexpr int kTwoPassNT = 256, kTwoPassU = 4;
// CTAs a cluster (a row's slices).  Measured at bf16 [1024, 524288], forward
// GB/s: 5046 / 5490 / 4785 with clusters of 16 / 8 / 4; more resident
// clusters keep more loads in flight, fewer CTAs a cluster make each exchange
// cheaper, and the rows in flight must stay in L2 for the second pass.  The
// backward (s4, fp32 [2048, 262144]): 4745 / 5278 / 4309 with clusters of
// 16 / 8 (two CTAs an SM) / 4 (three).  The binary32 forward chooses its
// cluster size at launch (two_pass_cs).
template <typename T, bool Fwd>
constexpr int kTwoPassCS = 8;

// The raw chunks c0 + b + u·NT (u < NU) of a row: the row's own 16-byte
// blocks, zeros for chunks past the slice or the row.
template <typename T, bool U, int NU>
__device__ __forceinline__ void load_batch(Raw16 (&r)[NU], const T* row_start, const Win<T, U>& w,
                                           int c0, int b, int SL, uint64_t pol) {
#pragma unroll
    for (int u = 0; u < NU; u++) {
        const int c = b + u * kTwoPassNT;
        r[u] = (c < SL && w.has(c0 + c)) ? ld_policy(row_start + w.at(c0 + c), pol) : raw_zero();
    }
}

// max(a, b, c) in one instruction (sm_100 and later; a NaN operand is
// ignored as by fmaxf).
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Whether every chunk b + u·NT (u < NU) of a batch lies inside the slice and,
// for aligned rows, inside the row: such a batch needs no per-chunk masking.
template <typename T, bool U, int NU>
__device__ __forceinline__ bool full_batch(const Win<T, U>& w, int c0, int b, int SL) {
    const int last = b + (NU - 1) * kTwoPassNT;
    return !U && last < SL && w.has(c0 + last);
}

// Chunk c of the slice (row chunk cc = c0 + c) widened, with −inf (Fwd) or 0
// outside the slice and the row.
template <typename T, bool U, bool Fwd>
__device__ __forceinline__ void widen_chunk(const Raw16& r, const Win<T, U>& w, int c, int cc,
                                            int SL, float (&f)[Elt<T>::V]) {
    using E = Elt<T>;
    if (c < SL && w.has(cc)) {
        E::widen(r, f);
        if (!w.full(cc))
#pragma unroll
            for (int v = 0; v < E::V; v++)
                if (!w.elt(cc, v)) f[v] = Fwd ? -INFINITY : 0.f;
    } else {
#pragma unroll
        for (int v = 0; v < E::V; v++) f[v] = Fwd ? -INFINITY : 0.f;
    }
}

// The loads are pipelined in registers: each thread holds the raw chunks of
// its next batch while it computes the current one; the last batch of the
// first pass fetches the second pass's first batch (before the exchange),
// and the last batch of the second pass the next row's first batch.
template <typename T, bool U>
__global__ void __launch_bounds__(kTwoPassNT, std::is_same<T, float>::value ? 4 : 3)
    softmax_fwd_cluster2(const T* __restrict__ x, int64_t ldx, T* __restrict__ y, int64_t ldy,
                         int64_t N, int D, int SL) {
    using E = Elt<T>;
    constexpr int V = E::V, NT = kTwoPassNT, W = NT / 32, UU = kTwoPassU, STEP = NT * UU;
    constexpr bool kComp = std::is_same<T, float>::value;
    __shared__ __align__(16) float4 xbuf[2][kClusterMaxCS * W][1];
    __shared__ __align__(8) uint64_t xbar[2];
    __shared__ float2 res[2];  // (row maximum, 1/sum), by turn parity
    SoftmaxPush<NT> xp{xbuf, xbar, &g_softmax_wait_timeouts, 0u, true};
    xp.init();
    cluster_sync();
    const int lane = threadIdx.x & 31;
    const int total = (int)cluster_nctarank() * W;
    const int c0 = (int)cluster_ctarank() * SL;  // this CTA's chunks [c0, c0 + SL)
    const int64_t cid = cluster_id_x(), ncl = cluster_count_x();
    pdl_wait();
    // first-pass reads keep their lines in L2 for the second (evict_last);
    // the second pass is their last use (evict_first)
    const uint64_t keep = l2_evict_last(), last = l2_evict_first();
    Raw16 nb[UU];  // the next batch's raw chunks
    if (cid < N) {
        const T* x0 = x + cid * ldx;
        load_batch<T, U, UU>(nb, x0, Win<T, U>{win_off<T, U>(x0), D}, c0, threadIdx.x, SL, keep);
    }
    for (int64_t row = cid; row < N; row += ncl) {
        const T* xr = x + row * ldx;
        const Win<T, U> win{win_off<T, U>(xr), D};
        // pass 1: this thread's maximum m and Σ exp(x − m) (binary32 rows:
        // two compensated lanes in packed f32x2 arithmetic, added together at
        // the end)
        float m = -INFINITY;
        Acc2 s = acc2_zero();
        Acc2x2 s2{0ull, 0ull};
        for (int b = threadIdx.x; b < SL; b += STEP) {
            Raw16 cur[UU];
#pragma unroll
            for (int u = 0; u < UU; u++) cur[u] = nb[u];
            // the next batch, or the second pass's first
            if (b + STEP < SL)
                load_batch<T, U, UU>(nb, xr, win, c0, b + STEP, SL, keep);
            else
                load_batch<T, U, UU>(nb, xr, win, c0, threadIdx.x, SL, last);
            const bool full = full_batch<T, U, UU>(win, c0, b, SL);
            // chunk u of the batch, widened (masked only when the batch is not full)
            auto chunk = [&](int u, float (&f)[V]) {
                if (full)
                    E::widen(cur[u], f);
                else
                    widen_chunk<T, U, true>(cur[u], win, b + u * NT, c0 + b + u * NT, SL, f);
            };
            float mb = m;
#pragma unroll
            for (int u = 0; u < UU; u++) {
                float f[V];
                chunk(u, f);
#pragma unroll
                for (int v = 0; v + 1 < V; v += 2) mb = max3(mb, f[v], f[v + 1]);
                if constexpr (V % 2) mb = fmaxf(mb, f[V - 1]);
            }
            if (mb == -INFINITY) continue;  // nothing finite yet
            if constexpr (kComp) {
                if (mb > m) {  // rescale both lanes to the new maximum (0 while m = −inf)
                    const float g = exp_diff_f32(m, mb);
                    const uint64_t g2 = f2_pack(g, g), ng2 = f2_pack(-g, -g);
                    const uint64_t nhi = f2_mul(s2.hi, ng2);  // −fl(hi·g)
                    s2.lo = f2_fma(s2.lo, g2, f2_fma(s2.hi, g2, nhi));
                    s2.hi = f2_mul(s2.hi, g2);
                }
                m = mb;
                const uint64_t nm2 = f2_pack(-m, -m);
                // the batch's exponentials, two lanes a value, added as a
                // pairwise tree (within 3·2^-24 of the batch's sum, every term
                // being positive), then into each lane's running sum by TwoSum
                constexpr int NP = UU * V / 2;
                static_assert((NP & (NP - 1)) == 0, "a power of two");
                uint64_t e[NP];
#pragma unroll
                for (int u = 0; u < UU; u++) {
                    float f[V];
                    chunk(u, f);
#pragma unroll
                    for (int q = 0; q < V / 2; q++)
                        e[u * (V / 2) + q] = exp_sum_f32x2(f2_pack(f[2 * q], f[2 * q + 1]), nm2);
                }
#pragma unroll
                for (int w = NP / 2; w >= 1; w /= 2)
#pragma unroll
                    for (int i = 0; i < w; i++) e[i] = f2_add(e[i], e[i + w]);
                const uint64_t t = f2_add(s2.hi, e[0]);
                const uint64_t bp = f2_sub(t, s2.hi);
                const uint64_t err = f2_add(f2_sub(s2.hi, f2_sub(t, bp)), f2_sub(e[0], bp));
                s2.hi = t;
                s2.lo = f2_add(s2.lo, err);
            } else {
                if (mb > m && s.hi != 0.f) s.hi *= rescale<kComp>(m, mb);
                m = mb;
#pragma unroll
                for (int u = 0; u < UU; u++) {
                    float f[V];
                    chunk(u, f);
#pragma unroll
                    for (int v = 0; v < V; v++)
                        add_to<kComp>(s, exp2_approx(fmaf(f[v], kLog2e, -m * kLog2e)));
                }
            }
        }
        if constexpr (kComp) {
            Acc2 l0, l1;
            acc2x2_unpack(s2, l0, l1);
            s = acc2_add(l0, l1);
        }
        // the warp's maximum and its sum relative to it
        const float mw = warp_max(m);
        Acc2 sw = acc2_zero();
        if (s.hi > 0.f) {
            const float g = rescale<kComp>(m, mw);
            if constexpr (kComp) {
                acc2_fma(sw, __fadd_rn(s.hi, s.lo), g);
            } else {
                sw.hi = s.hi * g;
            }
        }
        if constexpr (kComp)
            sw = group_sum2<32>(sw);
        else
            sw.hi = group_sum<32>(sw.hi);
        const float4 mine[1] = {make_float4(mw == -INFINITY ? 0.f : mw, sw.hi, sw.lo, 0.f)};
        const unsigned turn = xp.template push<1>(mine);
        float2* out = &res[turn & 1u];
        if (threadIdx.x < 32) {  // warp 0 combines the turn's entries
            const float4(*buf)[1] = xp.wait(turn);
            float M = -INFINITY;
            for (int j = lane; j < total; j += 32)
                if (buf[j][0].y > 0.f) M = fmaxf(M, buf[j][0].x);
            M = warp_max(M);
            Acc2 t = acc2_zero();
            for (int j = lane; j < total; j += 32) {
                const float4 en = buf[j][0];
                if (en.y > 0.f) {  // skip warps without a finite element
                    const float g = rescale<kComp>(en.x, M);
                    if constexpr (kComp)
                        acc2_fma(t, __fadd_rn(en.y, en.z), g);
                    else
                        t.hi = fmaf(en.y, g, t.hi);
                }
            }
            float inv;
            if constexpr (kComp) {
                t = group_sum2<32>(t);
                inv = 1.0f / (t.hi + t.lo);
            } else {
                inv = 1.0f / group_sum<32>(t.hi);
            }
            if (lane == 0) *out = make_float2(M, inv);
        }
        __syncthreads();
        const float2 Mi = *out;
        // pass 2: y = exp(x − M)/sum, the slice read again (from L2)
        T* yr = y + row * ldy;
        for (int b = threadIdx.x; b < SL; b += STEP) {
            Raw16 cur[UU];
#pragma unroll
            for (int u = 0; u < UU; u++) cur[u] = nb[u];
            if (b + STEP < SL) {
                load_batch<T, U, UU>(nb, xr, win, c0, b + STEP, SL, last);
            } else if (row + ncl < N) {  // the next row's first batch
                const T* xn = xr + ncl * ldx;
                load_batch<T, U, UU>(nb, xn, Win<T, U>{win_off<T, U>(xn), D}, c0, threadIdx.x, SL,
                                     keep);
            }
            const bool full = full_batch<T, U, UU>(win, c0, b, SL);
#pragma unroll
            for (int u = 0; u < UU; u++) {
                const int c = b + u * NT, cc = c0 + c;
                if (full || (c < SL && win.has(cc))) {
                    float f[V], o[V];
                    if (full)
                        E::widen(cur[u], f);
                    else
                        widen_chunk<T, U, true>(cur[u], win, c, cc, SL, f);
                    if constexpr (kComp) {
                        const uint64_t nM2 = f2_pack(-Mi.x, -Mi.x), inv2 = f2_pack(Mi.y, Mi.y);
#pragma unroll
                        for (int q = 0; q < V / 2; q++)
                            f2_unpack(f2_mul(exp_diff_f32x2(f2_pack(f[2 * q], f[2 * q + 1]), nM2),
                                             inv2),
                                      o[2 * q], o[2 * q + 1]);
                    } else {
#pragma unroll
                        for (int v = 0; v < V; v++)
                            o[v] = exp2_approx(fmaf(f[v], kLog2e, -Mi.x * kLog2e)) * Mi.y;
                    }
                    store_chunk<T, U>(yr, win, cc, o);
                }
            }
        }
    }
    cluster_sync();
    pdl_trigger();
}

template <typename T, bool U>
__global__ void __launch_bounds__(kTwoPassNT, 2)
    softmax_bwd_cluster2(const T* __restrict__ y, int64_t ldy, const T* __restrict__ dy,
                         int64_t lddy, T* __restrict__ dx, int64_t lddx, int64_t N, int D,
                         int SL) {
    using E = Elt<T>;
    // 16 elements of y and of dy a thread a batch
    constexpr int V = E::V, NT = kTwoPassNT, W = NT / 32, UU = 16 / V, STEP = NT * UU;
    constexpr bool kComp = std::is_same<T, float>::value;
    __shared__ __align__(16) float4 xbuf[2][kClusterMaxCS * W][1];
    __shared__ __align__(8) uint64_t xbar[2];
    __shared__ float res[2];  // Σ dy·y, by turn parity
    SoftmaxPush<NT> xp{xbuf, xbar, &g_softmax_wait_timeouts, 0u, true};
    xp.init();
    cluster_sync();
    const int lane = threadIdx.x & 31;
    const int total = (int)cluster_nctarank() * W;
    const int c0 = (int)cluster_ctarank() * SL;
    const int64_t cid = cluster_id_x(), ncl = cluster_count_x();
    pdl_wait();
    const uint64_t keep = l2_evict_last(), last = l2_evict_first();  // as in the forward
    Raw16 ny[UU], ng[UU];  // the next batch's raw chunks of y and dy
    if (cid < N) {
        const T* y0 = y + cid * ldy;
        const Win<T, U> w0{win_off<T, U>(y0), D};
        load_batch<T, U, UU>(ny, y0, w0, c0, threadIdx.x, SL, keep);
        load_batch<T, U, UU>(ng, dy + cid * lddy, w0, c0, threadIdx.x, SL, keep);
    }
    for (int64_t row = cid; row < N; row += ncl) {
        const T* yr = y + row * ldy;
        const T* gr = dy + row * lddy;
        const Win<T, U> win{win_off<T, U>(yr), D};
        // pass 1: this thread's part of Σ dy·y
        Acc2 s = acc2_zero();
        for (int b = threadIdx.x; b < SL; b += STEP) {
            Raw16 cy[UU], cg[UU];
#pragma unroll
            for (int u = 0; u < UU; u++) {
                cy[u] = ny[u];
                cg[u] = ng[u];
            }
            // the next batch, or the second pass's first
            const bool more = b + STEP < SL;
            const int bn = more ? b + STEP : (int)threadIdx.x;
            load_batch<T, U, UU>(ny, yr, win, c0, bn, SL, more ? keep : last);
            load_batch<T, U, UU>(ng, gr, win, c0, bn, SL, more ? keep : last);
#pragma unroll
            for (int u = 0; u < UU; u++) {
                float fy[V], fg[V];
                widen_chunk<T, U, false>(cy[u], win, b + u * NT, c0 + b + u * NT, SL, fy);
                widen_chunk<T, U, false>(cg[u], win, b + u * NT, c0 + b + u * NT, SL, fg);
#pragma unroll
                for (int v = 0; v < V; v++) {
                    if constexpr (kComp)
                        acc2_fma(s, fg[v], fy[v]);
                    else
                        s.hi = fmaf(fg[v], fy[v], s.hi);
                }
            }
        }
        if constexpr (kComp)
            s = group_sum2<32>(s);
        else
            s.hi = group_sum<32>(s.hi);
        const float4 mine[1] = {make_float4(s.hi, s.lo, 0.f, 0.f)};
        const unsigned turn = xp.template push<1>(mine);
        float* out = &res[turn & 1u];
        if (threadIdx.x < 32) {  // warp 0 combines the turn's entries
            const float4(*buf)[1] = xp.wait(turn);
            Acc2 t = acc2_zero();
            for (int j = lane; j < total; j += 32) {
                const float4 o = buf[j][0];
                if constexpr (kComp)
                    t = acc2_add(t, Acc2{o.x, o.y});
                else
                    t.hi += o.x;
            }
            float r;
            if constexpr (kComp) {
                t = group_sum2<32>(t);
                r = t.hi + t.lo;
            } else {
                r = group_sum<32>(t.hi);
            }
            if (lane == 0) *out = r;
        }
        __syncthreads();
        const float sv = *out;
        // pass 2: dx = y·(dy − Σ dy·y), y and dy read again (from L2)
        T* dxr = dx + row * lddx;
        for (int b = threadIdx.x; b < SL; b += STEP) {
            Raw16 cy[UU], cg[UU];
#pragma unroll
            for (int u = 0; u < UU; u++) {
                cy[u] = ny[u];
                cg[u] = ng[u];
            }
            if (b + STEP < SL) {
                load_batch<T, U, UU>(ny, yr, win, c0, b + STEP, SL, last);
                load_batch<T, U, UU>(ng, gr, win, c0, b + STEP, SL, last);
            } else if (row + ncl < N) {  // the next row's first batch
                const T* yn = yr + ncl * ldy;
                const Win<T, U> wn{win_off<T, U>(yn), D};
                load_batch<T, U, UU>(ny, yn, wn, c0, threadIdx.x, SL, keep);
                load_batch<T, U, UU>(ng, gr + ncl * lddy, wn, c0, threadIdx.x, SL, keep);
            }
#pragma unroll
            for (int u = 0; u < UU; u++) {
                const int c = b + u * NT, cc = c0 + c;
                if (c < SL && win.has(cc)) {
                    float fy[V], fg[V], o[V];
                    widen_chunk<T, U, false>(cy[u], win, c, cc, SL, fy);
                    widen_chunk<T, U, false>(cg[u], win, c, cc, SL, fg);
#pragma unroll
                    for (int v = 0; v < V; v++) o[v] = fy[v] * (fg[v] - sv);
                    store_chunk<T, U>(dxr, win, cc, o);
                }
            }
        }
    }
    cluster_sync();
    pdl_trigger();
}

// ---------------------------------------------------------------------------
static inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
static inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
static inline int next_pow2(int64_t v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

constexpr int kSoftmaxRowChunks = 2048;  // rows of up to 32 KB stay in registers

// Raise a kernel's dynamic shared-memory limit (idempotent, cheap); done from
// 32 KB up because the kernels' static shared memory counts against the
// default 48 KB too.
static cudaError_t allow_smem_sm(const void* kernel, size_t bytes) {
    if (bytes < 32 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// Row-path shapes: TPR threads per row, CPT chunks per thread, 256-thread
// CTAs; S stages of staged rows (fewer for wide rows to bound shared memory).
template <int TPR, int CPT, int S, typename F>
static cudaError_t with_rows(int64_t N, F&& go) {
    constexpr int NT = 256;
    constexpr int R = NT / TPR;
    const int64_t grid = std::min<int64_t>(cdiv(N, R), 8 * kDesignSMs);
    return go(std::integral_constant<int, TPR>{}, std::integral_constant<int, CPT>{},
              std::integral_constant<int, S>{}, dim3((unsigned)grid), dim3(NT));
}

// Measured on GB300 for rows of 512 chunks (4096 bf16): forward 128 threads x
// 4 chunks, backward 64 x 8, two stages; other widths follow the same idea.
// A windowed row spans one chunk more than its aligned width when it starts
// inside a 16-byte block; widths just past a power of two then take one more
// chunk a thread rather than twice the threads.
template <bool Fwd, bool U = false, typename F>
static cudaError_t dispatch_rows(int64_t Dv, int64_t N, F&& go) {
    if constexpr (U) {
        if (Dv > 64 && Dv <= 96) return with_rows<32, 3, 3>(N, go);
        if (Dv > 128 && Dv <= 160) return with_rows<32, 5, 3>(N, go);
        if (Dv > 256 && Dv <= 288) return with_rows<32, 9, 2>(N, go);
        if (Fwd && Dv > 512 && Dv <= 640) return with_rows<128, 5, 2>(N, go);
        if (!Fwd && Dv > 512 && Dv <= 576) return with_rows<64, 9, 2>(N, go);
        if (Dv > 1024 && Dv <= 1152) return with_rows<128, 9, 2>(N, go);
    }
    if (Dv <= 32) {
        switch (next_pow2(Dv)) {
            case 1: return with_rows<1, 1, 4>(N, go);
            case 2: return with_rows<2, 1, 4>(N, go);
            case 4: return with_rows<4, 1, 4>(N, go);
            case 8: return with_rows<8, 1, 4>(N, go);
            case 16: return with_rows<16, 1, 4>(N, go);
            default: return with_rows<32, 1, 4>(N, go);
        }
    }
    if (Dv <= 64) return with_rows<32, 2, 4>(N, go);
    if (Dv <= 128) return with_rows<32, 4, 3>(N, go);
    if (Dv <= 256) return with_rows<32, 8, 2>(N, go);
    if (Dv <= 512) {
        if constexpr (Fwd) return with_rows<128, 4, 2>(N, go);
        else return with_rows<64, 8, 2>(N, go);
    }
    if (Dv <= 1024) return with_rows<128, 8, 2>(N, go);
    return with_rows<256, 8, 2>(N, go);
}

// Cluster shapes: a CTA of NT threads holds NT·4 chunks of a row; rows of up
// to 16 CTAs of 256 threads (16,384 chunks, 256 KB) take clusters of
// 256-thread CTAs, wider rows 512-thread CTAs, up to 16 a cluster (32,768
// chunks, 512 KB).  Against 512-thread CTAs for rows over 8192 chunks, the
// smaller CTAs measured (bf16 [8192, 100000]) 4516 -> 5123 GB/s forward and
// 4586 -> 6534 backward: the backward's staged y and dy then take 64 KB a CTA,
// three CTAs an SM instead of one.
constexpr int64_t kClusterRowChunks = (int64_t)kClusterMaxCS * 512 * kClusterCPT;

static void cluster_shape(int64_t Dc, int& nt, unsigned& cs) {
    nt = Dc <= 16 * 256 * kClusterCPT ? 256 : 512;
    cs = (unsigned)cdiv(Dc, (int64_t)nt * kClusterCPT);
}

// Launch `kernel` as clusters of cs CTAs, as many clusters as the device
// holds at once (at most one a row); returns cudaErrorNotSupported when no
// cluster of that shape fits, so that the caller falls back.
template <auto kernel, typename... Args>
static cudaError_t go_cluster(int nt, unsigned cs, size_t smem, int64_t N, cudaStream_t s,
                              Args&&... args) {
    int fit = 0;
    const cudaError_t e = cluster_fit<kernel>(cs, nt, smem, fit);
    if (e != cudaSuccess) return e;
    const unsigned clusters = (unsigned)std::min<int64_t>(N, fit);
    return launch_cluster(kernel, clusters, cs, dim3(nt), smem, s, std::forward<Args>(args)...);
}

template <typename T, bool U>
static cudaError_t softmax_fwd_cluster_t(const T* x, int64_t ldx, T* y, int64_t ldy, int64_t N,
                                         int64_t D, int64_t Dc, cudaStream_t s) {
    int nt;
    unsigned cs;
    cluster_shape(Dc, nt, cs);
    if (nt == 256) {
        constexpr int S = 3;
        // five chunks a thread (three CTAs an SM) where they fill the row's
        // CTAs better by more than 3%: a last CTA with only a few chunks
        // costs a whole CTA's exchange and residency.  Measured (bf16, GB/s,
        // four / five chunks): rows of 50,257 (windowed) 4648 / 5222, of
        // 50,264 5090 / 5718 (7 CTAs, the last with 139 chunks, / 5), of
        // 20,480 5600 / 6040; of 49,152 (6 full CTAs / 5 at 96%) 6292 / 6015.
        const unsigned cs5 = (unsigned)cdiv(Dc, (int64_t)256 * kClusterCPT5);
        const double fill4 = (double)Dc / ((double)cs * 256 * kClusterCPT),
                     fill5 = (double)Dc / ((double)cs5 * 256 * kClusterCPT5);
        if (fill5 > fill4 + 0.03)
            return go_cluster<softmax_fwd_cluster<T, 256, S, U, kClusterCPT5>>(
                256, cs5, (size_t)S * kClusterCPT5 * 256 * 16, N, s, x, ldx, y, ldy, N, (int)D);
        return go_cluster<softmax_fwd_cluster<T, 256, S, U, kClusterCPT>>(
            256, cs, (size_t)S * kClusterCPT * 256 * 16, N, s, x, ldx, y, ldy, N, (int)D);
    }
    constexpr int S = 2;
    return go_cluster<softmax_fwd_cluster<T, 512, S, U, kClusterCPT>>(
        512, cs, (size_t)S * kClusterCPT * 512 * 16, N, s, x, ldx, y, ldy, N, (int)D);
}

template <typename T, bool U>
static cudaError_t softmax_bwd_cluster_t(const T* y, int64_t ldy, const T* dy, int64_t lddy, T* dx,
                                         int64_t lddx, int64_t N, int64_t D, int64_t Dc,
                                         cudaStream_t s) {
    int nt;
    unsigned cs;
    cluster_shape(Dc, nt, cs);
    constexpr int S = 2;
    if (nt == 256)
        return go_cluster<softmax_bwd_cluster<T, 256, S, U>>(
            256, cs, (size_t)2 * S * kClusterCPT * 256 * 16, N, s, y, ldy, dy, lddy, dx, lddx, N,
            (int)D);
    return go_cluster<softmax_bwd_cluster<T, 512, S, U>>(
        512, cs, (size_t)2 * S * kClusterCPT * 512 * 16, N, s, y, ldy, dy, lddy, dx, lddx, N,
        (int)D);
}

// Two-pass cluster launches (rows over kClusterRowChunks chunks, D < 2^30).
// The binary32 forward's second pass reads its slice again from L2, so the
// rows in flight (one a resident cluster) should fit in it: the smallest
// cluster of 4, 8 or 16 CTAs whose resident rows hold at most this many
// bytes, else 16.  Measured (GB/s, fp32 rows of 140,000 / 262,144 /
// 1,048,576 columns; clusters of 4, 8, 16): 5120 / 4462 / 3431,
// 4682 / 5190 / 4271, 4440 / 4604 / 4651.
constexpr int64_t kTwoPassL2Rows = (int64_t)96 << 20;

template <auto kernel>
static unsigned two_pass_cs(int64_t N, int64_t row_bytes) {
    for (unsigned cs : {4u, 8u}) {
        int fit = 0;
        if (cluster_fit<kernel>(cs, kTwoPassNT, 0, fit) == cudaSuccess &&
            std::min<int64_t>(N, fit) * row_bytes <= kTwoPassL2Rows)
            return cs;
    }
    return 16u;
}

template <typename T, bool U>
static cudaError_t softmax_fwd_cluster2_t(const T* x, int64_t ldx, T* y, int64_t ldy, int64_t N,
                                          int64_t D, int64_t Dc, cudaStream_t s) {
    constexpr auto k = softmax_fwd_cluster2<T, U>;
    const unsigned cs = std::is_same<T, float>::value ? two_pass_cs<k>(N, D * (int64_t)sizeof(T))
                                                      : (unsigned)kTwoPassCS<T, true>;
    const int SL = (int)cdiv(Dc, cs);
    return go_cluster<k>(kTwoPassNT, cs, 0, N, s, x, ldx, y, ldy, N, (int)D, SL);
}

template <typename T, bool U>
static cudaError_t softmax_bwd_cluster2_t(const T* y, int64_t ldy, const T* dy, int64_t lddy,
                                          T* dx, int64_t lddx, int64_t N, int64_t D, int64_t Dc,
                                          cudaStream_t s) {
    const int SL = (int)cdiv(Dc, kTwoPassCS<T, false>);
    return go_cluster<softmax_bwd_cluster2<T, U>>(kTwoPassNT, kTwoPassCS<T, false>, 0, N, s, y, ldy,
                                                  dy, lddy, dx, lddx, N, (int)D, SL);
}

constexpr int64_t kTwoPassMaxD = (int64_t)1 << 30;

// Row layouts of the vector paths: aligned (every array's rows start on 16
// bytes, D a whole number of chunks), or windowed (U: the arrays' rows share
// their offset inside a 16-byte block, row by row).  Dc = chunks a row spans
// (at most, for windowed rows).
template <typename T>
static bool aligned_rows(const void* p, int64_t ld) {
    return aligned16(p) && (ld * (int64_t)sizeof(T)) % 16 == 0;
}
template <typename T>
static bool same_offsets(const void* a, int64_t lda, const void* b, int64_t ldb) {
    return (((uintptr_t)a - (uintptr_t)b) & 15u) == 0 &&
           ((lda - ldb) * (int64_t)sizeof(T)) % 16 == 0;
}

template <typename T, bool U>
static cudaError_t softmax_fwd_vec(const T* x, int64_t ldx, T* y, int64_t ldy, int64_t N,
                                   int64_t D, int64_t Dc, cudaStream_t s) {
    if (Dc <= kSoftmaxRowChunks) {
        return dispatch_rows<true, U>(Dc, N, [&](auto tpr, auto cpt, auto st, dim3 grid, dim3 block) {
            constexpr int TPR = decltype(tpr)::value, CPT = decltype(cpt)::value;
            constexpr int S = decltype(st)::value;
            auto k = softmax_fwd_rows<T, TPR, CPT, 256, S, U>;
            const size_t smem = RowStage<TPR, CPT, 256, S>::bytes(1);
            cudaError_t e = allow_smem_sm((const void*)k, smem);
            if (e != cudaSuccess) return e;
            return launch(k, grid, block, smem, s, true, x, ldx, y, ldy, N, (int)D);
        });
    }
    if (Dc <= kClusterRowChunks && N > 0) return softmax_fwd_cluster_t<T, U>(x, ldx, y, ldy, N, D, Dc, s);
    if (D < kTwoPassMaxD && N > 0) return softmax_fwd_cluster2_t<T, U>(x, ldx, y, ldy, N, D, Dc, s);
    return cudaErrorNotSupported;
}

template <typename T, bool U>
static cudaError_t softmax_bwd_vec(const T* y, int64_t ldy, const T* dy, int64_t lddy, T* dx,
                                   int64_t lddx, int64_t N, int64_t D, int64_t Dc, cudaStream_t s) {
    if (Dc <= kSoftmaxRowChunks) {
        return dispatch_rows<false, U>(Dc, N, [&](auto tpr, auto cpt, auto st, dim3 grid, dim3 block) {
            constexpr int TPR = decltype(tpr)::value, CPT = decltype(cpt)::value;
            constexpr int S = decltype(st)::value;
            auto k = softmax_bwd_rows<T, TPR, CPT, 256, S, U>;
            const size_t smem = RowStage<TPR, CPT, 256, S>::bytes(2);
            cudaError_t e = allow_smem_sm((const void*)k, smem);
            if (e != cudaSuccess) return e;
            return launch(k, grid, block, smem, s, true, y, ldy, dy, lddy, dx, lddx, N, (int)D);
        });
    }
    if (Dc <= kClusterRowChunks && N > 0)
        return softmax_bwd_cluster_t<T, U>(y, ldy, dy, lddy, dx, lddx, N, D, Dc, s);
    if (D < kTwoPassMaxD && N > 0)
        return softmax_bwd_cluster2_t<T, U>(y, ldy, dy, lddy, dx, lddx, N, D, Dc, s);
    return cudaErrorNotSupported;
}

template <typename T>
static cudaError_t softmax_fwd_t(const T* x, int64_t ldx, T* y, int64_t ldy, int64_t N, int64_t D,
                                 cudaStream_t s) {
    constexpr int V = Elt<T>::V;
    cudaError_t e = cudaErrorNotSupported;
    if (D % V == 0 && aligned_rows<T>(x, ldx) && aligned_rows<T>(y, ldy))
        e = softmax_fwd_vec<T, false>(x, ldx, y, ldy, N, D, D / V, s);
    else if (same_offsets<T>(x, ldx, y, ldy))
        e = softmax_fwd_vec<T, true>(x, ldx, y, ldy, N, D, (D + 2 * V - 2) / V, s);
    if (e != cudaErrorNotSupported) return e;
    constexpr int NT = 256;
    return launch(softmax_fwd_wide<T, NT>, dim3((unsigned)std::min<int64_t>(N, 8 * kDesignSMs)),
                  dim3(NT), 0, s, true, x, ldx, y, ldy, N, D);
}

template <typename T>
static cudaError_t softmax_bwd_t(const T* y, int64_t ldy, const T* dy, int64_t lddy, T* dx,
                                 int64_t lddx, int64_t N, int64_t D, cudaStream_t s) {
    constexpr int V = Elt<T>::V;
    cudaError_t e = cudaErrorNotSupported;
    if (D % V == 0 && aligned_rows<T>(y, ldy) && aligned_rows<T>(dy, lddy) &&
        aligned_rows<T>(dx, lddx))
        e = softmax_bwd_vec<T, false>(y, ldy, dy, lddy, dx, lddx, N, D, D / V, s);
    else if (same_offsets<T>(y, ldy, dy, lddy) && same_offsets<T>(y, ldy, dx, lddx))
        e = softmax_bwd_vec<T, true>(y, ldy, dy, lddy, dx, lddx, N, D, (D + 2 * V - 2) / V, s);
    if (e != cudaErrorNotSupported) return e;
    constexpr int NT = 256;
    return launch(softmax_bwd_wide<T, NT>, dim3((unsigned)std::min<int64_t>(N, 8 * kDesignSMs)),
                  dim3(NT), 0, s, true, y, ldy, dy, lddy, dx, lddx, N, D);
}

cudaError_t softmax_wait_timeouts(unsigned* count, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(count, g_softmax_wait_timeouts, sizeof(unsigned));
    if (e == cudaSuccess && reset) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_softmax_wait_timeouts, &zero, sizeof(unsigned));
    }
    return e;
}

cudaError_t launch_softmax_fwd(const void* x, int64_t ldx, void* y, int64_t ldy, int64_t N,
                               int64_t D, int dtype, cudaStream_t s) {
    switch (dtype) {
        case 0: return softmax_fwd_t((const float*)x, ldx, (float*)y, ldy, N, D, s);
        case 1: return softmax_fwd_t((const __half*)x, ldx, (__half*)y, ldy, N, D, s);
        default:
            return softmax_fwd_t((const __nv_bfloat16*)x, ldx, (__nv_bfloat16*)y, ldy, N, D, s);
    }
}

cudaError_t launch_softmax_bwd(const void* y, int64_t ldy, const void* dy, int64_t lddy, void* dx,
                               int64_t lddx, int64_t N, int64_t D, int dtype, cudaStream_t s) {
    switch (dtype) {
        case 0:
            return softmax_bwd_t((const float*)y, ldy, (const float*)dy, lddy, (float*)dx, lddx, N,
                                 D, s);
        case 1:
            return softmax_bwd_t((const __half*)y, ldy, (const __half*)dy, lddy, (__half*)dx, lddx,
                                 N, D, s);
        default:
            return softmax_bwd_t((const __nv_bfloat16*)y, ldy, (const __nv_bfloat16*)dy, lddy,
                                 (__nv_bfloat16*)dx, lddx, N, D, s);
    }
}

}  // namespace wsf
