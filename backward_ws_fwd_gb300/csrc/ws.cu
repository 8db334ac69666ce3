// ws.cu — weighted-sum forward and backward kernels for sm_103a.
//
// Operator ("Writing Triton Kernels with Autograd: A Minimal End-to-End
// Example", §1 Problem Setup): y[i] = Σ_d x[i,d]·w[d], x [N,D], w [D].
// Backward (same page, §3 Backward: Deriving Gradients First; §4 Triton
// Backward Kernel): dx[i,d] = dy[i]·w[d] is elementwise and parallel over
// rows; grad_w[d] = Σ_i x[i,d]·dy[i] reduces over the batch axis, done in two
// stages: each row tile writes one partial row, then a fixed-order sum over
// tiles.  Every grad_w sum is a compensated fp32 pair (TwoSum of each
// product into a running sum, the rounding errors collected beside it), so
// the result is as accurate as a sum in twice the precision, rounded once.
//
// Kernel families, chosen on the host by row width and alignment:
//  * forward, register path (rows of <= 4 KB, 16-byte aligned): a row is
//    split over LPR lanes of a warp, each lane owning CPL 16-byte chunks of
//    columns and holding their weights in registers; a warp covers 32/LPR
//    rows per load instruction with U rows per lane in flight; row sums use
//    an xor butterfly inside the LPR-lane group.
//  * forward, wide path (rows > 4 KB): one CTA per row walks its columns;
//    the w chunks come from L2.
//  * backward, staged path (16-byte aligned): a 2-D grid of (row tile x
//    column slice); each thread owns one 16-byte column chunk (its V weights
//    and V grad_w accumulators in registers) and walks its share of the
//    tile's rows.  x is staged S steps ahead into shared memory with
//    cp.async — each thread copies and later reads only its own chunks — and
//    each step's slice of dy is staged the same way by a few threads.  The
//    bytes in flight are then bounded by shared memory, not registers.
//  * backward, tile path: the same thread layout with register-held loads,
//    for aligned x/dx whose dy or tile starts are not 16-byte aligned.
//  * scalar paths (any alignment, any D): element-wise loads, same tiling of
//    the grad_w partials.
// No atomics anywhere: every sum has a fixed operand order.
#include <algorithm>
#include <mutex>
#include <type_traits>
#include <utility>
#include <vector>

#include "wsf_device.cuh"
#include "wsf_internal.h"

namespace wsf {

// Rows [a, b) of row tile p.  block_n > 0 gives tiles of block_n rows (the
// last one ragged).  Otherwise the N rows are split into P near-equal tiles
// whose boundaries are multiples of 8 rows (the last tile ends at N), so that
// every tile's slice of dy starts on a 16-byte boundary.
__host__ __device__ __forceinline__ void tile_rows(int64_t p, int64_t P, int64_t N,
                                                   int64_t block_n, int64_t& a, int64_t& b) {
    if (block_n > 0) {
        a = p * block_n;
        b = (a + block_n < N) ? a + block_n : N;
    } else {
        a = ((p * N) / P) & ~(int64_t)7;
        b = (p + 1 == P) ? N : ((((p + 1) * N) / P) & ~(int64_t)7);
    }
}

// ---------------------------------------------------------------------------
// Tiling constants (chosen for 152 SMs; all are compile-time, so the
// reduction order depends on nothing but the sizes).
constexpr int kRegMaxChunks = 256;        // forward register path: rows of <= 256 x 16 B
constexpr int kSliceChunks = 256;         // backward: 16-byte chunks per column slice
constexpr int64_t kTileSlots = 6 * kDesignSMs;  // 912 CTAs per backward launch at most
constexpr int64_t kRowsPerTileMin = 64;

// P = number of row tiles.  A row of D elements is cut into column slices of
// kSliceChunks 16-byte chunks; P is the largest tile count that keeps
// slices x P within kTileSlots CTAs, at least kRowsPerTileMin rows per tile,
// and at least 1.
int64_t ws_tiles(int64_t N, int64_t D, int dtype, int64_t block_n) {
    if (N <= 0 || D <= 0) return 0;
    if (block_n > 0) return (N + block_n - 1) / block_n;
    const int64_t chunks = (D * elt_bytes(dtype) + 15) / 16;
    const int64_t slices = (chunks + kSliceChunks - 1) / kSliceChunks;
    int64_t p = (N + kRowsPerTileMin - 1) / kRowsPerTileMin;
    const int64_t cap = kTileSlots / slices;
    if (p > cap) p = cap;
    return p < 1 ? 1 : p;
}

// The forward sums use compensated accumulation when the output is binary32,
// whose stated tolerance (1e-6 relative) is below the error of a plain
// binary32 sum of tens of thousands of terms; 16-bit outputs round far above
// that error and use plain fp32 accumulation.
template <typename T>
constexpr bool kCompensated = std::is_same<T, float>::value;

// grad_w sums are compensated for every storage type (the stated 1e-5 bound
// holds for the exact value even where a column's sum cancels); the product
// x·dy is exact in binary32 for 16-bit storage and split with an FMA for
// binary32.
template <typename T>
constexpr bool kExactProduct = !std::is_same<T, float>::value;

// Load the lane's CPL chunks of w (V fp32 values each) into registers.
template <int LPR, int CPL, int V>
__device__ __forceinline__ void load_w(const float* __restrict__ w, int l, int Dv,
                                       float (&wr)[CPL][V]) {
#pragma unroll
    for (int k = 0; k < CPL; k++) {
        const int c = l + k * LPR;
#pragma unroll
        for (int q = 0; q < V / 4; q++) {
            Raw16 r = (c < Dv) ? ld_keep(w + (int64_t)c * V + 4 * q) : raw_zero();
#pragma unroll
            for (int i = 0; i < 4; i++) wr[k][4 * q + i] = __uint_as_float(r.u[i]);
        }
    }
}

// ===========================================================================
// Forward
// ===========================================================================

template <typename T, int LPR, int CPL, int U, int NT, int MINB>
__global__ void __launch_bounds__(NT, MINB)
    ws_fwd_reg(const T* __restrict__ x, int64_t ldx, const float* __restrict__ w,
               T* __restrict__ y, int64_t N, int Dv) {
    using E = Elt<T>;
    constexpr int V = E::V;
    constexpr int G = 32 / LPR;  // rows per warp load instruction
    constexpr int RW = G * U;    // rows per warp iteration
    const int lane = threadIdx.x & 31;
    const int g = lane / LPR, l = lane % LPR;

    pdl_wait();
    float wr[CPL][V];
    load_w<LPR, CPL, V>(w, l, Dv, wr);

    const int64_t warp = ((int64_t)blockIdx.x * NT + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * NT) >> 5;
    for (int64_t base = warp * RW; base < N; base += nwarps * RW) {
        Raw16 xr[U][CPL];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int64_t row = base + u * G + g;
#pragma unroll
            for (int k = 0; k < CPL; k++) {
                const int c = l + k * LPR;
                xr[u][k] = (row < N && c < Dv) ? ld_stream(x + row * ldx + (int64_t)c * V)
                                               : raw_zero();
            }
        }
        float acc[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
            if constexpr (kCompensated<T>) {
                Acc2 a = acc2_zero();
#pragma unroll
                for (int k = 0; k < CPL; k++) {
                    float f[V];
                    E::widen(xr[u][k], f);
#pragma unroll
                    for (int v = 0; v < V; v++) acc2_fma(a, f[v], wr[k][v]);
                }
                a = group_sum2<LPR>(a);
                acc[u] = a.hi + a.lo;
            } else {
                float a = 0.f;
#pragma unroll
                for (int k = 0; k < CPL; k++) {
                    float f[V];
                    E::widen(xr[u][k], f);
#pragma unroll
                    for (int v = 0; v < V; v++) a = fmaf(f[v], wr[k][v], a);
                }
                acc[u] = group_sum<LPR>(a);
            }
        }
        // every lane of a group holds all U row sums; lane l stores rows u = l, l+LPR, ...
        for (int u = l; u < U; u += LPR) {
            const int64_t row = base + u * G + g;
            if (row < N) E::store1(y + row, select<U>(acc, u));
        }
    }
    pdl_trigger();
}

// Wide rows: one CTA per row (grid-stride over rows).  Each thread sums the
// products of its chunks c0, c0 + NT, ... in order; for binary32 outputs the
// running sum is compensated (Kahan: the rounding error of every addition is
// carried in a second register), then the threads are combined with
// double-float additions (xor butterfly in each warp, warps in index order).
template <typename T, int UJ, int NT>
__global__ void __launch_bounds__(NT)
    ws_fwd_wide(const T* __restrict__ x, int64_t ldx, const float* __restrict__ w,
                T* __restrict__ y, int64_t N, int64_t Dv) {
    using E = Elt<T>;
    constexpr int V = E::V;
    constexpr int NW = NT / 32;
    __shared__ Acc2 red[NW];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    pdl_wait();
    for (int64_t row = blockIdx.x; row < N; row += gridDim.x) {
        const T* xrow = x + row * ldx;
        float s = 0.f, comp = 0.f;
        for (int64_t c0 = threadIdx.x; c0 < Dv; c0 += (int64_t)NT * UJ) {
            Raw16 xr[UJ];
            float wv[UJ][V];
#pragma unroll
            for (int j = 0; j < UJ; j++) {
                const int64_t c = c0 + (int64_t)j * NT;
                const bool ok = c < Dv;
#pragma unroll
                for (int q = 0; q < V / 4; q++) {
                    Raw16 rw = ok ? ld_keep(w + c * V + 4 * q) : raw_zero();
#pragma unroll
                    for (int i = 0; i < 4; i++) wv[j][4 * q + i] = __uint_as_float(rw.u[i]);
                }
                xr[j] = ok ? ld_stream(xrow + c * V) : raw_zero();
            }
#pragma unroll
            for (int j = 0; j < UJ; j++) {
                float f[V];
                E::widen(xr[j], f);
#pragma unroll
                for (int v = 0; v < V; v++) {
                    if constexpr (kCompensated<T>) {
                        const float yk = __fsub_rn(__fmul_rn(f[v], wv[j][v]), comp);
                        const float t = __fadd_rn(s, yk);
                        comp = __fsub_rn(__fsub_rn(t, s), yk);
                        s = t;
                    } else {
                        s = fmaf(f[v], wv[j][v], s);
                    }
                }
            }
        }
        Acc2 a{s, -comp};
        if constexpr (kCompensated<T>) {
            a = group_sum2<32>(a);
        } else {
            a.hi = group_sum<32>(a.hi);
        }
        if (lane == 0) red[wid] = a;
        __syncthreads();
        if (threadIdx.x == 0) {
            Acc2 t = red[0];
#pragma unroll
            for (int q = 1; q < NW; q++) t = acc2_add(t, red[q]);
            E::store1(y + row, t.hi + t.lo);
        }
        __syncthreads();
    }
    pdl_trigger();
}

// One warp per row, element-wise loads: any alignment, any D (D == 0 gives 0).
template <typename T, int NT>
__global__ void __launch_bounds__(NT)
    ws_fwd_scalar(const T* __restrict__ x, int64_t ldx, const float* __restrict__ w,
                  T* __restrict__ y, int64_t N, int64_t D) {
    using E = Elt<T>;
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * NT + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * NT) >> 5;
    pdl_wait();
    for (int64_t row = warp; row < N; row += nwarps) {
        Acc2 a = acc2_zero();
        for (int64_t d = lane; d < D; d += 32) {
            if constexpr (kCompensated<T>)
                acc2_fma(a, E::load1(x + row * ldx + d), __ldg(w + d));
            else
                a.hi = fmaf(E::load1(x + row * ldx + d), __ldg(w + d), a.hi);
        }
        float v;
        if constexpr (kCompensated<T>) {
            a = group_sum2<32>(a);
            v = a.hi + a.lo;
        } else {
            v = group_sum<32>(a.hi);
        }
        if (lane == 0) E::store1(y + row, v);
    }
    pdl_trigger();
}

// ===========================================================================
// Backward, stage 1: dx and the per-tile partial rows of grad_w
// ===========================================================================

// Write the CTA's partial row for columns [slice·LPRC·V, ...) as compensated
// pairs: the high parts to out[0, ncols), the low parts to out[plane, plane +
// ncols).  G == 1 writes each thread's V pairs directly; otherwise the G row
// groups are added in index order (double-float additions) through shared
// memory `red` (2·G·LPRC·V floats).  With ATOMIC the row is instead added
// into grad_w (`out`) with atomic additions of each pair's value (the
// measured comparison variant: the order of the additions, and so the bits
// of the result, then depend on scheduling).
template <int LPRC, int G, int V, int NT, bool ATOMIC = false>
__device__ __forceinline__ void write_partial(const Acc2 (&acc)[V], float* __restrict__ out,
                                              int64_t plane, int g, int l, bool cok,
                                              int64_t ncols, float* red) {
    if constexpr (G == 1) {
        if (cok) {
#pragma unroll
            for (int q = 0; q < V / 4; q++) {
                if constexpr (ATOMIC) {
                    atomicAdd(reinterpret_cast<float4*>(out + l * V + 4 * q),
                              make_float4(acc2_value(acc[4 * q]), acc2_value(acc[4 * q + 1]),
                                          acc2_value(acc[4 * q + 2]), acc2_value(acc[4 * q + 3])));
                } else {
                    Raw16 h, o;
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        h.u[i] = __float_as_uint(acc[4 * q + i].hi);
                        o.u[i] = __float_as_uint(acc[4 * q + i].lo);
                    }
                    *reinterpret_cast<Raw16*>(out + l * V + 4 * q) = h;
                    *reinterpret_cast<Raw16*>(out + plane + l * V + 4 * q) = o;
                }
            }
        }
    } else {
        constexpr int H = G * LPRC * V;
#pragma unroll
        for (int v = 0; v < V; v++) {
            red[(g * LPRC + l) * V + v] = acc[v].hi;
            red[H + (g * LPRC + l) * V + v] = acc[v].lo;
        }
        __syncthreads();
        for (int j = threadIdx.x; j < ncols; j += NT) {
            Acc2 t{red[j], red[H + j]};
#pragma unroll
            for (int q = 1; q < G; q++)
                t = acc2_add(t, Acc2{red[q * LPRC * V + j], red[H + q * LPRC * V + j]});
            if constexpr (ATOMIC) {
                atomicAdd(out + j, acc2_value(t));
            } else {
                out[j] = t.hi;
                out[plane + j] = t.lo;
            }
        }
        __syncthreads();
    }
}

// Staged path.  blockIdx.x = row tile p, blockIdx.y = column slice.  The
// CTA's NT threads form G = NT / LPRC row groups of LPRC threads; thread
// (g, l) owns chunk c = slice·LPRC + l (V columns).  Step k covers rows
// ra + k·SR .. ra + (k+1)·SR - 1 (SR = G·U); thread (g, l) handles rows
// ra + k·SR + u·G + g, u < U.  Its x chunks for step k + S - 1 are copied
// into its own shared slots while it computes step k; the step's dy slice
// (SR values, 16-byte aligned) is copied in 16-byte pieces by the first
// threads, so each step starts with a CTA barrier.
template <typename T, int LPRC, int U, int S, int NT, int MINB, bool ATOMIC = false>
__global__ void __launch_bounds__(NT, MINB)
    ws_bwd_staged(const T* __restrict__ x, int64_t ldx, const float* __restrict__ w,
                  const T* __restrict__ dy, T* __restrict__ dx, int64_t lddx,
                  float* __restrict__ partial, int64_t plane, int64_t N, int64_t Dv,
                  int64_t D, int64_t block_n, int64_t P) {
    using E = Elt<T>;
    constexpr int V = E::V;
    constexpr int G = NT / LPRC;
    constexpr int SR = G * U;                 // rows per step
    constexpr int DYB = SR * (int)sizeof(T);  // dy bytes per step
    static_assert(DYB % 16 == 0, "dy step must be whole 16-byte copies");
    static_assert(S * U * 16 >= 8 * V, "staging buffer must hold the partial combine");
    extern __shared__ __align__(16) unsigned char smem[];
    Raw16* xs = reinterpret_cast<Raw16*>(smem);                                // [S][U][NT]
    T* dys = reinterpret_cast<T*>(smem + (size_t)S * U * NT * sizeof(Raw16));  // [S][SR]

    const int tid = threadIdx.x;
    const int g = tid / LPRC, l = tid % LPRC;
    int64_t ra, rb;
    tile_rows(blockIdx.x, P, N, block_n, ra, rb);
    const int64_t c = (int64_t)blockIdx.y * LPRC + l;
    const bool cok = c < Dv;
    pdl_wait();

    // weights and accumulators as packed pairs of columns (f32x2 arithmetic)
    uint64_t w2[V / 2];
#pragma unroll
    for (int q = 0; q < V / 4; q++) {
        Raw16 r = cok ? ld_keep(w + c * V + 4 * q) : raw_zero();
        w2[2 * q] = f2_pack(__uint_as_float(r.u[0]), __uint_as_float(r.u[1]));
        w2[2 * q + 1] = f2_pack(__uint_as_float(r.u[2]), __uint_as_float(r.u[3]));
    }
    Acc2x2 acc[V / 2];
#pragma unroll
    for (int k = 0; k < V / 2; k++) acc[k] = Acc2x2{0ull, 0ull};

    const int64_t nsteps = (rb - ra + SR - 1) / SR;
    auto issue = [&](int64_t k) {
        if (k < nsteps) {
            const int slot = (int)(k % S);
            const int64_t r0 = ra + k * SR;
#pragma unroll
            for (int u = 0; u < U; u++) {
                const int64_t row = r0 + u * G + g;
                const bool ok = row < rb && cok;
                cp_async16(&xs[(slot * U + u) * NT + tid],
                           ok ? (const void*)(x + row * ldx + c * V) : (const void*)x, ok ? 16 : 0);
            }
            for (int j = tid; j < DYB / 16; j += NT) {
                const int64_t first = r0 + j * (16 / (int)sizeof(T));
                const int64_t rem = (N - first) * (int64_t)sizeof(T);
                const int bytes = rem >= 16 ? 16 : (rem > 0 ? (int)rem : 0);
                cp_async16(reinterpret_cast<unsigned char*>(dys) + slot * DYB + j * 16,
                           bytes > 0 ? (const void*)(dy + first) : (const void*)dy, bytes);
            }
        }
        cp_async_commit();  // empty groups past the end keep the group count uniform
    };

#pragma unroll
    for (int k = 0; k < S - 1; k++) issue(k);
    for (int64_t k = 0; k < nsteps; k++) {
        cp_async_wait<S - 2>();  // this thread's copies for step k have landed
        __syncthreads();         // ... and every thread's (dy), and step k-1 is consumed
        issue(k + S - 1);        // refills the slot of step k-1
        const int slot = (int)(k % S);
        const int64_t r0 = ra + k * SR;
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int64_t row = r0 + u * G + g;
            const bool ok = row < rb;
            const float gv = ok ? E::widen1(dys[slot * SR + u * G + g]) : 0.f;
            const uint64_t g2 = f2_pack(gv, gv), ng2 = f2_pack(-gv, -gv);
            const Raw16 xr = xs[(slot * U + u) * NT + tid];
            if (ok && cok) {
                float f[V];
#pragma unroll
                for (int k = 0; k < V / 2; k++) f2_unpack(f2_mul(g2, w2[k]), f[2 * k], f[2 * k + 1]);
                st_stream(dx + row * lddx + c * V, E::narrow(f));
            }
            float f[V];
            E::widen(xr, f);
#pragma unroll
            for (int k = 0; k < V / 2; k++)
                acc2x2_prod<kExactProduct<T>>(acc[k], f2_pack(f[2 * k], f[2 * k + 1]), g2, ng2);
        }
    }
    cp_async_wait<0>();  // no copy may still target shared memory when the CTA ends
    pdl_trigger();
    __syncthreads();
    const int64_t col0 = (int64_t)blockIdx.y * LPRC * V;
    const int64_t ncols = (D - col0) < LPRC * V ? D - col0 : LPRC * V;
    // ATOMIC: `partial` is grad_w itself and every tile adds into the same row
    float* out = partial + (ATOMIC ? 0 : (int64_t)blockIdx.x * D) + col0;
    Acc2 sums[V];
#pragma unroll
    for (int k = 0; k < V / 2; k++) acc2x2_unpack(acc[k], sums[2 * k], sums[2 * k + 1]);
    write_partial<LPRC, G, V, NT, ATOMIC>(sums, out, plane, g, l, cok, ncols,
                                          reinterpret_cast<float*>(smem));
}

// Tile path: the staged kernel's thread layout with register-held loads (U
// rows in flight per thread); column slices are taken by blockIdx.y,
// blockIdx.y + gridDim.y, ...
template <typename T, int LPRC, int U, int NT>
__global__ void __launch_bounds__(NT)
    ws_bwd_tile(const T* __restrict__ x, int64_t ldx, const float* __restrict__ w,
                const T* __restrict__ dy, T* __restrict__ dx, int64_t lddx,
                float* __restrict__ partial, int64_t plane, int64_t N, int64_t Dv, int64_t D,
                int64_t block_n, int64_t P) {
    using E = Elt<T>;
    constexpr int V = E::V;
    constexpr int G = NT / LPRC;
    __shared__ float red[G > 1 ? 2 * G * LPRC * V : 1];
    const int g = threadIdx.x / LPRC, l = threadIdx.x % LPRC;
    int64_t ra, rb;
    tile_rows(blockIdx.x, P, N, block_n, ra, rb);
    const int64_t nslices = (Dv + LPRC - 1) / LPRC;
    pdl_wait();
    for (int64_t slice = blockIdx.y; slice < nslices; slice += gridDim.y) {
        const int64_t c = slice * LPRC + l;
        const bool cok = c < Dv;
        uint64_t w2[V / 2];
#pragma unroll
        for (int q = 0; q < V / 4; q++) {
            Raw16 r = cok ? ld_keep(w + c * V + 4 * q) : raw_zero();
            w2[2 * q] = f2_pack(__uint_as_float(r.u[0]), __uint_as_float(r.u[1]));
            w2[2 * q + 1] = f2_pack(__uint_as_float(r.u[2]), __uint_as_float(r.u[3]));
        }
        Acc2x2 acc[V / 2];
#pragma unroll
        for (int k = 0; k < V / 2; k++) acc[k] = Acc2x2{0ull, 0ull};
        for (int64_t base = ra + g; base < rb; base += (int64_t)G * U) {
            Raw16 xr[U];
            float gv[U];
#pragma unroll
            for (int u = 0; u < U; u++) {
                const int64_t row = base + (int64_t)u * G;
                const bool ok = row < rb;
                gv[u] = ok ? E::load1(dy + row) : 0.f;
                xr[u] = (ok && cok) ? ld_stream(x + row * ldx + c * V) : raw_zero();
            }
#pragma unroll
            for (int u = 0; u < U; u++) {
                const int64_t row = base + (int64_t)u * G;
                const uint64_t g2 = f2_pack(gv[u], gv[u]), ng2 = f2_pack(-gv[u], -gv[u]);
                if (row < rb && cok) {
                    float f[V];
#pragma unroll
                    for (int k = 0; k < V / 2; k++)
                        f2_unpack(f2_mul(g2, w2[k]), f[2 * k], f[2 * k + 1]);
                    st_stream(dx + row * lddx + c * V, E::narrow(f));
                }
                float f[V];
                E::widen(xr[u], f);
#pragma unroll
                for (int k = 0; k < V / 2; k++)
                    acc2x2_prod<kExactProduct<T>>(acc[k], f2_pack(f[2 * k], f[2 * k + 1]), g2, ng2);
            }
        }
        const int64_t col0 = slice * LPRC * V;
        const int64_t ncols = (D - col0) < LPRC * V ? D - col0 : LPRC * V;
        Acc2 sums[V];
#pragma unroll
        for (int k = 0; k < V / 2; k++) acc2x2_unpack(acc[k], sums[2 * k], sums[2 * k + 1]);
        write_partial<LPRC, G, V, NT>(sums, partial + (int64_t)blockIdx.x * D + col0, plane, g, l,
                                      cok, ncols, red);
    }
    pdl_trigger();
}

// Scalar path: blockIdx.x = row tile; a thread owns columns
// blockIdx.y·NT + threadIdx.x + k·gridDim.y·NT.
template <typename T, int NT>
__global__ void __launch_bounds__(NT)
    ws_bwd_scalar(const T* __restrict__ x, int64_t ldx, const float* __restrict__ w,
                  const T* __restrict__ dy, T* __restrict__ dx, int64_t lddx,
                  float* __restrict__ partial, int64_t plane, int64_t N, int64_t D,
                  int64_t block_n, int64_t P) {
    using E = Elt<T>;
    int64_t ra, rb;
    tile_rows(blockIdx.x, P, N, block_n, ra, rb);
    pdl_wait();
    for (int64_t col = (int64_t)blockIdx.y * NT + threadIdx.x; col < D;
         col += (int64_t)gridDim.y * NT) {
        const float wv = __ldg(w + col);
        Acc2 acc = acc2_zero();
        for (int64_t row = ra; row < rb; row++) {
            const float gv = E::load1(dy + row);
            E::store1(dx + row * lddx + col, gv * wv);
            acc2_prod<kExactProduct<T>>(acc, E::load1(x + row * ldx + col), gv);
        }
        partial[(int64_t)blockIdx.x * D + col] = acc.hi;
        partial[plane + (int64_t)blockIdx.x * D + col] = acc.lo;
    }
    pdl_trigger();
}

// ===========================================================================
// Backward, stage 2: grad_w[d] = (accumulate ? grad_w[d] : 0) + Σ_p partial[p,d]
// Each partial is a compensated pair (high plane at `partial`, low plane
// `plane` floats further on), and so is every sum here.  Thread (tx, ty) sums
// p = ty, ty + RY, ... in ascending order; the RY stripe sums are then
// combined by a fixed halving tree; the pair is rounded once to binary32 and,
// when accumulating, added to the old value in one binary32 addition.  RY is
// 32 for rows of up to 4096 columns and 8 above; either way the order is
// fixed by D.
// ===========================================================================
template <int RY>
__global__ void __launch_bounds__(32 * RY)
    ws_bwd_reduce(const float* __restrict__ partial, int64_t plane, int64_t P, int64_t D,
                  float* __restrict__ grad_w, int accumulate) {
    __shared__ Acc2 sm[RY][33];
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int64_t col = (int64_t)blockIdx.x * 32 + tx;
    pdl_wait();
    Acc2 s = acc2_zero();
    if (col < D) {
#pragma unroll 8
        for (int64_t p = ty; p < P; p += RY)
            s = acc2_add(s, Acc2{partial[p * D + col], partial[plane + p * D + col]});
    }
    sm[ty][tx] = s;
    __syncthreads();
#pragma unroll
    for (int h = RY / 2; h > 0; h >>= 1) {
        if (ty < h) sm[ty][tx] = acc2_add(sm[ty][tx], sm[ty + h][tx]);
        __syncthreads();
    }
    if (ty == 0 && col < D) {
        const float v = acc2_value(sm[0][tx]);
        grad_w[col] = accumulate ? grad_w[col] + v : v;
    }
    pdl_trigger();
}

// ===========================================================================
// Host launchers
// ===========================================================================

static inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

static inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

static inline int next_pow2(int64_t v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

// Raise a kernel's dynamic shared-memory limit once per (kernel, device).
static cudaError_t allow_smem(const void* kernel, size_t bytes) {
    if (bytes < 32 * 1024) return cudaSuccess;  // static shared memory counts against 48 KB too
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::mutex mu;
    static std::vector<std::pair<const void*, int>> done;
    std::lock_guard<std::mutex> lock(mu);
    for (auto& d : done)
        if (d.first == kernel && d.second == dev) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) done.emplace_back(kernel, dev);
    return e;
}

template <typename T, int LPR, int CPL, int U, int NT, int MINB>
static cudaError_t fwd_reg(const T* x, int64_t ldx, const float* w, T* y, int64_t N, int Dv,
                           cudaStream_t s) {
    constexpr int rows_per_cta = (NT / 32) * (32 / LPR) * U;
    const int64_t grid = std::min<int64_t>(cdiv(N, rows_per_cta), (int64_t)MINB * kDesignSMs);
    return launch(ws_fwd_reg<T, LPR, CPL, U, NT, MINB>, dim3((unsigned)grid), dim3(NT), 0, s,
                  true, x, ldx, w, y, N, Dv);
}

// Register-path shapes (measured on GB300): rows of <= 32 chunks use 128
// threads, 4 rows per lane in flight and 8 CTAs per SM; rows of 128 chunks
// one row per lane at 4 CTAs per SM.
template <typename T>
static cudaError_t ws_fwd_t(const T* x, int64_t ldx, const float* w, T* y, int64_t N, int64_t D,
                            cudaStream_t s) {
    constexpr int V = Elt<T>::V;
    const bool vec = D > 0 && D % V == 0 && ldx % V == 0 && aligned16(x) && aligned16(w);
    const int64_t Dv = D / V;
    if (vec && Dv <= kRegMaxChunks) {
        const int dv = (int)Dv;
        if (dv <= 32) {
            switch (next_pow2(dv)) {
                case 1: return fwd_reg<T, 1, 1, 4, 128, 8>(x, ldx, w, y, N, dv, s);
                case 2: return fwd_reg<T, 2, 1, 4, 128, 8>(x, ldx, w, y, N, dv, s);
                case 4: return fwd_reg<T, 4, 1, 4, 128, 8>(x, ldx, w, y, N, dv, s);
                case 8: return fwd_reg<T, 8, 1, 4, 128, 8>(x, ldx, w, y, N, dv, s);
                case 16: return fwd_reg<T, 16, 1, 4, 128, 8>(x, ldx, w, y, N, dv, s);
                default: return fwd_reg<T, 32, 1, 4, 128, 8>(x, ldx, w, y, N, dv, s);
            }
        }
        if (dv <= 64) return fwd_reg<T, 32, 2, 2, 256, 4>(x, ldx, w, y, N, dv, s);
        if (dv <= 128) return fwd_reg<T, 32, 4, 1, 256, 4>(x, ldx, w, y, N, dv, s);
        return fwd_reg<T, 32, 8, 1, 256, 2>(x, ldx, w, y, N, dv, s);
    }
    if (vec) {
        constexpr int NT = 512, UJ = 4;
        const int64_t grid = std::min<int64_t>(N, 64 * kDesignSMs);
        return launch(ws_fwd_wide<T, UJ, NT>, dim3((unsigned)grid), dim3(NT), 0, s, true, x, ldx,
                      w, y, N, Dv);
    }
    constexpr int NT = 256;
    const int64_t grid = std::min<int64_t>(cdiv(N, NT / 32), 8 * kDesignSMs);
    return launch(ws_fwd_scalar<T, NT>, dim3((unsigned)grid), dim3(NT), 0, s, true, x, ldx, w, y,
                  N, D);
}

cudaError_t launch_ws_fwd(const void* x, int64_t ldx, const float* w, void* y, int64_t N,
                          int64_t D, int dtype, cudaStream_t s) {
    switch (dtype) {
        case 0: return ws_fwd_t((const float*)x, ldx, w, (float*)y, N, D, s);
        case 1: return ws_fwd_t((const __half*)x, ldx, w, (__half*)y, N, D, s);
        default:
            return ws_fwd_t((const __nv_bfloat16*)x, ldx, w, (__nv_bfloat16*)y, N, D, s);
    }
}

template <typename T>
struct BwdArgs {
    const T* x;
    int64_t ldx;
    const float* w;
    const T* dy;
    T* dx;
    int64_t lddx;
    float* partial;
    int64_t plane, N, Dv, D, block_n, P;
};

template <typename T, int LPRC, int U, int S, int NT, int MINB, bool ATOMIC = false>
static cudaError_t bwd_staged(const BwdArgs<T>& a, cudaStream_t s) {
    const size_t smem =
        (size_t)S * U * NT * sizeof(Raw16) + (size_t)S * (NT / LPRC) * U * sizeof(T);
    auto kernel = ws_bwd_staged<T, LPRC, U, S, NT, MINB, ATOMIC>;
    cudaError_t e = allow_smem((const void*)kernel, smem);
    if (e != cudaSuccess) return e;
    return launch(kernel, dim3((unsigned)a.P, (unsigned)cdiv(a.Dv, LPRC)), dim3(NT), smem, s,
                  true, a.x, a.ldx, a.w, a.dy, a.dx, a.lddx, a.partial, a.plane, a.N, a.Dv, a.D,
                  a.block_n, a.P);
}

template <typename T, int LPRC>
static cudaError_t bwd_tile(const BwdArgs<T>& a, cudaStream_t s) {
    constexpr int NT = LPRC < 128 ? 128 : LPRC, U = 4;
    const int64_t slices = std::min<int64_t>(cdiv(a.Dv, LPRC), 65535);
    return launch(ws_bwd_tile<T, LPRC, U, NT>, dim3((unsigned)a.P, (unsigned)slices), dim3(NT), 0,
                  s, true, a.x, a.ldx, a.w, a.dy, a.dx, a.lddx, a.partial, a.plane, a.N, a.Dv,
                  a.D, a.block_n, a.P);
}

// Staged-path shapes (measured on GB300 with the compensated accumulation):
// rows of <= 64 chunks use 128 threads, 4 rows per thread per step and 2
// steps in flight (16 KB of staging, 6 CTAs per SM); rows of 128 chunks 256
// threads as two row groups, 4 rows each and 2 steps (32 KB, 3 CTAs per SM);
// wider rows 256-chunk slices with 16 bytes of dy per step.  At c3's and
// c4's sizes these shapes beat the deeper staging they replaced (3-4 steps of
// 8 rows: 48-64 KB, 3-4 CTAs per SM) by 8% and 2.5%.
template <typename T, bool ATOMIC = false>
static cudaError_t bwd_staged_any(const BwdArgs<T>& a, int lprc, cudaStream_t s) {
    constexpr int UW = 16 / (int)sizeof(T);
    switch (lprc) {
        case 1: return bwd_staged<T, 1, 4, 2, 128, 6, ATOMIC>(a, s);
        case 2: return bwd_staged<T, 2, 4, 2, 128, 6, ATOMIC>(a, s);
        case 4: return bwd_staged<T, 4, 4, 2, 128, 6, ATOMIC>(a, s);
        case 8: return bwd_staged<T, 8, 4, 2, 128, 6, ATOMIC>(a, s);
        case 16: return bwd_staged<T, 16, 4, 2, 128, 6, ATOMIC>(a, s);
        case 32: return bwd_staged<T, 32, 4, 2, 128, 6, ATOMIC>(a, s);
        case 64: return bwd_staged<T, 64, 4, 2, 128, 6, ATOMIC>(a, s);
        case 128: return bwd_staged<T, 128, 4, 2, 256, 3, ATOMIC>(a, s);
        default: return bwd_staged<T, 256, UW, 3, 256, (sizeof(T) == 4 ? 4 : 3), ATOMIC>(a, s);
    }
}

template <typename T>
static cudaError_t bwd_vec(const BwdArgs<T>& a, int lprc, bool staged, cudaStream_t s) {
    if (staged) return bwd_staged_any<T>(a, lprc, s);
    switch (lprc) {
        case 1: return bwd_tile<T, 1>(a, s);
        case 2: return bwd_tile<T, 2>(a, s);
        case 4: return bwd_tile<T, 4>(a, s);
        case 8: return bwd_tile<T, 8>(a, s);
        case 16: return bwd_tile<T, 16>(a, s);
        case 32: return bwd_tile<T, 32>(a, s);
        case 64: return bwd_tile<T, 64>(a, s);
        case 128: return bwd_tile<T, 128>(a, s);
        default: return bwd_tile<T, 256>(a, s);
    }
}

template <typename T>
static cudaError_t ws_bwd_t(const T* x, int64_t ldx, const float* w, const T* dy, T* dx,
                            int64_t lddx, float* grad_w, int accumulate, float* partial,
                            int64_t block_n, int64_t N, int64_t D, int dtype, cudaStream_t s) {
    constexpr int V = Elt<T>::V;
    const int64_t P = ws_tiles(N, D, dtype, block_n);
    const int64_t plane = gradient_plane(P, D);
    cudaError_t e = cudaSuccess;
    if (P > 0) {
        const int64_t Dv = D / V;
        const bool vec = D % V == 0 && ldx % V == 0 && lddx % V == 0 && aligned16(x) &&
                         aligned16(w) && aligned16(dx) && aligned16(partial);
        if (vec) {
            const int lprc = Dv <= kSliceChunks ? next_pow2(Dv) : kSliceChunks;
            // staged path: every step's dy slice must start on a 16-byte boundary
            const bool staged = aligned16(dy) && (block_n * (int64_t)sizeof(T)) % 16 == 0 &&
                                cdiv(Dv, lprc) <= 65535;
            BwdArgs<T> a{x, ldx, w, dy, dx, lddx, partial, plane, N, Dv, D, block_n, P};
            e = bwd_vec<T>(a, lprc, staged, s);
        } else {
            constexpr int NT = 128;
            const int64_t slices = std::min<int64_t>(cdiv(D, NT), 65535);
            e = launch(ws_bwd_scalar<T, NT>, dim3((unsigned)P, (unsigned)slices), dim3(NT), 0, s,
                       true, x, ldx, w, dy, dx, lddx, partial, plane, N, D, block_n, P);
        }
        if (e != cudaSuccess) return e;
    }
    if (D > 0) {
        // narrow rows: 32 stripes of tiles per 32-column tile, so that a
        // handful of CTAs still keep many loads in flight
        if (D <= 4096)
            e = launch(ws_bwd_reduce<32>, dim3((unsigned)cdiv(D, 32)), dim3(32, 32), 0, s, true,
                       (const float*)partial, plane, P, D, grad_w, accumulate);
        else
            e = launch(ws_bwd_reduce<8>, dim3((unsigned)cdiv(D, 32)), dim3(32, 8), 0, s, true,
                       (const float*)partial, plane, P, D, grad_w, accumulate);
    }
    return e;
}

// ---------------------------------------------------------------------------
// Atomic comparison variant: zero grad_w (unless accumulating), then the
// staged stage-1 kernel adds each tile's partial row into grad_w with atomic
// additions.  One launch pair, no workspace, no fixed order.
__global__ void __launch_bounds__(256) zero_f32(float* __restrict__ p, int64_t n) {
    pdl_wait();
    for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (int64_t)gridDim.x * 256)
        p[i] = 0.f;
    pdl_trigger();
}

bool ws_bwd_atomic_supported(const void* x, int64_t ldx, const float* w, const void* dy,
                             const void* dx, int64_t lddx, const float* grad_w, int64_t D,
                             int dtype) {
    const int V = 16 / elt_bytes(dtype);
    const int64_t Dv = D / V;
    return D % V == 0 && ldx % V == 0 && lddx % V == 0 && aligned16(x) && aligned16(w) &&
           aligned16(dx) && aligned16(dy) && aligned16(grad_w) &&
           cdiv(Dv, Dv <= kSliceChunks ? next_pow2(Dv) : kSliceChunks) <= 65535;
}

template <typename T>
static cudaError_t ws_bwd_atomic_t(const T* x, int64_t ldx, const float* w, const T* dy, T* dx,
                                   int64_t lddx, float* grad_w, int accumulate, int64_t N,
                                   int64_t D, int dtype, cudaStream_t s) {
    constexpr int V = Elt<T>::V;
    cudaError_t e = cudaSuccess;
    if (!accumulate) {
        e = launch(zero_f32, dim3((unsigned)std::min<int64_t>(cdiv(D, 256), 1024)), dim3(256), 0,
                   s, true, grad_w, D);
        if (e != cudaSuccess) return e;
    }
    const int64_t P = ws_tiles(N, D, dtype, 0);
    if (P == 0) return e;
    const int64_t Dv = D / V;
    const int lprc = Dv <= kSliceChunks ? next_pow2(Dv) : kSliceChunks;
    BwdArgs<T> a{x, ldx, w, dy, dx, lddx, grad_w, 0, N, Dv, D, 0, P};
    return bwd_staged_any<T, true>(a, lprc, s);
}

cudaError_t launch_ws_bwd_atomic(const void* x, int64_t ldx, const float* w, const void* dy,
                                 void* dx, int64_t lddx, float* grad_w, int accumulate, int64_t N,
                                 int64_t D, int dtype, cudaStream_t s) {
    switch (dtype) {
        case 0:
            return ws_bwd_atomic_t((const float*)x, ldx, w, (const float*)dy, (float*)dx, lddx,
                                   grad_w, accumulate, N, D, dtype, s);
        case 1:
            return ws_bwd_atomic_t((const __half*)x, ldx, w, (const __half*)dy, (__half*)dx, lddx,
                                   grad_w, accumulate, N, D, dtype, s);
        default:
            return ws_bwd_atomic_t((const __nv_bfloat16*)x, ldx, w, (const __nv_bfloat16*)dy,
                                   (__nv_bfloat16*)dx, lddx, grad_w, accumulate, N, D, dtype, s);
    }
}

cudaError_t launch_ws_bwd(const void* x, int64_t ldx, const float* w, const void* dy, void* dx,
                          int64_t lddx, float* grad_w, int accumulate, float* partial,
                          int64_t block_n, int64_t N, int64_t D, int dtype, cudaStream_t s) {
    switch (dtype) {
        case 0:
            return ws_bwd_t((const float*)x, ldx, w, (const float*)dy, (float*)dx, lddx, grad_w,
                            accumulate, partial, block_n, N, D, dtype, s);
        case 1:
            return ws_bwd_t((const __half*)x, ldx, w, (const __half*)dy, (__half*)dx, lddx, grad_w,
                            accumulate, partial, block_n, N, D, dtype, s);
        default:
            return ws_bwd_t((const __nv_bfloat16*)x, ldx, w, (const __nv_bfloat16*)dy,
                            (__nv_bfloat16*)dx, lddx, grad_w, accumulate, partial, block_n, N, D,
                            dtype, s);
    }
}

}  // namespace wsf
