// ws.cu — weighted-sum forward and backward kernels for sm_103a.
//
// Operator ("Writing Triton Kernels with Autograd: A Minimal End-to-End
// Example", §1 Problem Setup): y[i] = Σ_d x[i,d]·w[d], x [N,D], w [D].
// Backward (same page, §3 Backward: Deriving Gradients First; §4 Triton
// Backward Kernel): dx[i,d] = dy[i]·w[d] is elementwise and parallel over
// rows; grad_w[d] = Σ_i x[i,d]·dy[i] reduces over the batch axis, done in two
// stages: each row tile writes one fp32 partial row, then a fixed-order sum
// over tiles.
//
// Kernel families, chosen on the host by row width and alignment:
//  * forward, register path (rows of <= 4 KB, 16-byte aligned): a row is
//    split over LPR lanes of a warp, each lane owning CPL 16-byte chunks of
//    columns and holding their weights in registers; a warp covers 32/LPR
//    rows per load instruction with U rows per lane in flight; row sums use
//    an xor butterfly inside the LPR-lane group.
//  * forward, wide path (rows > 4 KB): a CTA owns R rows and walks the
//    columns, reusing each w chunk (an L2 hit) for the R rows.
//  * backward, tile path (16-byte aligned): a 2-D grid of (column slice x row
//    tile); each thread owns one 16-byte column chunk (its V weights and V
//    grad_w accumulators in registers) and walks its share of the tile's rows.
//  * scalar paths (any alignment, any D): element-wise loads, same tiling of
//    the grad_w partials.
// No atomics anywhere: every sum has a fixed operand order.
#include <algorithm>
#include <type_traits>

#include "wsf_device.cuh"
#include "wsf_internal.h"

namespace wsf {

// Rows [a, b) of row tile p.  block_n > 0 gives tiles of block_n rows (the
// last one ragged); otherwise the N rows are split into P near-equal tiles.
__host__ __device__ __forceinline__ void tile_rows(int64_t p, int64_t P, int64_t N,
                                                   int64_t block_n, int64_t& a, int64_t& b) {
    if (block_n > 0) {
        a = p * block_n;
        b = (a + block_n < N) ? a + block_n : N;
    } else {
        a = (p * N) / P;
        b = ((p + 1) * N) / P;
    }
}

// ---------------------------------------------------------------------------
// Tiling constants (chosen for 152 SMs; all are compile-time, so the
// reduction order depends on nothing but the sizes).
constexpr int kRegMaxChunks = 256;       // forward register path: rows of <= 256 x 16 B
constexpr int kTileThreads = 256;        // backward tile kernel: threads per CTA
constexpr int kTileMinBlocks = 4;        // ... and CTAs resident per SM
constexpr int64_t kTileSlots = kTileMinBlocks * kDesignSMs;  // 608: one full wave
constexpr int64_t kRowsPerTileMin = 64;

// P = number of row tiles.  A row of D elements is cut into column slices of
// kTileThreads 16-byte chunks; P is the largest tile count that keeps
// slices x P within one wave of kTileSlots CTAs, at least kRowsPerTileMin
// rows per tile, and at least 1.
int64_t ws_tiles(int64_t N, int64_t D, int dtype, int64_t block_n) {
    if (N <= 0 || D <= 0) return 0;
    if (block_n > 0) return (N + block_n - 1) / block_n;
    const int64_t chunks = (D * elt_bytes(dtype) + 15) / 16;
    const int64_t slices = (chunks + kTileThreads - 1) / kTileThreads;
    int64_t p = (N + kRowsPerTileMin - 1) / kRowsPerTileMin;
    const int64_t cap = kTileSlots / slices;
    if (p > cap) p = cap;
    return p < 1 ? 1 : p;
}

// The forward sums use compensated accumulation (Acc2) when the output is
// binary32, whose stated tolerance (1e-6 relative) is below the error of a
// plain binary32 sum of tens of thousands of terms; 16-bit outputs round far
// above that error and use plain fp32 accumulation.
template <typename T>
constexpr bool kCompensated = std::is_same<T, float>::value;

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
}

template <typename T, int R, int UJ, int NT>
__global__ void __launch_bounds__(NT)
    ws_fwd_wide(const T* __restrict__ x, int64_t ldx, const float* __restrict__ w,
                T* __restrict__ y, int64_t N, int64_t Dv) {
    using E = Elt<T>;
    constexpr int V = E::V;
    constexpr int NW = NT / 32;
    __shared__ Acc2 red[NW][R];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int64_t r0 = (int64_t)blockIdx.x * R; r0 < N; r0 += (int64_t)gridDim.x * R) {
        Acc2 acc[R];  // lo stays 0 unless the storage type is binary32
#pragma unroll
        for (int r = 0; r < R; r++) acc[r] = acc2_zero();
        for (int64_t c0 = threadIdx.x; c0 < Dv; c0 += (int64_t)NT * UJ) {
            Raw16 xr[UJ][R];
            float wv[UJ][V];
#pragma unroll
            for (int j = 0; j < UJ; j++) {
                const int64_t c = c0 + (int64_t)j * NT;
#pragma unroll
                for (int q = 0; q < V / 4; q++) {
                    Raw16 rw = (c < Dv) ? ld_keep(w + c * V + 4 * q) : raw_zero();
#pragma unroll
                    for (int i = 0; i < 4; i++) wv[j][4 * q + i] = __uint_as_float(rw.u[i]);
                }
#pragma unroll
                for (int r = 0; r < R; r++)
                    xr[j][r] = (c < Dv && r0 + r < N) ? ld_stream(x + (r0 + r) * ldx + c * V)
                                                      : raw_zero();
            }
#pragma unroll
            for (int j = 0; j < UJ; j++)
#pragma unroll
                for (int r = 0; r < R; r++) {
                    float f[V];
                    E::widen(xr[j][r], f);
#pragma unroll
                    for (int v = 0; v < V; v++) {
                        if constexpr (kCompensated<T>)
                            acc2_fma(acc[r], f[v], wv[j][v]);
                        else
                            acc[r].hi = fmaf(f[v], wv[j][v], acc[r].hi);
                    }
                }
        }
#pragma unroll
        for (int r = 0; r < R; r++) {
            Acc2 s;
            if constexpr (kCompensated<T>) {
                s = group_sum2<32>(acc[r]);
            } else {
                s = Acc2{group_sum<32>(acc[r].hi), 0.f};
            }
            if (lane == 0) red[wid][r] = s;
        }
        __syncthreads();
        if (threadIdx.x < R && r0 + threadIdx.x < N) {
            Acc2 s = red[0][threadIdx.x];
#pragma unroll
            for (int q = 1; q < NW; q++) s = acc2_add(s, red[q][threadIdx.x]);
            E::store1(y + r0 + threadIdx.x, s.hi + s.lo);
        }
        __syncthreads();
    }
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
}

// ===========================================================================
// Backward, stage 1: dx and the per-tile partial rows of grad_w
// ===========================================================================

// Vector path.  blockIdx.x = row tile p; column slices of LPRC 16-byte
// chunks are taken by blockIdx.y, blockIdx.y + gridDim.y, ...  The CTA's NT threads form G = NT / LPRC row groups of
// LPRC threads; thread (g, l) owns chunk c = slice·LPRC + l (V columns) and
// handles rows ra + g, ra + g + G, ... of the tile, U of them in flight, in
// ascending order.  It keeps V weights and V accumulators in registers.  At
// the end the G row groups are added in index order through shared memory.
// Rows of up to NT chunks (4 KB) fit one slice; wider rows use several.
template <typename T, int LPRC, int U, int NT>
__global__ void __launch_bounds__(NT, kTileMinBlocks)
    ws_bwd_tile(const T* __restrict__ x, int64_t ldx, const float* __restrict__ w,
                const T* __restrict__ dy, T* __restrict__ dx, int64_t lddx,
                float* __restrict__ partial, int64_t N, int64_t Dv, int64_t D, int64_t block_n,
                int64_t P) {
    using E = Elt<T>;
    constexpr int V = E::V;
    constexpr int G = NT / LPRC;
    const int g = threadIdx.x / LPRC, l = threadIdx.x % LPRC;
    int64_t ra, rb;
    tile_rows(blockIdx.x, P, N, block_n, ra, rb);
    const int64_t nslices = (Dv + LPRC - 1) / LPRC;
    for (int64_t slice = blockIdx.y; slice < nslices; slice += gridDim.y) {
        const int64_t c = slice * LPRC + l;
        const bool cok = c < Dv;

        float wv[V];
    #pragma unroll
        for (int q = 0; q < V / 4; q++) {
            Raw16 r = cok ? ld_keep(w + c * V + 4 * q) : raw_zero();
    #pragma unroll
            for (int i = 0; i < 4; i++) wv[4 * q + i] = __uint_as_float(r.u[i]);
        }
        float acc[V];
    #pragma unroll
        for (int v = 0; v < V; v++) acc[v] = 0.f;

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
                if (row < rb && cok) {
                    float f[V];
    #pragma unroll
                    for (int v = 0; v < V; v++) f[v] = gv[u] * wv[v];
                    st_stream(dx + row * lddx + c * V, E::narrow(f));
                }
                float f[V];
                E::widen(xr[u], f);
    #pragma unroll
                for (int v = 0; v < V; v++) acc[v] = fmaf(f[v], gv[u], acc[v]);
            }
        }

        float* out = partial + (int64_t)blockIdx.x * D + slice * LPRC * V;
        if constexpr (G == 1) {
            if (cok) {
    #pragma unroll
                for (int q = 0; q < V / 4; q++) {
                    Raw16 r;
    #pragma unroll
                    for (int i = 0; i < 4; i++) r.u[i] = __float_as_uint(acc[4 * q + i]);
                    *reinterpret_cast<Raw16*>(out + l * V + 4 * q) = r;
                }
            }
        } else {
            __shared__ float red[G][LPRC * V];
    #pragma unroll
            for (int v = 0; v < V; v++) red[g][l * V + v] = acc[v];
            __syncthreads();
            const int64_t ncols = (D - slice * LPRC * V) < LPRC * V ? D - slice * LPRC * V
                                                                     : LPRC * V;
            for (int j = threadIdx.x; j < ncols; j += NT) {
                float s = red[0][j];
    #pragma unroll
                for (int q = 1; q < G; q++) s += red[q][j];
                out[j] = s;
            }
            __syncthreads();  // red[] is reused by the next slice
        }
    }  // slices
}

// Scalar path: blockIdx.x = row tile; a thread owns columns
// blockIdx.y·NT + threadIdx.x + k·gridDim.y·NT.
template <typename T, int NT>
__global__ void __launch_bounds__(NT)
    ws_bwd_scalar(const T* __restrict__ x, int64_t ldx, const float* __restrict__ w,
                  const T* __restrict__ dy, T* __restrict__ dx, int64_t lddx,
                  float* __restrict__ partial, int64_t N, int64_t D, int64_t block_n, int64_t P) {
    using E = Elt<T>;
    int64_t ra, rb;
    tile_rows(blockIdx.x, P, N, block_n, ra, rb);
    for (int64_t col = (int64_t)blockIdx.y * NT + threadIdx.x; col < D;
         col += (int64_t)gridDim.y * NT) {
        const float wv = __ldg(w + col);
        float acc = 0.f;
        for (int64_t row = ra; row < rb; row++) {
            const float gv = E::load1(dy + row);
            E::store1(dx + row * lddx + col, gv * wv);
            acc = fmaf(E::load1(x + row * ldx + col), gv, acc);
        }
        partial[(int64_t)blockIdx.x * D + col] = acc;
    }
}

// ===========================================================================
// Backward, stage 2: grad_w[d] = (accumulate ? grad_w[d] : 0) + Σ_p partial[p,d]
// Thread (tx, ty) sums p = ty, ty + RY, ... in ascending order; the RY
// stripe sums are then combined by a fixed halving tree.
// ===========================================================================
template <int RY>
__global__ void __launch_bounds__(32 * RY)
    ws_bwd_reduce(const float* __restrict__ partial, int64_t P, int64_t D,
                  float* __restrict__ grad_w, int accumulate) {
    __shared__ float sm[RY][33];
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int64_t col = (int64_t)blockIdx.x * 32 + tx;
    float s = 0.f;
    if (col < D)
        for (int64_t p = ty; p < P; p += RY) s += partial[p * D + col];
    sm[ty][tx] = s;
    __syncthreads();
#pragma unroll
    for (int h = RY / 2; h > 0; h >>= 1) {
        if (ty < h) sm[ty][tx] += sm[ty + h][tx];
        __syncthreads();
    }
    if (ty == 0 && col < D) {
        const float v = sm[0][tx];
        grad_w[col] = accumulate ? grad_w[col] + v : v;
    }
}

// ===========================================================================
// Host launchers
// ===========================================================================

static inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

static inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

static inline int next_pow2(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

template <typename T, int LPR, int CPL, int U>
static cudaError_t fwd_reg(const T* x, int64_t ldx, const float* w, T* y, int64_t N, int Dv,
                           cudaStream_t s) {
    constexpr int NT = 256;
    constexpr int rows_per_cta = (NT / 32) * (32 / LPR) * U;
    constexpr int MINB = CPL * Elt<T>::V <= 16 ? 4 : 2;
    const int64_t grid = std::min<int64_t>(cdiv(N, rows_per_cta), MINB * kDesignSMs);
    return launch(ws_fwd_reg<T, LPR, CPL, U, NT, MINB>, dim3((unsigned)grid), dim3(NT), 0, s, false, x,
                  ldx, w, y, N, Dv);
}

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
                case 1: return fwd_reg<T, 1, 1, 8>(x, ldx, w, y, N, dv, s);
                case 2: return fwd_reg<T, 2, 1, 8>(x, ldx, w, y, N, dv, s);
                case 4: return fwd_reg<T, 4, 1, 8>(x, ldx, w, y, N, dv, s);
                case 8: return fwd_reg<T, 8, 1, 8>(x, ldx, w, y, N, dv, s);
                case 16: return fwd_reg<T, 16, 1, 8>(x, ldx, w, y, N, dv, s);
                default: return fwd_reg<T, 32, 1, 8>(x, ldx, w, y, N, dv, s);
            }
        }
        if (dv <= 64) return fwd_reg<T, 32, 2, 4>(x, ldx, w, y, N, dv, s);
        if (dv <= 128) return fwd_reg<T, 32, 4, 2>(x, ldx, w, y, N, dv, s);
        return fwd_reg<T, 32, 8, 1>(x, ldx, w, y, N, dv, s);
    }
    if (vec) {
        constexpr int NT = 256, R = 4, UJ = 2;
        const int64_t grid = std::min<int64_t>(cdiv(N, R), 64 * kDesignSMs);
        return launch(ws_fwd_wide<T, R, UJ, NT>, dim3((unsigned)grid), dim3(NT), 0, s, false, x,
                      ldx, w, y, N, Dv);
    }
    constexpr int NT = 256;
    const int64_t grid = std::min<int64_t>(cdiv(N, NT / 32), 8 * kDesignSMs);
    return launch(ws_fwd_scalar<T, NT>, dim3((unsigned)grid), dim3(NT), 0, s, false, x, ldx, w, y,
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

template <typename T, int LPRC, int U>
static cudaError_t bwd_tile(const T* x, int64_t ldx, const float* w, const T* dy, T* dx,
                            int64_t lddx, float* partial, int64_t N, int64_t Dv, int64_t D,
                            int64_t block_n, int64_t P, cudaStream_t s) {
    constexpr int NT = kTileThreads;
    const int64_t slices = std::min<int64_t>(cdiv(Dv, LPRC), 65535);
    return launch(ws_bwd_tile<T, LPRC, U, NT>, dim3((unsigned)P, (unsigned)slices),
                  dim3(NT), 0, s, false, x, ldx, w, dy, dx, lddx, partial, N, Dv, D, block_n, P);
}

template <typename T>
static cudaError_t ws_bwd_t(const T* x, int64_t ldx, const float* w, const T* dy, T* dx,
                            int64_t lddx, float* grad_w, int accumulate, float* partial,
                            int64_t block_n, int64_t N, int64_t D, int dtype, cudaStream_t s) {
    constexpr int V = Elt<T>::V;
    const int64_t P = ws_tiles(N, D, dtype, block_n);
    cudaError_t e = cudaSuccess;
    if (P > 0) {
        const bool vec = D % V == 0 && ldx % V == 0 && lddx % V == 0 && aligned16(x) &&
                         aligned16(w) && aligned16(dx) && aligned16(partial);
        const int64_t Dv = D / V;
        if (vec) {
            switch (Dv <= kRegMaxChunks ? next_pow2((int)Dv) : kRegMaxChunks) {
                case 1: e = bwd_tile<T, 1, 4>(x, ldx, w, dy, dx, lddx, partial, N, Dv, D, block_n, P, s); break;
                case 2: e = bwd_tile<T, 2, 4>(x, ldx, w, dy, dx, lddx, partial, N, Dv, D, block_n, P, s); break;
                case 4: e = bwd_tile<T, 4, 4>(x, ldx, w, dy, dx, lddx, partial, N, Dv, D, block_n, P, s); break;
                case 8: e = bwd_tile<T, 8, 4>(x, ldx, w, dy, dx, lddx, partial, N, Dv, D, block_n, P, s); break;
                case 16: e = bwd_tile<T, 16, 4>(x, ldx, w, dy, dx, lddx, partial, N, Dv, D, block_n, P, s); break;
                case 32: e = bwd_tile<T, 32, 4>(x, ldx, w, dy, dx, lddx, partial, N, Dv, D, block_n, P, s); break;
                case 64: e = bwd_tile<T, 64, 4>(x, ldx, w, dy, dx, lddx, partial, N, Dv, D, block_n, P, s); break;
                case 128: e = bwd_tile<T, 128, 4>(x, ldx, w, dy, dx, lddx, partial, N, Dv, D, block_n, P, s); break;
                default: e = bwd_tile<T, 256, 4>(x, ldx, w, dy, dx, lddx, partial, N, Dv, D, block_n, P, s); break;
            }
        } else {
            constexpr int NT = 128;
            const int64_t slices = std::min<int64_t>(cdiv(D, NT), 65535);
            e = launch(ws_bwd_scalar<T, NT>, dim3((unsigned)P, (unsigned)slices), dim3(NT), 0,
                       s, false, x, ldx, w, dy, dx, lddx, partial, N, D, block_n, P);
        }
        if (e != cudaSuccess) return e;
    }
    if (D > 0) {
        constexpr int RY = 16;
        e = launch(ws_bwd_reduce<RY>, dim3((unsigned)cdiv(D, 32)), dim3(32, RY), 0, s, false,
                   (const float*)partial, P, D, grad_w, accumulate);
    }
    return e;
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
