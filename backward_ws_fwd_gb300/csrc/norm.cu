// norm.cu — RMSNorm and LayerNorm forward and backward for sm_103a.
//
// "Backward in Triton — autograd.Function and the backward grid", § Save vs
// recompute (the row statistic rstd is recomputed in the backward from x,
// not stored) and § The backward grid is not the forward grid (RMSNorm's dw:
// every row contributes a length-D partial that is summed across the batch,
// by a separate reduce over a partials buffer); "Backprop for kernel
// writers", §04 (LayerNorm collapses to two row scalars plus batch-axis
// parameter gradients).  The pages print no formulas; these are the
// textbook ones:
//   RMSNorm:   r = 1/sqrt(mean x² + eps), y = x·r·w;
//              g = dy·w, dx = r·(g − x̂·mean(g·x̂)) with x̂ = x·r,
//              dw = Σ_rows dy·x̂
//   LayerNorm: μ = mean x, r = 1/sqrt(mean (x−μ)² + eps), x̂ = (x−μ)·r,
//              y = x̂·w + b; dx = r·(g − mean g − x̂·mean(g·x̂)),
//              dw = Σ_rows dy·x̂, db = Σ_rows dy
//
// Row path (16-byte aligned rows of up to 8192 elements).  A row is held by a
// group of TPR threads, each owning CPT 16-byte chunks (at most 16 elements,
// so the backward's per-column accumulators stay in registers); the chunks
// are staged S rows ahead with cp.async into per-thread shared slots.
// RMSNorm needs one fused group reduction per row; LayerNorm two: Σx, then
// the sums over d = x − μ.  The mean is carried as μ₀ + c: μ₀ = fl(Σx/D) and
// c = (Σx − D·μ₀)/D from the remainder of the compensated Σx (hi + lo:
// fma(−D, μ₀, hi) is exact), and d = (x − μ₀) − c.  With μ₀ alone, its own
// rounding (up to ulp(μ)/2) would shift every x̂ of a row with a large common
// offset by the same amount, an error that does not cancel in Σ dy·x̂; and c
// cannot be taken from Σ(x − μ₀) either, since the rounding of x − μ₀ has
// one sign across a binade.  Σx must therefore be exact (center_row): for
// binary32 rows a compensated pair; for 16-bit rows the plain binary32 sum,
// which for at most 8192 elements of 8 or 11 significant bits stays exact
// unless the row spans many binades; for binary32 the other row sums are
// compensated too (Dot2), so that y and dx stay within 1e-6.  In the
// backward each thread sums dy·x̂ (and dy) for its own columns over the rows
// of its CTA's row tile; the CTA's row groups are combined in index order into
// one partial row per tile, and norm_bwd_reduce sums the tiles in a fixed
// order — the deterministic two-pass form, no atomics.  Other layouts take a
// multi-pass element-wise path with the same arithmetic.
#include <algorithm>
#include <type_traits>

#include "wsf_device.cuh"
#include "wsf_internal.h"

namespace wsf {

constexpr int64_t kNormTilesMax = 6 * kDesignSMs;  // 912 partial rows at most
constexpr int64_t kNormRowsPerTileMin = 64;
constexpr int64_t kNormRowMax = 8192;  // widest row (elements) of the row path

int64_t norm_tiles(int64_t N, int64_t D) {
    if (N <= 0 || D <= 0) return 0;
    const int64_t p = (N + kNormRowsPerTileMin - 1) / kNormRowsPerTileMin;
    return p < kNormTilesMax ? p : kNormTilesMax;
}

__device__ __forceinline__ void norm_tile_rows(int64_t p, int64_t P, int64_t N, int64_t& a,
                                               int64_t& b) {
    a = (p * N) / P;
    b = ((p + 1) * N) / P;
}

// ---------------------------------------------------------------------------
// Row sums: plain fp32 (C = false) or compensated (C = true, value hi + lo).
template <bool C>
__device__ __forceinline__ void s_add(Acc2& a, float v) {
    if constexpr (C) {
        float s, e;
        two_sum(a.hi, v, s, e);
        a.hi = s;
        a.lo += e;
    } else {
        a.hi += v;
    }
}

template <bool C>
__device__ __forceinline__ void s_fma(Acc2& a, float x, float y) {
    if constexpr (C)
        acc2_fma(a, x, y);
    else
        a.hi = fmaf(x, y, a.hi);
}

template <bool C>
__device__ __forceinline__ Acc2 s_comb(Acc2 a, Acc2 b) {
    if constexpr (C)
        return acc2_add(a, b);
    else
        return Acc2{a.hi + b.hi, 0.f};
}

__device__ __forceinline__ float s_val(const Acc2& a) { return a.hi + a.lo; }

// The sum of a packed pair's two lanes as a (plain) row sum.
__device__ __forceinline__ Acc2 lanes_sum(uint64_t a) {
    float a0, a1;
    f2_unpack(a, a0, a1);
    return Acc2{a0 + a1, 0.f};
}

// Reduce K sums over each aligned group of TPR threads: xor butterfly inside
// a warp; for groups wider than a warp, lane 0 of each warp posts its sums to
// `red` (K·NT/32 float2) and, after a barrier, every warp loads the group's
// NWG partials into its lanes (lane i takes partial i mod NWG) and runs a
// second butterfly over NWG lanes.  Every thread of the CTA calls it together;
// the order is fixed and every lane of a group ends with the same bits (the
// compensated addition is symmetric in its operands).  There is no barrier
// after the reads: callers alternate between two `red` buffers (RedRing), so
// a buffer is written again only after another reduction's barrier, which no
// thread passes before every thread has read this one.
template <int TPR, int NT, int K, bool C>
__device__ __forceinline__ void cross_warp(Acc2 (&v)[K], float2* red) {
    if constexpr (TPR > 32) {
        constexpr int NW = NT / 32, NWG = TPR / 32;
        const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int first = (threadIdx.x / TPR) * NWG;
        if (lane == 0)
#pragma unroll
            for (int q = 0; q < K; q++) red[q * NW + wid] = make_float2(v[q].hi, v[q].lo);
        __syncthreads();
#pragma unroll
        for (int q = 0; q < K; q++) {
            const float2 t = red[q * NW + first + (lane % NWG)];
            if constexpr (C)
                v[q] = group_sum2<NWG>(Acc2{t.x, t.y});
            else
                v[q] = Acc2{group_sum<NWG>(t.x), 0.f};
        }
    }
}

// Two shared reduction buffers used in turn (see cross_warp).  The turn is
// counted per thread: every thread of the CTA takes the buffers in the same
// sequence, so all of them agree on which one is current.
template <int N>
struct RedRing {
    float2 (*buf)[N];  // shared [2][N]
    int next;
    __device__ __forceinline__ float2* take() { return buf[(next++) & 1]; }
};

template <int TPR, int NT, int K, bool C>
__device__ __forceinline__ void group_reduce(Acc2 (&v)[K], float2* red) {
    constexpr int W = TPR < 32 ? TPR : 32;
#pragma unroll
    for (int q = 0; q < K; q++) {
        if constexpr (C)
            v[q] = group_sum2<W>(v[q]);
        else
            v[q].hi = group_sum<W>(v[q].hi);
    }
    cross_warp<TPR, NT, K, C>(v, red);
}

// 1/sqrt(ms + eps) with ms = Σ·(1/D).  Binary32 storage: IEEE square root
// and division (this library is built without fast-math), within about one
// ulp.  16-bit storage: the hardware reciprocal square root (a few ulp of
// binary32), far inside the half-ulp of the 16-bit output.
template <bool Exact>
__device__ __forceinline__ float rstd_of(float sum_sq, float inv_d, float eps) {
    const float ms = fmaf(sum_sq, inv_d, eps);
    if constexpr (Exact)
        return 1.0f / sqrtf(ms);
    else
        return rsqrtf(ms);
}

// The row mean as μ₀ + c from the pair s = Σx (hi + lo): μ₀ = (hi + lo)·(1/D)
// within two ulp, and c = (Σx − D·μ₀)/D.  hi − D·μ₀ is exact in one fma: it
// is a multiple of ulp(μ₀)/2^k no larger than a few ulp(hi), so it has at
// most log2(D) + 3 significant bits.  Adding lo and scaling by 1/D then round
// relative to c, which is only a correction.
struct Mean {
    float mu0, c;
};

__device__ __forceinline__ Mean mean_of(const Acc2& s, float d, float inv_d) {
    Mean m;
    m.mu0 = s_val(s) * inv_d;
    m.c = (fmaf(-d, m.mu0, s.hi) + s.lo) * inv_d;
    return m;
}

// Backward row scalars from sums = {Σ d², Σ g·d[, Σ g]}: r, mean(g) (zero for
// RMSNorm) and mean(g·x̂) = r·Σ g·d / D.
struct BwdStats {
    float r, mg, mgx;
};

template <bool LN, bool Exact, int K>
__device__ __forceinline__ BwdStats bwd_stats(const Acc2 (&sums)[K], float inv_d, float eps) {
    BwdStats st;
    st.r = rstd_of<Exact>(s_val(sums[0]), inv_d, eps);
    st.mgx = st.r * (s_val(sums[1]) * inv_d);
    st.mg = LN ? s_val(sums[K - 1]) * inv_d : 0.f;
    return st;
}

// LayerNorm's row mean, and x turned into d = x − μ in place (valid chunks).
// The mean is carried as μ₀ + c from a pair s = Σx (see mean_of).
// binary32 storage: TwoSum per element and compensated additions across the
// group, so no rounding of the sum reaches the mean.  16-bit storage: plain
// binary32 sums, which are exact where it matters — a row whose values share
// a large common offset has them on the coarse grid of that offset (ulp(100)
// is 0.5 in bfloat16, 1/16 in binary16), and the row sum stays below 2^24
// grid steps — while an addition rounds only where an element is fine-grained,
// i.e. small, and then errs by a few ulp of the partial sum, tiny next to the
// spread of the row.
template <typename T, int TPR, int NT, int CPT, int V>
__device__ __forceinline__ void center_row(float (&f)[CPT][V], unsigned valid, float fd,
                                           float inv_d, float2* red) {
    constexpr bool C = std::is_same<T, float>::value;
    Acc2 s[1] = {acc2_zero()};
    if constexpr (C) {
#pragma unroll
        for (int c = 0; c < CPT; c++)
#pragma unroll
            for (int v = 0; v < V; v++) s_add<true>(s[0], f[c][v]);  // invalid chunks are zero
    } else {
        // even and odd columns in the two lanes of a packed pair
        uint64_t a = 0ull;
#pragma unroll
        for (int c = 0; c < CPT; c++)
#pragma unroll
            for (int v = 0; v < V; v += 2) a = f2_add(a, f2_pack(f[c][v], f[c][v + 1]));
        float s0, s1;
        f2_unpack(a, s0, s1);
        s[0].hi = s0 + s1;
    }
    group_reduce<TPR, NT, 1, C>(s, red);
    const Mean m = mean_of(s[0], fd, inv_d);
    if constexpr (C) {
#pragma unroll
        for (int c = 0; c < CPT; c++)
            if (valid >> c & 1u)
#pragma unroll
                for (int v = 0; v < V; v++) f[c][v] = (f[c][v] - m.mu0) - m.c;
    } else {
        const uint64_t mu2 = f2_pack(m.mu0, m.mu0), c2 = f2_pack(m.c, m.c);
#pragma unroll
        for (int c = 0; c < CPT; c++)
            if (valid >> c & 1u)
#pragma unroll
                for (int v = 0; v < V; v += 2)
                    f2_unpack(f2_sub(f2_sub(f2_pack(f[c][v], f[c][v + 1]), mu2), c2), f[c][v],
                              f[c][v + 1]);
    }
}

// Per-thread cp.async staging of one row at a time: chunk c of the thread is
// the 16 bytes at chunk index l + c·TPR of the row.  The source pointer and
// the row index advance by a fixed step per staged row; rows at or past
// row_end, and chunks outside the row, are zero-filled without a read.
struct RowStager {
    const char* src;   // chunk 0 of the next row to stage
    const char* safe;  // any valid address (not read when the copy size is 0)
    int64_t src_step;  // bytes between staged rows
    int64_t row, row_step, row_end;
};

template <int TPR, int CPT, int NT>
__device__ __forceinline__ void stage_row(Raw16* slots, RowStager& st, unsigned valid) {
    const bool rok = st.row < st.row_end;
#pragma unroll
    for (int k = 0; k < CPT; k++) {
        const bool ok = rok && (valid >> k & 1u);
        cp_async16(&slots[k * NT + threadIdx.x], ok ? st.src + k * TPR * 16 : st.safe, ok ? 16 : 0);
    }
    st.src += st.src_step;
    st.row += st.row_step;
}

template <int TPR, int CPT>
__device__ __forceinline__ unsigned chunk_mask(int Dv, int l) {
    unsigned m = 0;
#pragma unroll
    for (int k = 0; k < CPT; k++) m |= (l + k * TPR < Dv ? 1u : 0u) << k;
    return m;
}

template <typename E, int CPT, int NT, int V>
__device__ __forceinline__ void load_row(const Raw16* cur, unsigned valid, float (&f)[CPT][V]) {
#pragma unroll
    for (int c = 0; c < CPT; c++) {
        if (valid >> c & 1u) {
            E::widen(cur[c * NT], f[c]);
        } else {
#pragma unroll
            for (int v = 0; v < V; v++) f[c][v] = 0.f;
        }
    }
}

template <int TPR, int CPT, int V>
__device__ __forceinline__ void load_params(const float* __restrict__ p, int Dv, int l,
                                            float (&out)[CPT][V]) {
#pragma unroll
    for (int k = 0; k < CPT; k++) {
        const int c = l + k * TPR;
#pragma unroll
        for (int q = 0; q < V / 4; q++) {
            const Raw16 r = (c < Dv) ? ld_keep(p + (int64_t)c * V + 4 * q) : raw_zero();
#pragma unroll
            for (int i = 0; i < 4; i++) out[k][4 * q + i] = __uint_as_float(r.u[i]);
        }
    }
}

// ===========================================================================
// Forward, row path: R = NT/TPR rows per CTA iteration, grid-stride.  The
// row is widened into registers once; LayerNorm turns it into d in place.
// ===========================================================================
template <typename T, bool LN, int TPR, int CPT, int NT, int S, int MINB>
__global__ void __launch_bounds__(NT, MINB)
    norm_fwd_rows(const T* __restrict__ x, int64_t ldx, const float* __restrict__ w,
                  const float* __restrict__ b, float eps, T* __restrict__ y, int64_t ldy,
                  int64_t N, int Dv) {
    using E = Elt<T>;
    constexpr int V = E::V;
    constexpr int R = NT / TPR;
    constexpr bool C = std::is_same<T, float>::value;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Raw16* xs = reinterpret_cast<Raw16*>(smem_raw);  // [S][CPT][NT]
    __shared__ float2 red_buf[2][NT / 32];
    RedRing<NT / 32> red{red_buf, 0};
    const int g = threadIdx.x / TPR, l = threadIdx.x % TPR;
    const float fd = (float)(Dv * V), inv_d = 1.0f / fd;
    const unsigned valid = chunk_mask<TPR, CPT>(Dv, l);
    pdl_wait();
    float wv[CPT][V], bv[CPT][V];
    load_params<TPR, CPT, V>(w, Dv, l, wv);
    if constexpr (LN) load_params<TPR, CPT, V>(b, Dv, l, bv);
    const int64_t base = (int64_t)blockIdx.x * R, stride = (int64_t)gridDim.x * R;
    const int64_t iters = base < N ? (N - base + stride - 1) / stride : 0;
    const int64_t ldb = ldx * (int64_t)sizeof(T);
    RowStager stg{reinterpret_cast<const char*>(x) + (base + g) * ldb + (int64_t)l * 16,
                  reinterpret_cast<const char*>(x), stride * ldb, base + g, stride, N};
    T* yrow = y + (base + g) * ldy + (int64_t)l * V;
    const int64_t ystep = stride * ldy;
#pragma unroll
    for (int k = 0; k < S - 1; k++) {
        if (k < iters) stage_row<TPR, CPT, NT>(xs + k * CPT * NT, stg, valid);
        cp_async_commit();
    }
    for (int64_t k = 0; k < iters; k++) {
        cp_async_wait<S - 2>();
        if (k + S - 1 < iters) stage_row<TPR, CPT, NT>(xs + ((k + S - 1) % S) * CPT * NT, stg, valid);
        cp_async_commit();
        const int64_t row = base + k * stride + g;
        float f[CPT][V];
        load_row<E, CPT, NT, V>(xs + (k % S) * CPT * NT + threadIdx.x, valid, f);
        if constexpr (LN) center_row<T, TPR, NT, CPT, V>(f, valid, fd, inv_d, red.take());
        Acc2 ss[1] = {acc2_zero()};  // Σ d², d = x (RMSNorm) or x − μ (LayerNorm)
#pragma unroll
        for (int c = 0; c < CPT; c++)
            if (valid >> c & 1u)
#pragma unroll
                for (int v = 0; v < V; v++) s_fma<C>(ss[0], f[c][v], f[c][v]);
        group_reduce<TPR, NT, 1, C>(ss, red.take());
        const float r = rstd_of<C>(s_val(ss[0]), inv_d, eps);
        if (row < N) {
#pragma unroll
            for (int c = 0; c < CPT; c++) {
                if (valid >> c & 1u) {
                    float o[V];
#pragma unroll
                    for (int v = 0; v < V; v++) {
                        const float xh = f[c][v] * r;
                        o[v] = LN ? fmaf(xh, wv[c][v], bv[c][v]) : xh * wv[c][v];
                    }
                    st_stream(yrow + (int64_t)c * TPR * V, E::narrow(o));
                }
            }
        }
        yrow += ystep;
    }
    cp_async_wait<0>();
    pdl_trigger();
}

// ===========================================================================
// Backward stage 1, row path: blockIdx.x = row tile p, rows [ra, rb).  x is
// widened into registers once per row and becomes d in place.  LEAN keeps
// fewer registers (so that more CTAs fit on an SM): w lives in this thread's
// own shared-memory slots (float4 per lane, lane-contiguous: no bank
// conflicts, and no thread reads another's, so no barrier) and dy is widened
// from its staged slot in each pass instead of being held.
// ===========================================================================
template <typename T, bool LN, int TPR, int CPT, int NT, int S, int MINB, bool LEAN>
__global__ void __launch_bounds__(NT, MINB)
    norm_bwd_rows(const T* __restrict__ x, int64_t ldx, const float* __restrict__ w,
                  const T* __restrict__ dy, int64_t lddy, float eps, T* __restrict__ dx,
                  int64_t lddx, float* __restrict__ part, int64_t N, int Dv, int64_t P) {
    using E = Elt<T>;
    constexpr int V = E::V;
    constexpr int R = NT / TPR;
    constexpr bool C = std::is_same<T, float>::value;
    constexpr int K = LN ? 3 : 2;
    const int64_t D = (int64_t)Dv * V;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Raw16* xs = reinterpret_cast<Raw16*>(smem_raw);  // [S][CPT][NT]
    Raw16* gs = xs + S * CPT * NT;                    // [S][CPT][NT]
    __shared__ float2 red_buf[2][K * (NT / 32)];
    RedRing<K * (NT / 32)> red{red_buf, 0};
    const int g = threadIdx.x / TPR, l = threadIdx.x % TPR;
    const float fd = (float)D, inv_d = 1.0f / fd;
    const unsigned valid = chunk_mask<TPR, CPT>(Dv, l);
    int64_t ra, rb;
    norm_tile_rows(blockIdx.x, P, N, ra, rb);
    pdl_wait();
    float wv[CPT][V];
    float4* ws4 = reinterpret_cast<float4*>(smem_raw + (size_t)2 * S * CPT * NT * 16);
    if constexpr (LEAN) {
#pragma unroll
        for (int c = 0; c < CPT; c++) {
            const int ch = l + c * TPR;
#pragma unroll
            for (int q = 0; q < V / 4; q++) {
                const Raw16 r = (ch < Dv) ? ld_keep(w + (int64_t)ch * V + 4 * q) : raw_zero();
                ws4[(c * (V / 4) + q) * NT + threadIdx.x] =
                    make_float4(__uint_as_float(r.u[0]), __uint_as_float(r.u[1]),
                                __uint_as_float(r.u[2]), __uint_as_float(r.u[3]));
            }
        }
    } else {
        load_params<TPR, CPT, V>(w, Dv, l, wv);
    }
    // this thread's w for chunk c
    auto w_of = [&](int c, float (&o)[V]) {
        if constexpr (LEAN) {
#pragma unroll
            for (int q = 0; q < V / 4; q++) {
                const float4 t = ws4[(c * (V / 4) + q) * NT + threadIdx.x];
                o[4 * q] = t.x;
                o[4 * q + 1] = t.y;
                o[4 * q + 2] = t.z;
                o[4 * q + 3] = t.w;
            }
        } else {
#pragma unroll
            for (int v = 0; v < V; v++) o[v] = wv[c][v];
        }
    };
    float aw[CPT][V], ab[CPT][V];
#pragma unroll
    for (int c = 0; c < CPT; c++)
#pragma unroll
        for (int v = 0; v < V; v++) aw[c][v] = ab[c][v] = 0.f;

    const int64_t iters = (rb - ra + R - 1) / R;
    const int64_t ldxb = ldx * (int64_t)sizeof(T), ldgb = lddy * (int64_t)sizeof(T);
    RowStager sx{reinterpret_cast<const char*>(x) + (ra + g) * ldxb + (int64_t)l * 16,
                 reinterpret_cast<const char*>(x), R * ldxb, ra + g, R, rb};
    RowStager sg{reinterpret_cast<const char*>(dy) + (ra + g) * ldgb + (int64_t)l * 16,
                 reinterpret_cast<const char*>(dy), R * ldgb, ra + g, R, rb};
    T* dxrow = dx + (ra + g) * lddx + (int64_t)l * V;
#pragma unroll
    for (int k = 0; k < S - 1; k++) {
        if (k < iters) {
            stage_row<TPR, CPT, NT>(xs + k * CPT * NT, sx, valid);
            stage_row<TPR, CPT, NT>(gs + k * CPT * NT, sg, valid);
        }
        cp_async_commit();
    }
    for (int64_t k = 0; k < iters; k++) {
        cp_async_wait<S - 2>();
        if (k + S - 1 < iters) {
            stage_row<TPR, CPT, NT>(xs + ((k + S - 1) % S) * CPT * NT, sx, valid);
            stage_row<TPR, CPT, NT>(gs + ((k + S - 1) % S) * CPT * NT, sg, valid);
        }
        cp_async_commit();
        const int64_t row = ra + k * R + g;
        const Raw16* cg = gs + (k % S) * CPT * NT + threadIdx.x;
        float f[CPT][V], gd[CPT][V];
        load_row<E, CPT, NT, V>(xs + (k % S) * CPT * NT + threadIdx.x, valid, f);
        if constexpr (!LEAN) load_row<E, CPT, NT, V>(cg, valid, gd);
        // dy of chunk c: held (gd) or widened again from the staged slot
        auto dy_of = [&](int c, float (&o)[V]) {
            if constexpr (LEAN) {
                E::widen(cg[c * NT], o);
            } else {
#pragma unroll
                for (int v = 0; v < V; v++) o[v] = gd[c][v];
            }
        };
        if constexpr (LN) center_row<T, TPR, NT, CPT, V>(f, valid, fd, inv_d, red.take());
        // sums[0] = Σ d², sums[1] = Σ g·d, and for LayerNorm sums[2] = Σ g;
        // d = x (RMSNorm) or x − μ (LayerNorm), g = dy·w
        Acc2 sums[K];
#pragma unroll
        for (int q = 0; q < K; q++) sums[q] = acc2_zero();
        uint64_t a0 = 0ull, a1 = 0ull, a2 = 0ull;  // 16-bit rows: packed lanes
#pragma unroll
        for (int c = 0; c < CPT; c++) {
            if (valid >> c & 1u) {
                float gc[V], wc[V];
                dy_of(c, gc);
                w_of(c, wc);
                if constexpr (C) {
#pragma unroll
                    for (int v = 0; v < V; v++) {
                        const float gg = gc[v] * wc[v];
                        s_fma<C>(sums[0], f[c][v], f[c][v]);
                        s_fma<C>(sums[1], gg, f[c][v]);
                        if constexpr (LN) s_add<C>(sums[2], gg);
                    }
                } else {
#pragma unroll
                    for (int h = 0; h < V / 2; h++) {
                        const uint64_t d2 = f2_pack(f[c][2 * h], f[c][2 * h + 1]);
                        const uint64_t g2 = f2_mul(f2_pack(gc[2 * h], gc[2 * h + 1]),
                                                   f2_pack(wc[2 * h], wc[2 * h + 1]));
                        a0 = f2_fma(d2, d2, a0);
                        a1 = f2_fma(g2, d2, a1);
                        if constexpr (LN) a2 = f2_add(a2, g2);
                    }
                }
            }
        }
        if constexpr (!C) {
            sums[0] = lanes_sum(a0);
            sums[1] = lanes_sum(a1);
            if constexpr (LN) sums[LN ? 2 : 0] = lanes_sum(a2);
        }
        group_reduce<TPR, NT, K, C>(sums, red.take());
        const BwdStats st = bwd_stats<LN, C>(sums, inv_d, eps);
        if (row < rb) {
            const float r = st.r, rmg = st.r * st.mg, rmgx = st.r * st.mgx;
            const uint64_t r2 = f2_pack(r, r), nrmgx2 = f2_pack(-rmgx, -rmgx),
                           nrmg2 = f2_pack(-rmg, -rmg);
#pragma unroll
            for (int c = 0; c < CPT; c++) {
                if (valid >> c & 1u) {
                    float o[V], gc[V], wc[V];
                    dy_of(c, gc);
                    w_of(c, wc);
                    // r·((g − mean g) − x̂·mean(g·x̂)); the LayerNorm form (three
                    // accumulators a column) stays scalar: packed, it spills
                    if constexpr (LN) {
#pragma unroll
                        for (int v = 0; v < V; v++) {
                            const float xh = f[c][v] * r;
                            const float gg = gc[v] * wc[v];
                            o[v] = fmaf(-xh, rmgx, fmaf(gg, r, -rmg));
                            aw[c][v] = fmaf(gc[v], xh, aw[c][v]);
                            ab[c][v] += gc[v];
                        }
                    } else {
#pragma unroll
                        for (int h = 0; h < V / 2; h++) {
                            const uint64_t dy2 = f2_pack(gc[2 * h], gc[2 * h + 1]);
                            const uint64_t xh = f2_mul(f2_pack(f[c][2 * h], f[c][2 * h + 1]), r2);
                            const uint64_t gg = f2_mul(dy2, f2_pack(wc[2 * h], wc[2 * h + 1]));
                            f2_unpack(f2_fma(xh, nrmgx2, f2_fma(gg, r2, nrmg2)), o[2 * h],
                                      o[2 * h + 1]);
                            f2_unpack(f2_fma(dy2, xh, f2_pack(aw[c][2 * h], aw[c][2 * h + 1])),
                                      aw[c][2 * h], aw[c][2 * h + 1]);
                        }
                    }
                    st_stream(dxrow + (int64_t)c * TPR * V, E::narrow(o));
                }
            }
        }
        dxrow += R * lddx;
    }
    cp_async_wait<0>();
    pdl_trigger();
    // Combine the R row groups, in index order, into the tile's partial row(s).
    __syncthreads();
    float* sm = reinterpret_cast<float*>(smem_raw);  // [R][CPT][TPR][V]
    constexpr int NOUT = LN ? 2 : 1;
#pragma unroll
    for (int o = 0; o < NOUT; o++) {
#pragma unroll
        for (int c = 0; c < CPT; c++) {
            float4* dst = reinterpret_cast<float4*>(sm + ((g * CPT + c) * TPR + l) * V);
#pragma unroll
            for (int q = 0; q < V / 4; q++) {
                const float(&a)[CPT][V] = (o == 0) ? aw : ab;
                dst[q] = make_float4(a[c][4 * q], a[c][4 * q + 1], a[c][4 * q + 2],
                                     a[c][4 * q + 3]);
            }
        }
        __syncthreads();
        float* out = part + ((int64_t)o * P + blockIdx.x) * D;
        for (int64_t j = threadIdx.x; j < D; j += NT) {
            const int cid = (int)(j / V), v = (int)(j % V);
            const int c = cid / TPR, ll = cid % TPR;
            float s = sm[(c * TPR + ll) * V + v];
#pragma unroll
            for (int q = 1; q < R; q++) s += sm[((q * CPT + c) * TPR + ll) * V + v];
            out[j] = s;
        }
        __syncthreads();
    }
}

// ===========================================================================
// Cluster path (16-byte aligned rows of 8193..65536 elements).  A row is
// split over a thread-block cluster of CS CTAs of NT = 256 threads: the CTA
// of rank r owns the chunks [r·NT·CPT, (r+1)·NT·CPT) (16 elements a thread,
// 4096 a CTA) and stages them S rows ahead into the threads' private slots.
// The forward holds its slice of w (and b) in registers; the backward keeps
// w in per-thread shared-memory slots, re-widens x and dy from their slots in
// each pass, and holds only the dw/db accumulators of exactly those columns.
// The row sums are reduced inside each warp (xor butterfly)
// and exchanged as one entry a warp with WarpPush: every CTA receives the
// entries of all CS·NT/32 warps of the cluster in its own shared memory;
// warp 0 combines them (lane ℓ takes entries ℓ, ℓ+32, …, then an xor
// butterfly over the lanes) and hands the sums to the other warps through
// shared memory and a CTA barrier (RMSNorm's backward: every warp combines
// them itself, without the barrier), so every CTA derives the same bits of
// the row statistics, with the arithmetic of the row path.
//
// RMSNorm keeps two rows in flight: the sums of row k + 1 are pushed before
// the exchange of row k is awaited, so the exchange's latency overlaps the
// next row's first pass (two turns outstanding: four exchange buffers).
//
// One exchange a row.  LayerNorm's sums about the mean need the mean first.
// The forward carries it one row ahead: the exchange of row k carries Σ d²
// of row k and Σx of row k + 1 (staged already), so that the mean of row
// k + 1 is known when its turn comes; only the first row's Σx is exchanged on
// its own.  The backward takes its sums about a shift s instead, the previous
// row's mean
// (zero for a cluster's first row, or after a row whose mean is not
// finite): d = x − s, and the row's turn carries Σ d², Σ x[, Σ g, Σ g·d].
// The mean μ₀ + c comes from Σ x as on the row path (Σ x compensated across
// warps for every storage type: the plain binary32 row sum that suffices for
// 16-bit rows of the row path is exact only while Σx stays below 2^24 steps
// of the data's grid, i.e. up to 2^24/2^11 = 8192 binary16 elements of one
// binade, 2^24/2^8 = 65536 for bfloat16, and wider binary16 rows with a large
// common offset would shift every x̂ of a row by the rounding of their mean;
// a warp's 512 16-bit elements stay below 2^20 steps, so within a warp they
// are added plainly).  With m = μ − s,
//     Σ (x − μ)² = Σ d² − D·m²,    Σ g·(x − μ) = Σ g·d − m·Σ g
// (exact identities), and the row is centred on μ₀ + c.  The turn of row
// k + 1 is pushed as soon as row k's is read, before row k's second pass,
// which its exchange then overlaps (one turn outstanding: two buffers).
// When the shift is far from the mean the first identity cancels: if D·m² >
// Σ d²/2 (more than one bit lost; also a NaN) the row's sums are taken again
// about μ in a turn of their own — every CTA sees the same sums, so every
// CTA takes the same turns.  Rows whose mean drifts by less than their
// spread from one row to the next never take it.
//
// The forward takes rows cid, cid + ncl, … (cluster cid of ncl).  The
// backward keeps the row tiles of the row path (a function of N alone, so
// dw/db have the same bits on any device): cluster cid takes tiles cid,
// cid + ncl, … one after the other, staging across tile boundaries, and at
// the end of a tile each CTA writes its columns of the tile's partial row.
// Every CTA of a cluster runs the same rows, hence the same exchanges.
// ===========================================================================
constexpr int kNormClusterNT = 256;
// Rows of up to this many elements use CTAs of 128 threads (2048 elements,
// clusters of up to 8, 6 CTAs an SM): at bf16 widths 12,288 / 16,384 this
// measured 2-6% faster than 256 threads; at 32,768 (clusters of 16) slower.
constexpr int64_t kNormClusterSmallMaxD = 16384;
// backward stages (indexed by LayerNorm) and whether w sits in per-thread
// shared-memory slots, for 16-bit and binary32 rows
constexpr int kNormBwdStages16[2] = {3, 3};
constexpr int kNormBwdStages32[2] = {3, 3};
constexpr bool kNormBwdWSlots[2] = {true, true};
constexpr int kNormFwdStages[2] = {4, 4};
constexpr int64_t kNormClusterRowMax = (int64_t)kClusterMaxCS * kNormClusterNT * 16;  // 65536

// Waits of the cluster exchanges that ran out (see WarpPush); zero unless
// the exchange protocol failed.
__device__ unsigned g_norm_wait_timeouts;

// Most CTAs a cluster of CTAs of NT threads takes: 128-thread CTAs serve rows
// of up to kNormClusterSmallMaxD elements (8 CTAs of 2048 elements).
template <int NT>
constexpr int kNormMaxCS = NT == 128 ? 8 : kClusterMaxCS;

template <int NT, int NB = 2, int NV = 2>
using NormPush = WarpPush<NT / 32, kNormMaxCS<NT>*(NT / 32), NV, NB>;

__device__ __forceinline__ Acc2 warp_sum(Acc2 v, bool comp) {
    return comp ? group_sum2<32>(v) : Acc2{group_sum<32>(v.hi), 0.f};
}

// An entry carries K sums as float4s: as (hi, lo) pairs, two to a float4,
// or, when no sum is compensated (CM = 0, so every lo is zero), as values,
// four to a float4.
template <int K, unsigned CM>
constexpr int kEntryX = CM == 0 ? (K + 3) / 4 : (K + 1) / 2;

template <int K, unsigned CM>
__device__ __forceinline__ void entry_put(float4* e, const Acc2 (&v)[K]) {
    float f[4 * kEntryX<K, CM>];
#pragma unroll
    for (int i = 0; i < 4 * kEntryX<K, CM>; i++) f[i] = 0.f;
#pragma unroll
    for (int q = 0; q < K; q++) {
        if constexpr (CM == 0) {
            f[q] = v[q].hi;
        } else {
            f[2 * q] = v[q].hi;
            f[2 * q + 1] = v[q].lo;
        }
    }
#pragma unroll
    for (int n = 0; n < kEntryX<K, CM>; n++)
        e[n] = make_float4(f[4 * n], f[4 * n + 1], f[4 * n + 2], f[4 * n + 3]);
}

template <unsigned CM>
__device__ __forceinline__ Acc2 entry_get(const float4* e, int q) {
    if constexpr (CM == 0) {
        const float4 v = e[q / 4];
        const int h = q % 4;
        return Acc2{h == 0 ? v.x : h == 1 ? v.y : h == 2 ? v.z : v.w, 0.f};
    } else {
        const float4 v = e[q / 2];
        return (q & 1) ? Acc2{v.z, v.w} : Acc2{v.x, v.y};
    }
}

// Add the K sums of one entry into s (compensated for the sums in CM).
template <int K, unsigned CM>
__device__ __forceinline__ void entry_add(Acc2 (&s)[K], const float4* e) {
#pragma unroll
    for (int q = 0; q < K; q++) {
        const Acc2 o = entry_get<CM>(e, q);
        s[q] = ((CM >> q) & 1u) ? acc2_add(s[q], o) : Acc2{s[q].hi + o.hi, 0.f};
    }
}

// Sum K (up to 4) row sums over the cluster in two steps.  cluster_push: each
// warp's sums (xor butterfly; compensated for the sums in CMW) pushed as the
// warp's entry; returns the turn.  cluster_finish: warp 0 waits for the turn,
// combines the entries (lane ℓ takes entries ℓ, ℓ+32, …, then an xor
// butterfly; compensated for the sums in CM) and posts the sums in `out`
// (one of two slots, taken in turn by successive calls, so that a slot is
// written again only after the CTA barrier of the call in between); a CTA
// barrier hands them to every warp (and orders the turn's reads before any
// warp's later pushes).  Every thread of every CTA of the cluster calls
// both together; other work may sit between them (other turns' pushes when
// NB is 4 or more).
template <int NT, int K, unsigned CM, unsigned CMW, int NB, int NV>
__device__ __forceinline__ unsigned cluster_push(Acc2 (&v)[K], NormPush<NT, NB, NV>& xp) {
    static_assert(K >= 1 && K <= 4, "up to four sums");
    static_assert((CMW & ~CM) == 0, "warp-level compensation implies exchange-level");
    Acc2 w[K];
#pragma unroll
    for (int q = 0; q < K; q++) w[q] = warp_sum(v[q], (CMW >> q) & 1u);
    float4 e[kEntryX<K, CM>];
    entry_put<K, CM>(e, w);
    return xp.template push<kEntryX<K, CM>>(e);
}

template <int NT, int K, unsigned CM, int NB, int NV>
__device__ __forceinline__ void cluster_finish(unsigned t, Acc2 (&v)[K], NormPush<NT, NB, NV>& xp,
                                               float4* out) {
    constexpr int W = NT / 32;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x < 32) {
        const float4(*buf)[NV] = xp.wait(t);
        const int total = (int)cluster_nctarank() * W;
        Acc2 s[K];
#pragma unroll
        for (int q = 0; q < K; q++) s[q] = acc2_zero();
        for (int j = lane; j < total; j += 32) entry_add<K, CM>(s, buf[j]);  // bound uniform
#pragma unroll
        for (int q = 0; q < K; q++) s[q] = warp_sum(s[q], (CM >> q) & 1u);
        if (lane == 0) entry_put<K, CM>(out, s);
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < K; q++) v[q] = entry_get<CM>(out, q);
}

// cluster_finish without the CTA barrier: every warp waits for turn t and
// combines the entries itself, in the same order, so every warp of every CTA
// derives the same bits.  The __syncwarp orders the warp's reads of the
// turn's buffer before its later pushes, whose release lets the other CTAs
// write that buffer again.  For callers that push turn t + 1 before reading
// turn t and turn t + 2 after it (NB = 4): a CTA writes a buffer again, turn
// t + 4, only after every warp of the cluster pushed turn t + 2.
template <int NT, int K, unsigned CM, int NB, int NV>
__device__ __forceinline__ void cluster_combine(unsigned t, Acc2 (&v)[K],
                                                NormPush<NT, NB, NV>& xp) {
    static_assert(NB == 4, "two turns outstanding");
    constexpr int W = NT / 32;
    const int lane = threadIdx.x & 31;
    const float4(*buf)[NV] = xp.wait(t);
    const int total = (int)cluster_nctarank() * W;
#pragma unroll
    for (int q = 0; q < K; q++) v[q] = acc2_zero();
    for (int j = lane; j < total; j += 32) entry_add<K, CM>(v, buf[j]);  // bound uniform
    __syncwarp();
#pragma unroll
    for (int q = 0; q < K; q++) v[q] = warp_sum(v[q], (CM >> q) & 1u);
}

template <int NT, int K, unsigned CM, unsigned CMW = CM, int NB, int NV>
__device__ __forceinline__ void cluster_reduce(Acc2 (&v)[K], NormPush<NT, NB, NV>& xp,
                                               float4* out) {
    const unsigned t = cluster_push<NT, K, CM, CMW, NB, NV>(v, xp);
    cluster_finish<NT, K, CM, NB, NV>(t, v, xp, out);
}

// Σx over this thread's valid chunks of a staged row: binary32 elements with
// TwoSum each; 16-bit elements (8 or 11 significant bits) in plain binary32,
// as are the warp's 512 (fewer than 2^20 steps of one binade's grid): exact
// unless a warp's elements span more than 7 (bfloat16) or 4 (binary16)
// binades, and then off by a few roundings of 2^-24 of the warp's partial
// sum.  The levels above the warp are compensated.
template <typename E, int CPT, int NT, int V, bool Comp>
__device__ __forceinline__ Acc2 staged_sum_x(const Raw16* slot, unsigned valid) {
    Acc2 s = acc2_zero();
    float s1 = 0.f;
#pragma unroll
    for (int c = 0; c < CPT; c++) {
        if (valid >> c & 1u) {
            float f[V];
            E::widen(slot[c * NT], f);
#pragma unroll
            for (int v = 0; v < V; v++) {
                if constexpr (Comp)
                    s_add<true>(s, f[v]);
                else if (v & 1)
                    s1 += f[v];
                else
                    s.hi += f[v];
            }
        }
    }
    if constexpr (!Comp) s.hi += s1;
    return s;
}

// Σx² over this thread's valid chunks of a staged row (the arithmetic of the
// in-register Σ d² of RMSNorm).
template <typename E, int CPT, int NT, int V, bool Comp>
__device__ __forceinline__ Acc2 staged_sum_sq(const Raw16* slot, unsigned valid) {
    Acc2 s = acc2_zero();
    uint64_t a = 0ull;  // 16-bit rows: even and odd columns in two packed lanes
#pragma unroll
    for (int c = 0; c < CPT; c++) {
        if (valid >> c & 1u) {
            float f[V];
            E::widen(slot[c * NT], f);
            if constexpr (Comp) {
#pragma unroll
                for (int v = 0; v < V; v++) s_fma<Comp>(s, f[v], f[v]);
            } else {
#pragma unroll
                for (int h = 0; h < V / 2; h++) {
                    const uint64_t d = f2_pack(f[2 * h], f[2 * h + 1]);
                    a = f2_fma(d, d, a);
                }
            }
        }
    }
    if constexpr (!Comp) {
        float a0, a1;
        f2_unpack(a, a0, a1);
        s.hi = a0 + a1;
    }
    return s;
}

template <int CPT, int V>
__device__ __forceinline__ void center(float (&f)[CPT][V], unsigned valid, const Mean& m) {
#pragma unroll
    for (int c = 0; c < CPT; c++)
        if (valid >> c & 1u)
#pragma unroll
            for (int v = 0; v < V; v++) f[c][v] = (f[c][v] - m.mu0) - m.c;
}

// center on packed pairs: (x − μ₀) − c per lane, the bits of `center`.
template <int CPT, int V>
__device__ __forceinline__ void center2(float (&f)[CPT][V], unsigned valid, const Mean& m) {
    const uint64_t mu2 = f2_pack(m.mu0, m.mu0), c2 = f2_pack(m.c, m.c);
#pragma unroll
    for (int c = 0; c < CPT; c++)
        if (valid >> c & 1u)
#pragma unroll
            for (int q = 0; q < V / 2; q++)
                f2_unpack(f2_sub(f2_sub(f2_pack(f[c][2 * q], f[c][2 * q + 1]), mu2), c2),
                          f[c][2 * q], f[c][2 * q + 1]);
}

// Plain binary32 Σ f² over the valid chunks, even and odd columns in two
// packed lanes, the lanes added at the end (16-bit rows).
template <int CPT, int V>
__device__ __forceinline__ Acc2 sum_sq2(const float (&f)[CPT][V], unsigned valid) {
    uint64_t a = 0ull;
#pragma unroll
    for (int c = 0; c < CPT; c++)
        if (valid >> c & 1u)
#pragma unroll
            for (int q = 0; q < V / 2; q++) {
                const uint64_t d = f2_pack(f[c][2 * q], f[c][2 * q + 1]);
                a = f2_fma(d, d, a);
            }
    float a0, a1;
    f2_unpack(a, a0, a1);
    return Acc2{a0 + a1, 0.f};
}

// Whether sums about a shift give Σ (x − μ)² = Σ d² − D·m² (m = μ − s) to
// within one bit of cancellation: D·m² ≤ Σ d² / 2.  Otherwise the row's
// sums are taken again about μ.  False for NaN sums.
__device__ __forceinline__ bool shift_ok(float sdd, float m, float fd) {
    return fd * m * m <= 0.5f * sdd;
}

template <typename T, bool LN, int NT, int S>
__global__ void __launch_bounds__(NT, 768 / NT)
    norm_fwd_cluster(const T* __restrict__ x, int64_t ldx, const float* __restrict__ w,
                     const float* __restrict__ b, float eps, T* __restrict__ y, int64_t ldy,
                     int64_t N, int Dv) {
    using E = Elt<T>;
    constexpr int V = E::V, CPT = 16 / V;
    constexpr bool C = std::is_same<T, float>::value;
    // RMSNorm keeps two rows in flight: row k + 1's Σx² is pushed before
    // row k's exchange is awaited (four exchange buffers, see WarpPush)
    constexpr bool PIPE = !LN;
    constexpr int NB = PIPE ? 4 : 2;
    static_assert(S >= 3, "two staged rows");
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Raw16* xs = reinterpret_cast<Raw16*>(smem_raw);  // [S][CPT][NT]
    constexpr int NV = 1;  // one float4 an entry: up to two sums
    __shared__ __align__(16) float4 xbuf[NB][kNormMaxCS<NT> * (NT / 32)][NV];
    __shared__ __align__(8) uint64_t xbar[NB];
    __shared__ __align__(16) float4 xres[2][2];  // combined sums, by turn parity
    NormPush<NT, NB, NV> xc{xbuf, xbar, &g_norm_wait_timeouts, 0u, true};
    xc.init();
    cluster_sync();
    const int l = (int)cluster_ctarank() * NT * CPT + (int)threadIdx.x;  // chunk l + c·NT
    const float fd = (float)(Dv * V), inv_d = 1.0f / fd;
    const unsigned valid = chunk_mask<NT, CPT>(Dv, l);
    const int64_t cid = cluster_id_x(), ncl = cluster_count_x();
    const int64_t iters = cid < N ? (N - 1 - cid) / ncl + 1 : 0;
    pdl_wait();
    float wv[CPT][V], bv[CPT][V];
    load_params<NT, CPT, V>(w, Dv, l, wv);
    if constexpr (LN) load_params<NT, CPT, V>(b, Dv, l, bv);
    const int64_t ldb = ldx * (int64_t)sizeof(T);
    RowStager stg{reinterpret_cast<const char*>(x) + cid * ldb + (int64_t)l * 16,
                  reinterpret_cast<const char*>(x), ncl * ldb, cid, ncl, N};
    T* yrow = y + cid * ldy + (int64_t)l * V;
    const int64_t ystep = ncl * ldy;
#pragma unroll
    for (int k = 0; k < S - 1; k++) {
        if (k < iters) stage_row<NT, CPT, NT>(xs + k * CPT * NT, stg, valid);
        cp_async_commit();
    }
    Mean mn{0.f, 0.f};
    if (LN && iters > 0) {  // the first row's Σx
        cp_async_wait<S - 2>();
        Acc2 s0[1] = {staged_sum_x<E, CPT, NT, V, C>(xs + threadIdx.x, valid)};
        cluster_reduce<NT, 1, 1u, C ? 1u : 0u>(s0, xc, xres[0]);
        mn = mean_of(s0[0], fd, inv_d);
    }
    if (PIPE && iters > 0) {  // the first row's Σx², turn 0
        cp_async_wait<S - 2>();
        Acc2 q[1] = {staged_sum_sq<E, CPT, NT, V, C>(xs + threadIdx.x, valid)};
        cluster_push<NT, 1, C ? 1u : 0u, C ? 1u : 0u>(q, xc);
    }
    for (int64_t k = 0; k < iters; k++) {
        cp_async_wait<S - 3>();  // rows k and k + 1
        if (k + S - 1 < iters) stage_row<NT, CPT, NT>(xs + ((k + S - 1) % S) * CPT * NT, stg, valid);
        cp_async_commit();
        // LayerNorm centres the row before its sums; RMSNorm loads it after
        // its turn (fewer registers live across the exchange)
        float f[CPT][V];
        if constexpr (LN) {
            load_row<E, CPT, NT, V>(xs + (k % S) * CPT * NT + threadIdx.x, valid, f);
            if constexpr (C)
                center<CPT, V>(f, valid, mn);
            else
                center2<CPT, V>(f, valid, mn);
        }
        if constexpr (PIPE) {
            if (k + 1 < iters) {  // row k + 1's Σx², turn k + 1
                Acc2 q[1] = {staged_sum_sq<E, CPT, NT, V, C>(
                    xs + ((k + 1) % S) * CPT * NT + threadIdx.x, valid)};
                cluster_push<NT, 1, C ? 1u : 0u, C ? 1u : 0u>(q, xc);
            }
        }
        // Σ d², d = x (RMSNorm) or x − μ (LayerNorm); LayerNorm: Σx of row k + 1
        Acc2 sm[LN ? 2 : 1];
        sm[0] = acc2_zero();
        if constexpr (LN) {
            if constexpr (C) {
#pragma unroll
                for (int c = 0; c < CPT; c++)
                    if (valid >> c & 1u)
#pragma unroll
                        for (int v = 0; v < V; v++) s_fma<C>(sm[0], f[c][v], f[c][v]);
            } else {
                sm[0] = sum_sq2<CPT, V>(f, valid);
            }
            sm[LN ? 1 : 0] = k + 1 < iters
                ? staged_sum_x<E, CPT, NT, V, C>(xs + ((k + 1) % S) * CPT * NT + threadIdx.x, valid)
                : acc2_zero();
            cluster_reduce<NT, 2, (C ? 1u : 0u) | 2u, C ? 3u : 0u>(sm, xc, xres[(k + 1) & 1]);
        } else {
            cluster_finish<NT, 1, C ? 1u : 0u>((unsigned)k, sm, xc, xres[k & 1]);  // row k's turn
            load_row<E, CPT, NT, V>(xs + (k % S) * CPT * NT + threadIdx.x, valid, f);
        }
        const float r = rstd_of<C>(s_val(sm[0]), inv_d, eps);
        if constexpr (LN) mn = mean_of(sm[LN ? 1 : 0], fd, inv_d);
        const uint64_t r2 = f2_pack(r, r);
#pragma unroll
        for (int c = 0; c < CPT; c++) {
            if (valid >> c & 1u) {
                float o[V];
#pragma unroll
                for (int q = 0; q < V / 2; q++) {
                    // x̂·w (+ b) on two columns at once, each lane rounded as the
                    // scalar form would be
                    const uint64_t xh = f2_mul(f2_pack(f[c][2 * q], f[c][2 * q + 1]), r2);
                    const uint64_t w2 = f2_pack(wv[c][2 * q], wv[c][2 * q + 1]);
                    f2_unpack(LN ? f2_fma(xh, w2, f2_pack(bv[c][2 * q], bv[c][2 * q + 1]))
                                 : f2_mul(xh, w2),
                              o[2 * q], o[2 * q + 1]);
                }
                st_stream(yrow + (int64_t)c * NT * V, E::narrow(o));
            }
        }
        yrow += ystep;
    }
    cp_async_wait<0>();
    cluster_sync();
    pdl_trigger();
}

// A cursor over the rows of tiles t, t + step, … (of P tiles over N rows).
struct TileCursor {
    int tile;
    int64_t row, end;
};

__device__ __forceinline__ void tile_seek(TileCursor& c, int P, int64_t N) {
    if (c.tile < P)
        norm_tile_rows(c.tile, P, N, c.row, c.end);
    else
        c.row = c.end = 0;
}

__device__ __forceinline__ void tile_advance(TileCursor& c, int step, int P, int64_t N) {
    if (++c.row == c.end) {
        c.tile += step;
        tile_seek(c, P, N);
    }
}

// binary32 rows: at most four CTAs an SM fit their staged rows, so their
// threads may hold more registers
template <typename T, bool LN, int NT, int S, bool WS>
__global__ void __launch_bounds__(NT, (std::is_same<T, float>::value ? 512 : 768) / NT)
    norm_bwd_cluster(const T* __restrict__ x, int64_t ldx, const float* __restrict__ w,
                     const T* __restrict__ dy, int64_t lddy, float eps, T* __restrict__ dx,
                     int64_t lddx, float* __restrict__ part, int64_t N, int Dv, int64_t P) {
    using E = Elt<T>;
    constexpr int V = E::V, CPT = 16 / V;
    constexpr bool C = std::is_same<T, float>::value;
    static_assert(S >= 3, "two staged rows");
    // sums: Σ d², Σ g·d[, Σ g, Σ x], d = x (RMSNorm) or x − s (LayerNorm,
    // about a shift s); Σ x is compensated across warps for every type
    constexpr int K = LN ? 4 : 2;
    constexpr unsigned CM = (C ? (LN ? 7u : 3u) : 0u) | (LN ? 8u : 0u);
    // Two rows in flight.  RMSNorm pushes row k + 1's sums before awaiting
    // row k's exchange (four exchange buffers, see WarpPush).  LayerNorm
    // takes its sums about a shift, the previous row's mean, and pushes row
    // k + 1's sums once row k's turn is read, before row k's second pass,
    // which its exchange overlaps (one turn outstanding: two buffers); when
    // the shift is far from the row's mean, the sums are taken again about
    // the mean in a turn of their own.
    constexpr int NB = LN ? 2 : 4, NV = kEntryX<K, CM>;
    const int64_t D = (int64_t)Dv * V;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Raw16* xs = reinterpret_cast<Raw16*>(smem_raw);  // [S][CPT][NT]
    Raw16* gs = xs + S * CPT * NT;                    // [S][CPT][NT]
    __shared__ __align__(16) float4 xbuf[NB][kNormMaxCS<NT> * (NT / 32)][NV];
    __shared__ __align__(8) uint64_t xbar[NB];
    __shared__ __align__(16) float4 xres[2][2];  // combined sums, by turn parity
    NormPush<NT, NB, NV> xc{xbuf, xbar, &g_norm_wait_timeouts, 0u, true};
    xc.init();
    cluster_sync();
    const int l = (int)cluster_ctarank() * NT * CPT + (int)threadIdx.x;
    const float fd = (float)D, inv_d = 1.0f / fd;
    const unsigned valid = chunk_mask<NT, CPT>(Dv, l);
    const int64_t cid = cluster_id_x(), ncl = cluster_count_x();
    pdl_wait();
    // w of chunk c: this thread's own shared-memory slots (WS), or read-only
    // loads of the CTA's slice
    float4* ws4 = reinterpret_cast<float4*>(gs + S * CPT * NT);  // [CPT·V/4][NT]
    if constexpr (WS) {
#pragma unroll
        for (int c = 0; c < CPT; c++) {
            const int ch = l + c * NT;
#pragma unroll
            for (int q = 0; q < V / 4; q++) {
                const Raw16 r = (ch < Dv) ? ld_keep(w + (int64_t)ch * V + 4 * q) : raw_zero();
                ws4[(c * (V / 4) + q) * NT + threadIdx.x] =
                    make_float4(__uint_as_float(r.u[0]), __uint_as_float(r.u[1]),
                                __uint_as_float(r.u[2]), __uint_as_float(r.u[3]));
            }
        }
    }
    auto w_of = [&](int c, float (&o)[V]) {
#pragma unroll
        for (int q = 0; q < V / 4; q++) {
            float4 t;
            if constexpr (WS) {
                t = ws4[(c * (V / 4) + q) * NT + threadIdx.x];
            } else {
                const Raw16 r = ld_keep(w + (int64_t)(l + c * NT) * V + 4 * q);
                t = make_float4(__uint_as_float(r.u[0]), __uint_as_float(r.u[1]),
                                __uint_as_float(r.u[2]), __uint_as_float(r.u[3]));
            }
            o[4 * q] = t.x;
            o[4 * q + 1] = t.y;
            o[4 * q + 2] = t.z;
            o[4 * q + 3] = t.w;
        }
    };
    // rows of this cluster: its tiles in order
    int64_t iters = 0;
    for (int64_t t = cid; t < P; t += ncl) {
        int64_t a, b2;
        norm_tile_rows(t, P, N, a, b2);
        iters += b2 - a;
    }
    const int Pi = (int)P, step = (int)ncl;
    TileCursor cw{(int)cid, 0, 0}, sw{(int)cid, 0, 0};
    tile_seek(cw, Pi, N);
    tile_seek(sw, Pi, N);
    const int64_t ldxb = ldx * (int64_t)sizeof(T), ldgb = lddy * (int64_t)sizeof(T);
    const char* xb = reinterpret_cast<const char*>(x) + (int64_t)l * 16;
    const char* gb = reinterpret_cast<const char*>(dy) + (int64_t)l * 16;
    auto stage = [&](int slot) {
        if (sw.tile < Pi) {
            const char* px = xb + sw.row * ldxb;
            const char* pg = gb + sw.row * ldgb;
#pragma unroll
            for (int c = 0; c < CPT; c++) {
                const bool ok = valid >> c & 1u;
                cp_async16(&xs[(slot * CPT + c) * NT + threadIdx.x],
                           ok ? px + c * NT * 16 : reinterpret_cast<const char*>(x), ok ? 16 : 0);
                cp_async16(&gs[(slot * CPT + c) * NT + threadIdx.x],
                           ok ? pg + c * NT * 16 : reinterpret_cast<const char*>(dy), ok ? 16 : 0);
            }
            tile_advance(sw, step, Pi, N);
        }
    };
    float aw[CPT][V], ab[CPT][V];
#pragma unroll
    for (int c = 0; c < CPT; c++)
#pragma unroll
        for (int v = 0; v < V; v++) aw[c][v] = ab[c][v] = 0.f;
#pragma unroll
    for (int k = 0; k < S - 1; k++) {
        stage(k);
        cp_async_commit();
    }
    // row sums of the staged row in `slot` (g = dy·w): Σ d², Σ g·d[, Σ g,
    // Σ x], d = x (RMSNorm) or x − sh (LayerNorm)
    auto row_sums = [&](int slot, float sh, Acc2 (&q)[K]) {
        const Raw16* px = xs + slot * CPT * NT + threadIdx.x;
        const Raw16* pg = gs + slot * CPT * NT + threadIdx.x;
#pragma unroll
        for (int n = 0; n < K; n++) q[n] = acc2_zero();
        uint64_t a0 = 0ull, a1 = 0ull, a2 = 0ull, a3 = 0ull;  // 16-bit rows: packed lanes
        const uint64_t sh2 = f2_pack(sh, sh);
#pragma unroll
        for (int c = 0; c < CPT; c++) {
            if (valid >> c & 1u) {
                float dc[V], gc[V], wc[V];
                E::widen(px[c * NT], dc);
                E::widen(pg[c * NT], gc);
                w_of(c, wc);
                if constexpr (C) {
#pragma unroll
                    for (int v = 0; v < V; v++) {
                        const float d = LN ? dc[v] - sh : dc[v];
                        const float gg = gc[v] * wc[v];
                        s_fma<C>(q[0], d, d);
                        s_fma<C>(q[1], gg, d);
                        if constexpr (LN) {
                            s_add<C>(q[LN ? 2 : 0], gg);
                            s_add<C>(q[LN ? 3 : 0], dc[v]);  // Σ x
                        }
                    }
                } else {
#pragma unroll
                    for (int h = 0; h < V / 2; h++) {
                        const uint64_t x2 = f2_pack(dc[2 * h], dc[2 * h + 1]);
                        const uint64_t d2 = LN ? f2_sub(x2, sh2) : x2;
                        const uint64_t g2 = f2_mul(f2_pack(gc[2 * h], gc[2 * h + 1]),
                                                   f2_pack(wc[2 * h], wc[2 * h + 1]));
                        a0 = f2_fma(d2, d2, a0);
                        a1 = f2_fma(g2, d2, a1);
                        if constexpr (LN) {
                            a2 = f2_add(a2, g2);
                            a3 = f2_add(a3, x2);
                        }
                    }
                }
            }
        }
        if constexpr (!C) {
            q[0] = lanes_sum(a0);
            q[1] = lanes_sum(a1);
            if constexpr (LN) {
                q[LN ? 2 : 0] = lanes_sum(a2);
                q[LN ? 3 : 0] = lanes_sum(a3);
            }
        }
    };
    // LayerNorm: the shift of row k and the turn of row k
    float s_cur = 0.f;
    unsigned t_cur = 0u;
    if (iters > 0) {  // the first row's sums
        cp_async_wait<S - 2>();
        Acc2 q[K];
        row_sums(0, 0.f, q);
        t_cur = cluster_push<NT, K, CM, C ? CM : 0u>(q, xc);
    }
    for (int64_t k = 0; k < iters; k++) {
        cp_async_wait<S - 3>();  // rows k and k + 1
        stage((int)((k + S - 1) % S));
        cp_async_commit();
        const int64_t row = cw.row;
        const Raw16* cx = xs + (k % S) * CPT * NT + threadIdx.x;
        const Raw16* cg = gs + (k % S) * CPT * NT + threadIdx.x;
        auto push_next = [&](float sh) {  // row k + 1's sums
            Acc2 q[K];
            row_sums((int)((k + 1) % S), sh, q);
            return cluster_push<NT, K, CM, C ? CM : 0u>(q, xc);
        };
        if (!LN && k + 1 < iters) push_next(0.f);
        // d of chunk c (x, or x − μ with μ = μ₀ + c), widened from the staged
        // slot in each pass rather than held across the exchange
        auto d_of = [&](int c, const Mean& m, float (&o)[V]) {
            E::widen(cx[c * NT], o);
            if constexpr (LN) {
                if constexpr (C) {
#pragma unroll
                    for (int v = 0; v < V; v++) o[v] = (o[v] - m.mu0) - m.c;
                } else {
                    const uint64_t mu2 = f2_pack(m.mu0, m.mu0), mc2 = f2_pack(m.c, m.c);
#pragma unroll
                    for (int h = 0; h < V / 2; h++)
                        f2_unpack(f2_sub(f2_sub(f2_pack(o[2 * h], o[2 * h + 1]), mu2), mc2),
                                  o[2 * h], o[2 * h + 1]);
                }
            }
        };
        // row k's turn: Σ (x − μ)², Σ g·(x − μ)[, Σ g]
        Acc2 sums[K];
        Mean mn{0.f, 0.f};
        float ss, sgd, sg = 0.f;
        if constexpr (LN) {
            cluster_finish<NT, K, CM>(t_cur, sums, xc, xres[t_cur & 1u]);
            const float sdd = s_val(sums[0]);
            mn = mean_of(sums[LN ? 3 : 0], fd, inv_d);
            const float m = (mn.mu0 - s_cur) + mn.c;  // μ − s
            sg = s_val(sums[LN ? 2 : 0]);
            ss = sdd - fd * m * m;
            sgd = s_val(sums[1]) - m * sg;
            if (!shift_ok(sdd, m, fd)) {  // the same in every thread of the cluster
                Acc2 q[2] = {acc2_zero(), acc2_zero()};
                uint64_t a0 = 0ull, a1 = 0ull;
#pragma unroll
                for (int c = 0; c < CPT; c++) {
                    if (valid >> c & 1u) {
                        float dc[V], gc[V], wc[V];
                        d_of(c, mn, dc);
                        E::widen(cg[c * NT], gc);
                        w_of(c, wc);
                        if constexpr (C) {
#pragma unroll
                            for (int v = 0; v < V; v++) {
                                s_fma<C>(q[0], dc[v], dc[v]);
                                s_fma<C>(q[1], gc[v] * wc[v], dc[v]);
                            }
                        } else {
#pragma unroll
                            for (int h = 0; h < V / 2; h++) {
                                const uint64_t d2 = f2_pack(dc[2 * h], dc[2 * h + 1]);
                                const uint64_t g2 = f2_mul(f2_pack(gc[2 * h], gc[2 * h + 1]),
                                                           f2_pack(wc[2 * h], wc[2 * h + 1]));
                                a0 = f2_fma(d2, d2, a0);
                                a1 = f2_fma(g2, d2, a1);
                            }
                        }
                    }
                }
                if constexpr (!C) {
                    q[0] = lanes_sum(a0);
                    q[1] = lanes_sum(a1);
                }
                cluster_reduce<NT, 2, C ? 3u : 0u, C ? 3u : 0u>(q, xc, xres[(t_cur + 1u) & 1u]);
                ss = s_val(q[0]);
                sgd = s_val(q[1]);
            }
            if (k + 1 < iters) {  // row k + 1's sums, about this row's mean
                s_cur = mn.mu0 + mn.c;
                if (!isfinite(s_cur)) s_cur = 0.f;  // a row with a NaN or ∞ shifts no other
                t_cur = push_next(s_cur);
            }
        } else {
            cluster_combine<NT, K, CM>((unsigned)k, sums, xc);  // row k's turn, in every warp
            ss = s_val(sums[0]);
            sgd = s_val(sums[1]);
        }
        const float r = rstd_of<C>(ss, inv_d, eps);
        const float rmgx = r * (r * (sgd * inv_d));
        const float rmg = LN ? r * (sg * inv_d) : 0.f;
        T* dxrow = dx + row * lddx + (int64_t)l * V;
        const uint64_t r2 = f2_pack(r, r), nrmgx2 = f2_pack(-rmgx, -rmgx),
                       nrmg2 = f2_pack(-rmg, -rmg);
#pragma unroll
        for (int c = 0; c < CPT; c++) {
            if (valid >> c & 1u) {
                float o[V], dc[V], gc[V], wc[V];
                d_of(c, mn, dc);
                E::widen(cg[c * NT], gc);
                w_of(c, wc);
                // dx = r·((g − mean g) − x̂·mean(g·x̂)), g = dy·w, two columns
                // an instruction (each lane rounded as the scalar form would be)
#pragma unroll
                for (int h = 0; h < V / 2; h++) {
                    const uint64_t dy2 = f2_pack(gc[2 * h], gc[2 * h + 1]);
                    const uint64_t xh = f2_mul(f2_pack(dc[2 * h], dc[2 * h + 1]), r2);
                    const uint64_t gg = f2_mul(dy2, f2_pack(wc[2 * h], wc[2 * h + 1]));
                    f2_unpack(f2_fma(xh, nrmgx2, f2_fma(gg, r2, nrmg2)), o[2 * h], o[2 * h + 1]);
                    f2_unpack(f2_fma(dy2, xh, f2_pack(aw[c][2 * h], aw[c][2 * h + 1])),
                              aw[c][2 * h], aw[c][2 * h + 1]);
                    if constexpr (LN)
                        f2_unpack(f2_add(f2_pack(ab[c][2 * h], ab[c][2 * h + 1]), dy2),
                                  ab[c][2 * h], ab[c][2 * h + 1]);
                }
                st_stream(dxrow + (int64_t)c * NT * V, E::narrow(o));
            }
        }
        if (row + 1 == cw.end) {  // the tile's last row: its partial row(s)
            float* pw = part + cw.tile * D;
            float* pb = part + (P + cw.tile) * D;
#pragma unroll
            for (int c = 0; c < CPT; c++) {
                if (valid >> c & 1u) {
                    const int64_t col = (int64_t)(l + c * NT) * V;
#pragma unroll
                    for (int v = 0; v < V; v++) {
                        pw[col + v] = aw[c][v];
                        aw[c][v] = 0.f;
                        if constexpr (LN) {
                            pb[col + v] = ab[c][v];
                            ab[c][v] = 0.f;
                        }
                    }
                }
            }
        }
        tile_advance(cw, step, Pi, N);
    }
    cp_async_wait<0>();
    cluster_sync();
    pdl_trigger();
}

// ===========================================================================
// Element-wise paths (any alignment, any D): one CTA per row (forward) or per
// row tile (backward), several passes over each row.
// ===========================================================================
template <typename T, bool LN, int NT>
__global__ void __launch_bounds__(NT)
    norm_fwd_scalar(const T* __restrict__ x, int64_t ldx, const float* __restrict__ w,
                    const float* __restrict__ b, float eps, T* __restrict__ y, int64_t ldy,
                    int64_t N, int64_t D) {
    using E = Elt<T>;
    constexpr bool C = std::is_same<T, float>::value;
    __shared__ float2 red_buf[2][NT / 32];
    RedRing<NT / 32> red{red_buf, 0};
    const float fd = (float)D, inv_d = 1.0f / fd;
    pdl_wait();
    for (int64_t row = blockIdx.x; row < N; row += gridDim.x) {
        const T* xr = x + row * ldx;
        Mean m{0.f, 0.f};
        if constexpr (LN) {
            Acc2 s[1] = {acc2_zero()};
            for (int64_t j = threadIdx.x; j < D; j += NT) s_add<true>(s[0], E::load1(xr + j));
            group_reduce<NT, NT, 1, true>(s, red.take());
            m = mean_of(s[0], fd, inv_d);
        }
        Acc2 ss[1] = {acc2_zero()};
        for (int64_t j = threadIdx.x; j < D; j += NT) {
            const float d = (E::load1(xr + j) - m.mu0) - m.c;
            s_fma<C>(ss[0], d, d);
        }
        group_reduce<NT, NT, 1, C>(ss, red.take());
        const float r = rstd_of<C>(s_val(ss[0]), inv_d, eps);
        for (int64_t j = threadIdx.x; j < D; j += NT) {
            const float xh = ((E::load1(xr + j) - m.mu0) - m.c) * r;
            E::store1(y + row * ldy + j,
                      LN ? fmaf(xh, __ldg(w + j), __ldg(b + j)) : xh * __ldg(w + j));
        }
    }
    pdl_trigger();
}

template <typename T, bool LN, int NT>
__global__ void __launch_bounds__(NT)
    norm_bwd_scalar(const T* __restrict__ x, int64_t ldx, const float* __restrict__ w,
                    const T* __restrict__ dy, int64_t lddy, float eps, T* __restrict__ dx,
                    int64_t lddx, float* __restrict__ part, int64_t N, int64_t D, int64_t P) {
    using E = Elt<T>;
    constexpr bool C = std::is_same<T, float>::value;
    constexpr int K = LN ? 3 : 2;
    __shared__ float2 red_buf[2][K * (NT / 32)];
    RedRing<K * (NT / 32)> red{red_buf, 0};
    const float fd = (float)D, inv_d = 1.0f / fd;
    int64_t ra, rb;
    norm_tile_rows(blockIdx.x, P, N, ra, rb);
    pdl_wait();
    // thread t owns the columns j ≡ t (mod NT) of the tile's partial row(s)
    float* pw = part + (int64_t)blockIdx.x * D;
    float* pb = part + ((int64_t)P + blockIdx.x) * D;
    for (int64_t j = threadIdx.x; j < D; j += NT) {
        pw[j] = 0.f;
        if constexpr (LN) pb[j] = 0.f;
    }
    for (int64_t row = ra; row < rb; row++) {
        const T* xr = x + row * ldx;
        const T* gr = dy + row * lddy;
        Mean m{0.f, 0.f};
        if constexpr (LN) {
            Acc2 s[1] = {acc2_zero()};
            for (int64_t j = threadIdx.x; j < D; j += NT) s_add<true>(s[0], E::load1(xr + j));
            group_reduce<NT, NT, 1, true>(s, red.take());
            m = mean_of(s[0], fd, inv_d);
        }
        Acc2 sums[K];
#pragma unroll
        for (int q = 0; q < K; q++) sums[q] = acc2_zero();
        for (int64_t j = threadIdx.x; j < D; j += NT) {
            const float d = (E::load1(xr + j) - m.mu0) - m.c;
            const float gg = E::load1(gr + j) * __ldg(w + j);
            s_fma<C>(sums[0], d, d);
            s_fma<C>(sums[1], gg, d);
            if constexpr (LN) s_add<C>(sums[2], gg);
        }
        group_reduce<NT, NT, K, C>(sums, red.take());
        const BwdStats st = bwd_stats<LN, C>(sums, inv_d, eps);
        for (int64_t j = threadIdx.x; j < D; j += NT) {
            const float g0 = E::load1(gr + j);
            const float xh = ((E::load1(xr + j) - m.mu0) - m.c) * st.r;
            E::store1(dx + row * lddx + j,
                      st.r * ((g0 * __ldg(w + j) - st.mg) - xh * st.mgx));
            pw[j] = fmaf(g0, xh, pw[j]);
            if constexpr (LN) pb[j] += g0;
        }
    }
    pdl_trigger();
}

// Stage 2: out[d] (+)= Σ_p part[o][p][d] for o = 0 (dw) and, for LayerNorm,
// o = 1 (db); blockIdx.y picks o.  Stripes of p are summed in order, then a
// fixed halving tree runs over the RY stripes.
template <int RY>
__global__ void __launch_bounds__(32 * RY)
    norm_bwd_reduce(const float* __restrict__ part, int64_t P, int64_t D, float* __restrict__ gw,
                    float* __restrict__ gb, int accumulate) {
    __shared__ float sm[RY][33];
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int64_t col = (int64_t)blockIdx.x * 32 + tx;
    float* out = blockIdx.y == 0 ? gw : gb;
    const float* pp = part + (int64_t)blockIdx.y * P * D;
    pdl_wait();
    float s = 0.f;
    if (col < D) {
#pragma unroll 8
        for (int64_t p = ty; p < P; p += RY) s += pp[p * D + col];
    }
    sm[ty][tx] = s;
    __syncthreads();
#pragma unroll
    for (int h = RY / 2; h > 0; h >>= 1) {
        if (ty < h) sm[ty][tx] += sm[ty + h][tx];
        __syncthreads();
    }
    if (ty == 0 && col < D) {
        const float v = sm[0][tx];
        out[col] = accumulate ? out[col] + v : v;
    }
    pdl_trigger();
}

// ===========================================================================
// Host launchers
// ===========================================================================
static inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
static inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

static cudaError_t allow_smem_norm(const void* kernel, size_t bytes) {
    if (bytes < 32 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// Row shape for Dv 16-byte chunks per row: each thread owns CPT chunks (16
// elements); TPR = the power of two >= ceil(Dv / CPT) threads per row; 256
// threads per CTA (R = 256/TPR rows at a time), or 512 for one row of
// 4097..8192 elements.
template <int CPT, typename F>
static cudaError_t norm_shape(int64_t Dv, F&& go) {
    using std::integral_constant;
    auto pick = [&](auto tpr) -> cudaError_t {
        constexpr int TPR = decltype(tpr)::value;
        constexpr int NT = TPR > 256 ? TPR : 256;
        return go(integral_constant<int, TPR>{}, integral_constant<int, CPT>{},
                  integral_constant<int, NT>{});
    };
    const int64_t t = cdiv(Dv, CPT);
    if (t <= 1) return pick(integral_constant<int, 1>{});
    if (t <= 2) return pick(integral_constant<int, 2>{});
    if (t <= 4) return pick(integral_constant<int, 4>{});
    if (t <= 8) return pick(integral_constant<int, 8>{});
    if (t <= 16) return pick(integral_constant<int, 16>{});
    if (t <= 32) return pick(integral_constant<int, 32>{});
    if (t <= 64) return pick(integral_constant<int, 64>{});
    if (t <= 128) return pick(integral_constant<int, 128>{});
    if (t <= 256) return pick(integral_constant<int, 256>{});
    return pick(integral_constant<int, 512>{});
}

// Cluster launches with CTAs of NT threads (16 elements a thread);
// cudaErrorNotSupported when no cluster of that shape fits.
template <typename T, bool LN, int NT>
static cudaError_t norm_fwd_cluster_go(const T* x, int64_t ldx, const float* w, const float* b,
                                       float eps, T* y, int64_t ldy, int64_t N, int64_t Dv,
                                       cudaStream_t s) {
    constexpr int V = Elt<T>::V, S = kNormFwdStages[LN], CPT = 16 / V;
    constexpr auto k = norm_fwd_cluster<T, LN, NT, S>;
    const unsigned cs = (unsigned)cdiv(Dv, (int64_t)NT * CPT);
    const size_t smem = (size_t)S * CPT * NT * 16;
    if (cs > (unsigned)kNormMaxCS<NT>) return cudaErrorNotSupported;
    int fit = 0;
    const cudaError_t e = cluster_fit<k>(cs, NT, smem, fit);
    if (e != cudaSuccess) return e;
    return launch_cluster(k, (unsigned)std::min<int64_t>(N, fit), cs, dim3(NT), smem, s, x, ldx, w,
                          b, eps, y, ldy, N, (int)Dv);
}

template <typename T, bool LN, int NT>
static cudaError_t norm_bwd_cluster_go(const T* x, int64_t ldx, const float* w, const T* dy,
                                       int64_t lddy, float eps, T* dx, int64_t lddx, float* part,
                                       int64_t N, int64_t Dv, int64_t P, cudaStream_t s) {
    constexpr int V = Elt<T>::V, CPT = 16 / V;
    constexpr int S = V == 4 ? kNormBwdStages32[LN] : kNormBwdStages16[LN];
    constexpr bool WS = kNormBwdWSlots[LN];
    constexpr auto k = norm_bwd_cluster<T, LN, NT, S, WS>;
    const unsigned cs = (unsigned)cdiv(Dv, (int64_t)NT * CPT);
    // staged x and dy, then (WS) this thread's w slots
    const size_t smem = (size_t)2 * S * CPT * NT * 16 + (WS ? (size_t)CPT * V * NT * 4 : 0);
    if (cs > (unsigned)kNormMaxCS<NT>) return cudaErrorNotSupported;
    int fit = 0;
    const cudaError_t e = cluster_fit<k>(cs, NT, smem, fit);
    if (e != cudaSuccess) return e;
    return launch_cluster(k, (unsigned)std::min<int64_t>(P, fit), cs, dim3(NT), smem, s, x, ldx, w,
                          dy, lddy, eps, dx, lddx, part, N, (int)Dv, P);
}

template <typename T, bool LN>
static cudaError_t norm_fwd_t(const T* x, int64_t ldx, const float* w, const float* b, float eps,
                              T* y, int64_t ldy, int64_t N, int64_t D, cudaStream_t s) {
    constexpr int V = Elt<T>::V;
    const int64_t Dv = D / V;
    if (D % V == 0 && D <= kNormRowMax && ldx % V == 0 && ldy % V == 0 && aligned16(x) &&
        aligned16(y) && aligned16(w) && (!LN || aligned16(b))) {
        return norm_shape<16 / V>(Dv, [&](auto tpr, auto cpt, auto nt) {
            constexpr int TPR = decltype(tpr)::value, CPT = decltype(cpt)::value;
            constexpr int NT = decltype(nt)::value;
            constexpr int S = 3;
            auto k = norm_fwd_rows<T, LN, TPR, CPT, NT, S, NT == 256 ? 3 : 1>;
            const size_t smem = (size_t)S * CPT * NT * 16;
            cudaError_t e = allow_smem_norm((const void*)k, smem);
            if (e != cudaSuccess) return e;
            const int64_t grid = std::min<int64_t>(cdiv(N, NT / TPR), 8 * kDesignSMs);
            return launch(k, dim3((unsigned)grid), dim3(NT), smem, s, true, x, ldx, w, b, eps, y,
                          ldy, N, (int)Dv);
        });
    }
    if (D % V == 0 && D <= kNormClusterRowMax && ldx % V == 0 && ldy % V == 0 && aligned16(x) &&
        aligned16(y) && aligned16(w) && (!LN || aligned16(b))) {
        const cudaError_t e = D <= kNormClusterSmallMaxD
                                  ? norm_fwd_cluster_go<T, LN, 128>(x, ldx, w, b, eps, y, ldy, N, Dv, s)
                                  : norm_fwd_cluster_go<T, LN, kNormClusterNT>(x, ldx, w, b, eps, y,
                                                                               ldy, N, Dv, s);
        if (e != cudaErrorNotSupported) return e;
    }
    return launch(norm_fwd_scalar<T, LN, 256>,
                  dim3((unsigned)std::min<int64_t>(N, 8 * kDesignSMs)), dim3(256), 0, s, true, x,
                  ldx, w, b, eps, y, ldy, N, D);
}

template <typename T, bool LN>
static cudaError_t norm_bwd_t(const T* x, int64_t ldx, const float* w, const T* dy, int64_t lddy,
                              float eps, T* dx, int64_t lddx, float* gw, float* gb, int accumulate,
                              float* part, int64_t N, int64_t D, cudaStream_t s) {
    constexpr int V = Elt<T>::V;
    const int64_t P = norm_tiles(N, D);
    const int64_t Dv = D / V;
    cudaError_t e = cudaSuccess;
    if (P > 0) {
        if (D % V == 0 && D <= kNormRowMax && ldx % V == 0 && lddy % V == 0 && lddx % V == 0 &&
            aligned16(x) && aligned16(dy) && aligned16(dx) && aligned16(w)) {
            e = norm_shape<16 / V>(Dv, [&](auto tpr, auto cpt, auto nt) {
                constexpr int TPR = decltype(tpr)::value, CPT = decltype(cpt)::value;
                constexpr int NT = decltype(nt)::value;
                constexpr int S = (NT > 256 && V == 4) ? 2 : 3;
                // LayerNorm: the lean layout at 3 CTAs per SM (80 registers)
                // measured 3.5% faster at bf16 65,536 x 4096; RMSNorm, with
                // one reduction per row, 7% slower — it keeps w and dy in
                // registers at 2 CTAs per SM
                constexpr bool LEAN = LN;
                auto k = norm_bwd_rows<T, LN, TPR, CPT, NT, S,
                                       NT == 256 ? (LEAN ? 3 : 2) : 1, LEAN>;
                // staging (x, dy), then (LEAN) this thread's w slots; the
                // epilogue reuses the start for the row groups' partials
                const size_t smem = std::max<size_t>(
                    (size_t)2 * S * CPT * NT * 16 + (LEAN ? (size_t)CPT * V * NT * 4 : 0),
                    (size_t)NT * CPT * V * sizeof(float));
                cudaError_t e2 = allow_smem_norm((const void*)k, smem);
                if (e2 != cudaSuccess) return e2;
                return launch(k, dim3((unsigned)P), dim3(NT), smem, s, true, x, ldx, w, dy, lddy,
                              eps, dx, lddx, part, N, (int)Dv, P);
            });
        } else {
            e = cudaErrorNotSupported;
            if (D % V == 0 && D <= kNormClusterRowMax && ldx % V == 0 && lddy % V == 0 &&
                lddx % V == 0 && aligned16(x) && aligned16(dy) && aligned16(dx) && aligned16(w)) {
                e = D <= kNormClusterSmallMaxD
                        ? norm_bwd_cluster_go<T, LN, 128>(x, ldx, w, dy, lddy, eps, dx, lddx, part,
                                                          N, Dv, P, s)
                        : norm_bwd_cluster_go<T, LN, kNormClusterNT>(x, ldx, w, dy, lddy, eps, dx,
                                                                     lddx, part, N, Dv, P, s);
            }
            if (e == cudaErrorNotSupported)
                e = launch(norm_bwd_scalar<T, LN, 256>, dim3((unsigned)P), dim3(256), 0, s, true,
                           x, ldx, w, dy, lddy, eps, dx, lddx, part, N, D, P);
        }
        if (e != cudaSuccess) return e;
    }
    const unsigned nout = LN ? 2 : 1;
    if (D <= 4096)
        return launch(norm_bwd_reduce<32>, dim3((unsigned)cdiv(D, 32), nout), dim3(32, 32), 0, s,
                      true, (const float*)part, P, D, gw, gb, accumulate);
    return launch(norm_bwd_reduce<8>, dim3((unsigned)cdiv(D, 32), nout), dim3(32, 8), 0, s, true,
                  (const float*)part, P, D, gw, gb, accumulate);
}

template <bool LN>
static cudaError_t norm_fwd_any(const void* x, int64_t ldx, const float* w, const float* b,
                                float eps, void* y, int64_t ldy, int64_t N, int64_t D, int dtype,
                                cudaStream_t s) {
    switch (dtype) {
        case 0:
            return norm_fwd_t<float, LN>((const float*)x, ldx, w, b, eps, (float*)y, ldy, N, D, s);
        case 1:
            return norm_fwd_t<__half, LN>((const __half*)x, ldx, w, b, eps, (__half*)y, ldy, N, D,
                                          s);
        default:
            return norm_fwd_t<__nv_bfloat16, LN>((const __nv_bfloat16*)x, ldx, w, b, eps,
                                                 (__nv_bfloat16*)y, ldy, N, D, s);
    }
}

template <bool LN>
static cudaError_t norm_bwd_any(const void* x, int64_t ldx, const float* w, const void* dy,
                                int64_t lddy, float eps, void* dx, int64_t lddx, float* gw,
                                float* gb, int accumulate, float* part, int64_t N, int64_t D,
                                int dtype, cudaStream_t s) {
    switch (dtype) {
        case 0:
            return norm_bwd_t<float, LN>((const float*)x, ldx, w, (const float*)dy, lddy, eps,
                                         (float*)dx, lddx, gw, gb, accumulate, part, N, D, s);
        case 1:
            return norm_bwd_t<__half, LN>((const __half*)x, ldx, w, (const __half*)dy, lddy, eps,
                                          (__half*)dx, lddx, gw, gb, accumulate, part, N, D, s);
        default:
            return norm_bwd_t<__nv_bfloat16, LN>((const __nv_bfloat16*)x, ldx, w,
                                                 (const __nv_bfloat16*)dy, lddy, eps,
                                                 (__nv_bfloat16*)dx, lddx, gw, gb, accumulate,
                                                 part, N, D, s);
    }
}

cudaError_t norm_wait_timeouts(unsigned* count, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(count, g_norm_wait_timeouts, sizeof(unsigned));
    if (e == cudaSuccess && reset) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_norm_wait_timeouts, &zero, sizeof(unsigned));
    }
    return e;
}

cudaError_t launch_norm_fwd(const void* x, int64_t ldx, const float* w, const float* b, float eps,
                            void* y, int64_t ldy, int64_t N, int64_t D, int dtype, int layer,
                            cudaStream_t s) {
    return layer ? norm_fwd_any<true>(x, ldx, w, b, eps, y, ldy, N, D, dtype, s)
                 : norm_fwd_any<false>(x, ldx, w, b, eps, y, ldy, N, D, dtype, s);
}

cudaError_t launch_norm_bwd(const void* x, int64_t ldx, const float* w, const void* dy,
                            int64_t lddy, float eps, void* dx, int64_t lddx, float* gw, float* gb,
                            int accumulate, float* part, int64_t N, int64_t D, int dtype,
                            int layer, cudaStream_t s) {
    return layer ? norm_bwd_any<true>(x, ldx, w, dy, lddy, eps, dx, lddx, gw, gb, accumulate, part,
                                      N, D, dtype, s)
                 : norm_bwd_any<false>(x, ldx, w, dy, lddy, eps, dx, lddx, gw, gb, accumulate,
                                       part, N, D, dtype, s);
}

}  // namespace wsf
