// wsf_device.cuh — device helpers shared by the libwsfwd kernels (sm_103a):
// 128-bit streaming loads/stores, widening of 16-bit storage types to fp32,
// round-to-nearest-even narrowing, warp reductions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace wsf {

constexpr unsigned FULL_MASK = 0xffffffffu;

// Number of SMs the launch shapes are designed for (GB300: 2 dies x 76).
// It fixes grid sizes and tile counts as constants so that the reduction
// order, and therefore every bit of grad_w / dw, never depends on the device.
constexpr int kDesignSMs = 152;

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of the library is launched so
// that it may be scheduled while the previous kernel on the stream drains;
// each one therefore calls pdl_wait() before its first global memory access
// (read or write), which blocks until the previous grid has completed and its
// writes are visible.  pdl_trigger() tells the hardware that this CTA's main
// work is done, so the next kernel may begin launching.  Both are no-ops when
// a kernel is launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// 16-byte vector of raw storage.
struct alignas(16) Raw16 {
    uint32_t u[4];
};

__device__ __forceinline__ Raw16 raw_zero() {
    Raw16 r;
    r.u[0] = r.u[1] = r.u[2] = r.u[3] = 0u;
    return r;
}

// Streaming read of 16 bytes that is used once: read-only path, no L1
// allocation, and a 256-byte L2 prefetch so DRAM serves whole bursts.
__device__ __forceinline__ Raw16 ld_stream(const void* p) {
    Raw16 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.u[0]), "=r"(r.u[1]), "=r"(r.u[2]), "=r"(r.u[3])
                 : "l"(p));
    return r;
}

// Read of 16 bytes expected to be reused from L1/L2 (weights).
__device__ __forceinline__ Raw16 ld_keep(const void* p) {
    Raw16 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.u[0]), "=r"(r.u[1]), "=r"(r.u[2]), "=r"(r.u[3])
                 : "l"(p));
    return r;
}

// Streaming write of 16 bytes (evict-first in L2).
__device__ __forceinline__ void st_stream(void* p, const Raw16& r) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(r.u[0]), "r"(r.u[1]),
                 "r"(r.u[2]), "r"(r.u[3])
                 : "memory");
}

// L2 cache policies: lines read under evict_last stay ahead of others, lines
// read under evict_first are the first to leave.
__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Read of 16 bytes (read-only path, no L1 allocation) under an L2 policy.
__device__ __forceinline__ Raw16 ld_policy(const void* p, uint64_t pol) {
    Raw16 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(r.u[0]), "=r"(r.u[1]), "=r"(r.u[2]), "=r"(r.u[3])
                 : "l"(p), "l"(pol));
    return r;
}

// Bulk prefetch of `bytes` (a multiple of 16) from global memory into L2,
// starting at a 16-byte aligned address, under an L2 policy; nothing waits
// for it.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes, uint64_t pol) {
    asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(p),
                 "r"(bytes), "l"(pol)
                 : "memory");
}

// Asynchronous 16-byte global -> shared copy (cp.async, bypassing L1, with a
// 256-byte L2 prefetch).  Only the first src_bytes (0..16) are read; the
// rest of the 16 shared bytes are zero-filled.  A thread waits for its own
// copies with cp_async_wait<N>() (at most N most recent groups pending); no
// other synchronisation is involved, so nothing here can wait forever.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem),
                 "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------
// Storage-type traits: V elements per 16 bytes, widening, narrowing.
template <typename T>
struct Elt;

template <>
struct Elt<float> {
    static constexpr int V = 4;
    __device__ __forceinline__ static void widen(const Raw16& r, float (&f)[4]) {
#pragma unroll
        for (int i = 0; i < 4; i++) f[i] = __uint_as_float(r.u[i]);
    }
    __device__ __forceinline__ static Raw16 narrow(const float (&f)[4]) {
        Raw16 r;
#pragma unroll
        for (int i = 0; i < 4; i++) r.u[i] = __float_as_uint(f[i]);
        return r;
    }
    __device__ __forceinline__ static float widen1(float v) { return v; }
    __device__ __forceinline__ static float load1(const float* p) { return __ldg(p); }
    __device__ __forceinline__ static void store1(float* p, float v) { *p = v; }
};

template <>
struct Elt<__half> {
    static constexpr int V = 8;
    __device__ __forceinline__ static void widen(const Raw16& r, float (&f)[8]) {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            __half2 h;
            memcpy(&h, &r.u[i], 4);
            const float2 v = __half22float2(h);
            f[2 * i] = v.x;
            f[2 * i + 1] = v.y;
        }
    }
    __device__ __forceinline__ static Raw16 narrow(const float (&f)[8]) {
        Raw16 r;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
            memcpy(&r.u[i], &h, 4);
        }
        return r;
    }
    __device__ __forceinline__ static float widen1(__half v) { return __half2float(v); }
    __device__ __forceinline__ static float load1(const __half* p) { return __half2float(__ldg(p)); }
    __device__ __forceinline__ static void store1(__half* p, float v) { *p = __float2half_rn(v); }
};

template <>
struct Elt<__nv_bfloat16> {
    static constexpr int V = 8;
    __device__ __forceinline__ static void widen(const Raw16& r, float (&f)[8]) {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            // bfloat16 is the upper half of a binary32 pattern: widening is a shift.
            f[2 * i] = __uint_as_float(r.u[i] << 16);
            f[2 * i + 1] = __uint_as_float(r.u[i] & 0xffff0000u);
        }
    }
    __device__ __forceinline__ static Raw16 narrow(const float (&f)[8]) {
        Raw16 r;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            memcpy(&r.u[i], &h, 4);
        }
        return r;
    }
    __device__ __forceinline__ static float widen1(__nv_bfloat16 v) { return __bfloat162float(v); }
    __device__ __forceinline__ static float load1(const __nv_bfloat16* p) {
        return __bfloat162float(__ldg(p));
    }
    __device__ __forceinline__ static void store1(__nv_bfloat16* p, float v) {
        *p = __float2bfloat16_rn(v);
    }
};

// ---------------------------------------------------------------------------
// Sum over the lanes of aligned groups of `Width` lanes (xor butterfly); every
// lane of a group ends with the group's sum.  The operand order is fixed, so
// the result is the same bits on every run.
template <int Width>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int off = Width / 2; off > 0; off >>= 1) v += __shfl_xor_sync(FULL_MASK, v, off);
    return v;
}

// ---------------------------------------------------------------------------
// Compensated fp32 dot-product accumulation (the "Dot2" scheme of Ogita,
// Rump and Oishi, "Accurate sum and dot product", SIAM J. Sci. Comput. 26,
// 2005): each product is split exactly into p + ep with an FMA, each addition
// into its rounded sum and exact error (Knuth's TwoSum); the errors are
// collected in `lo`.  The result hi + lo is as accurate as if computed in
// twice the working precision, then rounded.  Used where a binary32 output
// must stay within 1e-6 of the exact sum over up to 65,536 terms, and for
// every parameter-gradient sum (grad_w, dw), whose stated bound is 1e-5 of
// the exact value even where the sum cancels to a small fraction of its
// terms' magnitudes.
struct Acc2 {
    float hi, lo;
};

__device__ __forceinline__ Acc2 acc2_zero() { return Acc2{0.f, 0.f}; }

// The _rn intrinsics are never contracted into fused multiply-adds, which
// would break the exactness of the splits.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bp = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

__device__ __forceinline__ void acc2_fma(Acc2& a, float x, float w) {
    const float p = __fmul_rn(x, w);
    const float ep = fmaf(x, w, -p);
    float s, e;
    two_sum(a.hi, p, s, e);
    a.hi = s;
    a.lo += e + ep;
}

__device__ __forceinline__ Acc2 acc2_add(Acc2 a, Acc2 b) {
    float s, e;
    two_sum(a.hi, b.hi, s, e);
    return Acc2{s, a.lo + b.lo + e};
}

// Add one binary32 value whose own rounding is not in question (an exact
// product, or a term taken as given): TwoSum into hi, the error into lo.
__device__ __forceinline__ void acc2_add1(Acc2& a, float p) {
    float s, e;
    two_sum(a.hi, p, s, e);
    a.hi = s;
    a.lo += e;
}

// Compensated accumulation of the product x·g.  The product of two values of
// a 16-bit storage type is exact in binary32 (at most 11 + 11 significant
// bits, within the exponent range unless it falls below 2^-126), so only the
// addition needs its error kept; a binary32 product is split with an FMA.
template <bool ExactProduct>
__device__ __forceinline__ void acc2_prod(Acc2& a, float x, float g) {
    if constexpr (ExactProduct)
        acc2_add1(a, __fmul_rn(x, g));
    else
        acc2_fma(a, x, g);
}

// Value of a compensated pair, rounded once to binary32.
__device__ __forceinline__ float acc2_value(Acc2 a) { return __fadd_rn(a.hi, a.lo); }

// ---------------------------------------------------------------------------
// Packed binary32 pairs (sm_100 and later: add/sub/mul/fma.rn.f32x2 operate
// on two binary32 values held in one 64-bit register, each lane rounded to
// nearest-even on its own, exactly as the scalar instruction would).  Lane 0
// is the low half.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(a), "f"(b));
    return d;
}
__device__ __forceinline__ void f2_unpack(uint64_t d, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(d));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// Two compensated pairs, packed: hi holds the two running sums, lo their
// collected rounding errors.
struct Acc2x2 {
    uint64_t hi, lo;
};

// acc2_prod on two columns at once: a += x·g lane by lane (x2 the two
// values of x, g2 = (g, g), ng2 = (−g, −g)).  The steps are Knuth's TwoSum
// written with b − b' as fma(x, g, −b') where the product is exact (and with
// an FMA split of the product where it is not), so every lane gets the bits
// that acc2_prod gives.
template <bool ExactProduct>
__device__ __forceinline__ void acc2x2_prod(Acc2x2& a, uint64_t x2, uint64_t g2, uint64_t ng2) {
    if constexpr (ExactProduct) {
        const uint64_t s = f2_fma(x2, g2, a.hi);    // fl(hi + x·g)
        const uint64_t nbp = f2_sub(a.hi, s);       // −(s − hi)
        const uint64_t ap = f2_add(s, nbp);         // s − (s − hi)
        const uint64_t e = f2_add(f2_sub(a.hi, ap), f2_fma(x2, g2, nbp));
        a.hi = s;
        a.lo = f2_add(a.lo, e);
    } else {
        const uint64_t np = f2_mul(x2, ng2);        // −fl(x·g)
        const uint64_t ep = f2_fma(x2, g2, np);     // x·g − fl(x·g), exact
        const uint64_t s = f2_sub(a.hi, np);        // fl(hi + p)
        const uint64_t nbp = f2_sub(a.hi, s);
        const uint64_t ap = f2_add(s, nbp);
        const uint64_t e = f2_add(f2_sub(a.hi, ap), f2_sub(nbp, np));
        a.hi = s;
        a.lo = f2_add(a.lo, f2_add(e, ep));
    }
}

__device__ __forceinline__ void acc2x2_unpack(const Acc2x2& a, Acc2& first, Acc2& second) {
    f2_unpack(a.hi, first.hi, second.hi);
    f2_unpack(a.lo, first.lo, second.lo);
}

template <int Width>
__device__ __forceinline__ Acc2 group_sum2(Acc2 v) {
#pragma unroll
    for (int off = Width / 2; off > 0; off >>= 1) {
        Acc2 o{__shfl_xor_sync(FULL_MASK, v.hi, off), __shfl_xor_sync(FULL_MASK, v.lo, off)};
        v = acc2_add(v, o);
    }
    return v;
}

// Pick a[i] for a runtime i without dynamic register indexing.
template <int K>
__device__ __forceinline__ float select(const float (&a)[K], int i) {
    float v = a[0];
#pragma unroll
    for (int k = 1; k < K; k++) v = (i == k) ? a[k] : v;
    return v;
}

// ---------------------------------------------------------------------------
// Thread-block clusters (sm_90 and later).  A cluster's CTAs are scheduled
// together and can reach one another's shared memory ("distributed shared
// memory"): mapa turns a local shared-memory address into the address of the
// same variable in the CTA of a given rank (the target of st.async below).
// cluster_sync() is the hardware cluster barrier (every thread of every CTA
// of the cluster arrives; .release/.acquire make shared-memory writes made
// before the arrival visible to reads made after the wait).  It is not a
// spin loop: like __syncthreads() it completes once every thread has
// arrived, so each CTA of a cluster must execute the same number of them.
__device__ __forceinline__ unsigned cluster_ctarank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ unsigned cluster_nctarank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ unsigned cluster_id_x() {
    unsigned r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ unsigned cluster_count_x() {
    unsigned r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
}
// Address of the shared variable at local address `p` in the CTA of rank `r`.
__device__ __forceinline__ uint32_t cluster_map(const void* p, unsigned r) {
    uint32_t out;
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(a), "r"(r));
    return out;
}
// ---------------------------------------------------------------------------
// mbarrier-completed pushes into another CTA's shared memory (sm_90 and
// later).  st.async writes a value into the shared memory of a CTA of the
// cluster and counts its bytes against that CTA's mbarrier; the receiver
// posts how many bytes it expects (arrive.expect_tx) and waits on the
// barrier's phase, after which the pushed data is visible to it.
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;"
                 :: "r"((uint32_t)__cvta_generic_to_shared(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\t"
                 "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
                 :: "r"((uint32_t)__cvta_generic_to_shared(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done) : "r"((uint32_t)__cvta_generic_to_shared(bar)), "r"(parity)
                 : "memory");
    return done != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for the phase of `bar` with the given parity to complete, for at most
// about `limit_ns` nanoseconds; false if the limit ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > limit_ns) return false;
    return true;
}
// Push 16 bytes to the cluster shared address `dst`, completing `bar` (the
// cluster shared address of the receiving CTA's mbarrier).
__device__ __forceinline__ void st_async_f32x4(uint32_t dst, float4 v, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
                 :: "r"(dst), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar) : "memory");
}

// One entry a warp (NV float4, the same in every lane) exchanged among the
// CTAs of a cluster: lane q of each warp pushes the warp's entry into slot
// rank·W + warp of CTA q; a CTA's turn is complete when the entries of all
// cs·W warps of the cluster have arrived in its own buffer.  Turns cycle
// through NB buffers, each with its own mbarrier (phase parity = turn/NB).
// Thread 0 posts the bytes expected (pushes that land before it leave the
// phase pending); the threads that wait (wait()) may then read the turn's
// buffer.  A buffer is written again NB turns later, which no CTA can reach
// before every CTA has finished reading it, provided that a warp pushes turn
// t + NB − 1 only after this CTA's readers of turn t are done (the callers
// put a CTA barrier between them: NB = 2 when a CTA pushes turn t + 1 after
// reading turn t, NB = 4 when it pushes turn t + 1 before reading turn t)
// and that every turn is waited for by thread 0.  A wait longer than
// limit_ns (a second unless set) marks the exchange dead for the waiting
// thread (later waits are skipped) and counts a timeout (one a warp), so
// that a fault in the protocol ends the kernel with wrong results and a
// raised counter instead of a hang.  Each CTA of a cluster must run the same
// turns, and every CTA's barriers must be initialised (init(), then a
// cluster barrier) before the first push.
template <int W, int SLOTS, int NV, int NB = 2>
struct WarpPush {
    float4 (*buf)[SLOTS][NV];  // shared [NB][SLOTS][NV]
    uint64_t* bar;             // shared [NB]
    unsigned* timeouts;        // device counter of waits that ran out
    unsigned turn;
    bool live;
    uint64_t limit_ns = 1000000000ull;  // how long a wait may take

    __device__ __forceinline__ void init() {
        if (threadIdx.x == 0) {
#pragma unroll
            for (int i = 0; i < NB; i++) mbar_init(&bar[i], 1);
            mbar_init_fence();
        }
    }

    // Push `e` (the first NX float4 of an entry); returns the turn's number.
    template <int NX>
    __device__ __forceinline__ unsigned push(const float4 (&e)[NX]) {
        static_assert(NX >= 1 && NX <= NV, "entry size");
        const unsigned t = turn++, p = t % NB;
        const unsigned cs = cluster_nctarank(), me = cluster_ctarank();
        const unsigned lane = threadIdx.x & 31u, wid = threadIdx.x >> 5;
        if (threadIdx.x == 0) mbar_expect_tx(&bar[p], cs * W * NX * 16u);
        if (lane < cs) {
            const uint32_t dst = cluster_map(&buf[p][me * W + wid][0], lane);
            const uint32_t rb = cluster_map(&bar[p], lane);
#pragma unroll
            for (int q = 0; q < NX; q++) st_async_f32x4(dst + 16u * q, e[q], rb);
        }
        return t;
    }

    // Wait until turn t is complete; returns its buffer.
    __device__ __forceinline__ const float4 (*wait(unsigned t))[NV] {
        if (live && !mbar_wait(&bar[t % NB], (t / NB) & 1u, limit_ns)) {
            live = false;
            if ((threadIdx.x & 31u) == 0) atomicAdd(timeouts, 1u);
        }
        return buf[t % NB];
    }
};

}  // namespace wsf
