// selftest.cu — a check of the bounded waits of the cluster exchange.
//
// The cluster paths (softmax rows over 2048 chunks, RMSNorm / LayerNorm rows
// of 8193..65536 elements) wait on an mbarrier for the partial sums that the
// other CTAs of their cluster push (WarpPush).  Every such wait gives up after
// a time limit and counts the timeout instead of hanging the GPU.  This entry
// point runs that wait where nothing ever completes it: one cluster of two
// CTAs posts the bytes a turn expects and waits, but no CTA pushes.  Each
// waiting warp counts one timeout, the kernel returns, and the context stays
// usable.  Nothing is pushed, so no data is in flight when the waits give up.
#include "wsf_device.cuh"
#include "wsf_internal.h"

namespace wsf {

constexpr int kSelftestNT = 64;
constexpr unsigned kSelftestCS = 2;

__global__ void __launch_bounds__(kSelftestNT)
    exchange_timeout_kernel(unsigned* __restrict__ count, uint64_t limit_ns) {
    constexpr int W = kSelftestNT / 32;
    __shared__ __align__(16) float4 xbuf[2][kClusterMaxCS * W][1];
    __shared__ __align__(8) uint64_t xbar[2];
    WarpPush<W, kClusterMaxCS * W, 1> xp{xbuf, xbar, count, 0u, true, limit_ns};
    xp.init();
    cluster_sync();
    pdl_wait();
    // turn 0 as the cluster paths post it, without any push
    if (threadIdx.x == 0) mbar_expect_tx(&xbar[0], cluster_nctarank() * W * 16u);
    (void)xp.wait(0);
    cluster_sync();
    pdl_trigger();
}

int selftest_waiting_warps() { return (int)kSelftestCS * (kSelftestNT / 32); }

cudaError_t launch_exchange_timeout(unsigned* count, uint64_t limit_ns, cudaStream_t s) {
    return launch_cluster(exchange_timeout_kernel, 1, kSelftestCS, dim3(kSelftestNT), 0, s, count,
                          limit_ns);
}

}  // namespace wsf
