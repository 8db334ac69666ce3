// wsf_internal.h — host-side interface between the C ABI (abi.cu) and the
// kernel launchers (ws.cu, silu.cu, softmax.cu, norm.cu).  Not installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

namespace wsf {

// Bytes per element of a storage type (0 for an invalid code).
inline int elt_bytes(int dtype) { return dtype == 0 ? 4 : (dtype == 1 || dtype == 2) ? 2 : 0; }

// Number of row tiles P of the weighted-sum backward (rows of the partial
// buffer).  Depends only on the sizes, the storage type and block_n.
int64_t ws_tiles(int64_t N, int64_t D, int dtype, int64_t block_n);

// Number of per-block partials of the scaled-SiLU backward.
int64_t silu_tiles(int64_t n);

// The partial sums of a parameter gradient are compensated pairs: the
// workspace holds a plane of high parts [P, D] and, `gradient_plane(P, D)`
// floats further on (a 256-byte multiple), a plane of low parts.
inline int64_t gradient_plane(int64_t P, int64_t D) { return (P * D + 63) / 64 * 64; }

cudaError_t launch_ws_fwd(const void* x, int64_t ldx, const float* w, void* y, int64_t N,
                          int64_t D, int dtype, cudaStream_t s);

// Host-side validation of ws_bwd's arguments (abi.cu); check_ws = false
// leaves out the workspace (ws_bwd_noalloc).  Returns a WSF_* status and sets
// *need to the workspace bytes the sizes require.
int ws_bwd_check(const void* x, int64_t ldx, const float* w, const void* dy, void* dx,
                 int64_t lddx, float* grad_w, int accumulate, const void* workspace,
                 size_t workspace_bytes, bool check_ws, int64_t block_n, int64_t N, int64_t D,
                 int dtype, size_t* need);

cudaError_t launch_ws_bwd(const void* x, int64_t ldx, const float* w, const void* dy, void* dx,
                          int64_t lddx, float* grad_w, int accumulate, float* partial,
                          int64_t block_n, int64_t N, int64_t D, int dtype, cudaStream_t s);

// Atomic comparison variants (grad_w / dw summed with atomic additions).
bool ws_bwd_atomic_supported(const void* x, int64_t ldx, const float* w, const void* dy,
                             const void* dx, int64_t lddx, const float* grad_w, int64_t D,
                             int dtype);
cudaError_t launch_ws_bwd_atomic(const void* x, int64_t ldx, const float* w, const void* dy,
                                 void* dx, int64_t lddx, float* grad_w, int accumulate, int64_t N,
                                 int64_t D, int dtype, cudaStream_t s);
cudaError_t launch_silu_bwd_atomic(const void* dy, const void* x, const float* w, void* dx,
                                   float* dw, int accumulate, int64_t n, int dtype, cudaStream_t s);

cudaError_t launch_softmax_fwd(const void* x, int64_t ldx, void* y, int64_t ldy, int64_t N,
                               int64_t D, int dtype, cudaStream_t s);
cudaError_t launch_softmax_bwd(const void* y, int64_t ldy, const void* dy, int64_t lddy, void* dx,
                               int64_t lddx, int64_t N, int64_t D, int dtype, cudaStream_t s);

// RMSNorm (layer == 0) / LayerNorm (layer == 1) rows; norm_tiles is the
// number of row tiles P of the backward's partial buffer ([P, D] per
// parameter gradient).
int64_t norm_tiles(int64_t N, int64_t D);
cudaError_t launch_norm_fwd(const void* x, int64_t ldx, const float* w, const float* b, float eps,
                            void* y, int64_t ldy, int64_t N, int64_t D, int dtype, int layer,
                            cudaStream_t s);
cudaError_t launch_norm_bwd(const void* x, int64_t ldx, const float* w, const void* dy,
                            int64_t lddy, float eps, void* dx, int64_t lddx, float* gw, float* gb,
                            int accumulate, float* part, int64_t N, int64_t D, int dtype,
                            int layer, cudaStream_t s);

// Read (and optionally zero) the count of cluster-exchange waits that ran
// out in the norm (softmax) kernels on the current device; synchronises the
// device.
cudaError_t norm_wait_timeouts(unsigned* count, bool reset);
cudaError_t softmax_wait_timeouts(unsigned* count, bool reset);

// One cluster whose exchange wait nothing completes (selftest.cu): each
// waiting warp adds one to *count (device memory) after limit_ns.
cudaError_t launch_exchange_timeout(unsigned* count, uint64_t limit_ns, cudaStream_t s);
int selftest_waiting_warps();

cudaError_t launch_silu_fwd(const void* x, const float* w, void* y, int64_t n, int dtype,
                            cudaStream_t s);

cudaError_t launch_silu_bwd(const void* dy, const void* x, const float* w, void* dx, float* dw,
                            int accumulate, float* part, int64_t n, int dtype, cudaStream_t s);

// Launch through cudaLaunchKernelEx so that the status returned is this
// launch's own.  `pdl` lets the kernel start while the previous kernel on
// the stream drains; every kernel of the library begins with
// griddepcontrol.wait, so nothing it reads or writes is touched before the
// previous kernel has finished.
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                   bool pdl, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Launch `clusters` thread-block clusters of `cs` CTAs each (grid = clusters x
// cs CTAs along x), with programmatic dependent launch as above.
template <typename... KArgs, typename... Args>
cudaError_t launch_cluster(void (*kernel)(KArgs...), unsigned clusters, unsigned cs, dim3 block,
                           size_t smem, cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(clusters * cs);
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cs;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// How many clusters of `cs` CTAs of `kernel` (block threads, smem dynamic
// bytes) the current device holds at once; 0 if none fits or the query fails.
// Kernel attributes (shared-memory limit, non-portable cluster size) must be
// set before the query.
template <typename... KArgs>
int max_active_clusters(void (*kernel)(KArgs...), unsigned cs, dim3 block, size_t smem) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs);
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (const void*)kernel, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

// Clusters of `cs` CTAs of `kernel` resident at once on the current device,
// queried once per device, kernel and cluster size (the kernel's shape and
// shared memory are fixed for a given cs).  Sets the kernel's dynamic
// shared-memory limit and, for cs > 8, allows the non-portable cluster size.
// `fit` = 0 with cudaErrorNotSupported when no such cluster fits.
constexpr int kClusterMaxCS = 16;
constexpr int kMaxDevices = 64;

template <auto kernel>
cudaError_t cluster_fit(unsigned cs, int nt, size_t smem, int& fit) {
    static std::atomic<int> fits[kMaxDevices][kClusterMaxCS + 1];
    fit = 0;
    if (cs < 1 || cs > (unsigned)kClusterMaxCS) return cudaErrorNotSupported;
    cudaError_t e = cudaFuncSetAttribute((const void*)kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess && cs > 8)
        e = cudaFuncSetAttribute((const void*)kernel,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int f = dev < kMaxDevices ? fits[dev][cs].load(std::memory_order_relaxed) : 0;
    if (f == 0) {
        f = max_active_clusters(kernel, cs, dim3(nt), smem);
        if (f <= 0) f = -1;
        if (dev < kMaxDevices) fits[dev][cs].store(f, std::memory_order_relaxed);
    }
    if (f < 0) return cudaErrorNotSupported;
    fit = f;
    return cudaSuccess;
}

}  // namespace wsf
