// noalloc.cu — ws_bwd_noalloc: the weighted-sum backward for callers that
// cannot allocate device memory.
//
// Some callers are handed only their input and output buffers and have no
// way to obtain more device memory: a plugin inside a host program that owns
// every byte of device memory through its own pool, or a latency-critical
// loop in which cudaMalloc's implicit device-wide synchronisation is not
// acceptable.  ws_bwd needs a caller-provided workspace for its per-tile
// grad_w partials; this entry point instead uses a fixed scratch array that
// lives in the library's own device memory (file-scope, one copy per device
// that loads the library, held until the process exits).
//
// The call allocates nothing: no cudaMalloc, no cudaFree, no allocating
// library routine.  On the first call on a device it looks up that device's
// copy of the array with cudaGetSymbolAddress (the array's name in host code
// is only a host-side stand-in, not a device address); that first call on
// each device should therefore come before any stream capture.  Every call
// shares the one array, which keeps the last call's contents: the backward
// writes every partial it later reads, so nothing needs clearing, but calls
// whose kernels overlap on the GPU (e.g. on two streams) race on the array
// and must be serialised by the caller.
#include <mutex>

#include "wsf.h"
#include "wsf_internal.h"

namespace {

static __device__ __align__(256) float g_ws_scratch[WSF_NOALLOC_SCRATCH_BYTES / sizeof(float)];

constexpr int kMaxDevices = 128;
std::mutex g_mutex;
float* g_scratch_ptr[kMaxDevices] = {};

// Device address of the current device's copy of g_ws_scratch, looked up
// once per device with that device current.
int scratch_for_current_device(float** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return WSF_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_ws_scratch) != cudaSuccess || p == nullptr)
            return WSF_ERR_CUDA;
        g_scratch_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_ptr[dev];
    return WSF_OK;
}

}  // namespace

extern "C" int ws_bwd_noalloc(const void* x, int64_t ldx, const float* w, const void* dy,
                              void* dx, int64_t lddx, float* grad_w, int accumulate,
                              int64_t block_n, int64_t N, int64_t D, int dtype,
                              wsf_stream_t stream) {
    // the same argument checks, in the same order, as ws_bwd (less the
    // workspace); only then the scratch limit and the device lookup
    size_t need = 0;
    int rc = wsf::ws_bwd_check(x, ldx, w, dy, dx, lddx, grad_w, accumulate, nullptr, 0, false,
                               block_n, N, D, dtype, &need);
    if (rc != WSF_OK) return rc;
    if (need > WSF_NOALLOC_SCRATCH_BYTES) return WSF_ERR_WORKSPACE;
    if (D == 0) return WSF_OK;
    float* scratch = nullptr;
    if (need > 0) {
        rc = scratch_for_current_device(&scratch);
        if (rc != WSF_OK) return rc;
    }
    return wsf::launch_ws_bwd(x, ldx, w, dy, dx, lddx, grad_w, accumulate, scratch, block_n, N, D,
                              dtype, (cudaStream_t)stream) == cudaSuccess
               ? WSF_OK
               : WSF_ERR_CUDA;
}
