// Status strings, per-thread CUDA error record and cached device facts.
#include <atomic>
#include <cstdlib>

#include "common.cuh"

namespace gact {
namespace {

thread_local int g_last_cuda_error = 0;

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];   // 0 = not queried yet

}  // namespace

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0)
        return 1;
    if (dev < kMaxDevices) {
        const int cached = g_sm_count[dev].load(std::memory_order_relaxed);
        if (cached > 0)
            return cached;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 1;
    if (dev < kMaxDevices)
        g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

bool pdl_enabled() {
    static const bool on = [] {
        const char *v = std::getenv("GATED_ACT_PDL");
        return !(v && v[0] == '0' && v[1] == '\0');
    }();
    return on;
}

int resolve_ptr(const void *p, const void **dev, bool *host) {
    *dev = p;
    *host = false;
    if (!p)
        return GATED_ACT_OK;
    cudaPointerAttributes a;
    const cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) {
        cudaGetLastError();   // not sticky, but keep the error state clean
        return GATED_ACT_ERR_HOST;
    }
    switch (a.type) {
    case cudaMemoryTypeDevice: {
        // kernels run on the current device: another GPU's memory would be
        // reached over a peer mapping, if one exists at all
        int cur = -1;
        if (cudaGetDevice(&cur) != cudaSuccess || a.device != cur)
            return GATED_ACT_ERR_DEVICE;
        return GATED_ACT_OK;
    }
    case cudaMemoryTypeManaged:
        return GATED_ACT_OK;
    case cudaMemoryTypeHost:
        if (!a.devicePointer)
            return GATED_ACT_ERR_HOST;
        *dev = a.devicePointer;
        *host = true;
        return GATED_ACT_OK;
    default:   // not registered with CUDA: pageable host memory, or no allocation at all
        return GATED_ACT_ERR_HOST;
    }
}

int cuda_status(cudaError_t e) {
    if (e == cudaSuccess)
        return GATED_ACT_OK;
    g_last_cuda_error = static_cast<int>(e);
    return GATED_ACT_ERR_CUDA;
}

// Empty kernel with the library's launch attributes (launch-overhead probe).
__global__ void noop_kernel() {
    pdl_wait();
    pdl_trigger();
}

}  // namespace gact

extern "C" int gated_act_noop(cudaStream_t stream) {
    const cudaError_t e = gact::launch_kernel(gact::noop_kernel, dim3(1), dim3(32), 0, stream, 1);
    if (e != cudaSuccess)
        return gact::cuda_status(e);
    return gact::cuda_status(cudaGetLastError());
}

extern "C" const char *gated_act_status_string(int status) {
    switch (status) {
    case GATED_ACT_OK: return "ok";
    case GATED_ACT_ERR_NULL: return "null input or output pointer";
    case GATED_ACT_ERR_SIZE: return "bad size: rows must be >= 0 and d >= 1";
    case GATED_ACT_ERR_STRIDE: return "row_stride is smaller than 2*d";
    case GATED_ACT_ERR_TOO_LARGE: return "problem too large for the index arithmetic";
    case GATED_ACT_ERR_OVERLAP: return "output overlaps the input";
    case GATED_ACT_ERR_VARIANT: return "requested launch geometry does not fit this call";
    case GATED_ACT_ERR_CUDA: return "CUDA runtime error at launch (see gated_act_last_cuda_error)";
    case GATED_ACT_ERR_ALIGN: return "pointer is not aligned to its element size";
    case GATED_ACT_ERR_DTYPE: return "unknown or unsupported element type";
    case GATED_ACT_ERR_HOST: return "memory the CUDA runtime does not know (pageable or unallocated)";
    case GATED_ACT_ERR_SCRATCH: return "needs more scratch than the library's static array holds";
    case GATED_ACT_ERR_DEVICE: return "device memory of a GPU other than the current one";
    default: return "unknown status";
    }
}

extern "C" int gated_act_last_cuda_error(void) { return gact::g_last_cuda_error; }
