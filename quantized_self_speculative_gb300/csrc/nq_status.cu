// nq_status.cu -- the sticky per-device status word and small host utilities.
#include <mutex>

#include "nq_internal.cuh"

namespace nq {

// Sticky error bits (NQ_DEV_*) set by kernels that detect bad data.
__device__ unsigned int g_device_status;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int *g_status_ptr[kMaxDevices];
int g_sms[kMaxDevices];
}  // namespace

unsigned int *device_status_ptr()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<unsigned int *>(p);
    }
    return g_status_ptr[dev];
}

int sm_count()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_sms[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

}  // namespace nq

extern "C" const char *nq_status_string(int status)
{
    switch (status) {
    case NQ_OK: return "NQ_OK";
    case NQ_ERR_ARG: return "NQ_ERR_ARG: invalid argument";
    case NQ_ERR_SHAPE: return "NQ_ERR_SHAPE: unsupported shape";
    case NQ_ERR_ALIGN: return "NQ_ERR_ALIGN: device pointer not 16-byte aligned";
    case NQ_ERR_CUDA: return "NQ_ERR_CUDA: CUDA runtime error";
    case NQ_ERR_NONFINITE: return "NQ_ERR_NONFINITE: non-finite logits";
    case NQ_ERR_TIMEOUT: return "NQ_ERR_TIMEOUT: bounded device wait expired";
    case NQ_ERR_WORKSPACE: return "NQ_ERR_WORKSPACE: workspace too small";
    case NQ_ERR_TOKEN: return "NQ_ERR_TOKEN: draft token outside [0, V)";
    default: return "unknown nq_status";
    }
}

extern "C" nq_status nq_get_device_status(cudaStream_t stream, uint32_t *out)
{
    if (!out) return NQ_ERR_ARG;
    unsigned int *p = nq::device_status_ptr();
    if (!p) return NQ_ERR_CUDA;
    unsigned int h = 0;
    if (cudaMemcpyAsync(&h, p, sizeof(h), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return NQ_ERR_CUDA;
    if (cudaMemsetAsync(p, 0, sizeof(unsigned int), stream) != cudaSuccess) return NQ_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return NQ_ERR_CUDA;
    *out = h;
    return NQ_OK;
}
