// Library-wide pieces of the C ABI: status strings, the per-device error word
// that kernels set when they meet an index outside the pool (or a bounded wait
// runs out), and cached device queries.
#include <mutex>

#include "pa_internal.h"

namespace pa {

__device__ unsigned int g_error_word;

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing
// arrives at, with the same helper the attention kernel uses, and records a
// timeout in the error word when the limit runs out.
__global__ void selftest_wait_kernel(unsigned long long limit_ns, unsigned int *err) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(smem_u32(&bar), 1);
    fence_mbarrier_init();
    if (!mbar_wait_bounded(smem_u32(&bar), 0, limit_ns)) atomicOr(err, kErrTimeout);
}

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int *g_err_ptr[kMaxDevices];
int g_sms[kMaxDevices];
}  // namespace

unsigned int *device_error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_err_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = (unsigned int *)p;
    }
    return g_err_ptr[dev];
}

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_sms[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

}  // namespace pa

using namespace pa;

extern "C" const char *pa_status_string(pa_status_t status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported combination (no kernel variant)";
        case PA_ERR_CUDA: return "CUDA error";
        case PA_ERR_NO_BLOCKS: return "no free KV blocks";
        case PA_ERR_HOST_MEMORY: return "host memory allocation failed";
        case PA_ERR_DEVICE_BOUNDS: return "kernel met an index outside the pool or table";
        case PA_ERR_DEVICE_TIMEOUT: return "kernel wait timed out";
        case PA_ERR_WORKSPACE: return "workspace too small";
        case PA_ERR_DEVICE_PLAN: return "shared-prefix plan does not match the decode call";
    }
    return "unknown status";
}

extern "C" const char *pa_version(void) { return "paged_kv_cache_150_gb300 0.1 (sm_103a)"; }

extern "C" pa_status_t pa_get_device_error(pa_stream_t stream) {
    unsigned int *err = device_error_word();
    if (!err) return PA_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    unsigned int word = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaMemcpyAsync(&word, err, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaMemsetAsync(err, 0, sizeof(word), s) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
    if (word & kErrTimeout) return PA_ERR_DEVICE_TIMEOUT;
    if (word & (kErrBounds | kErrLength)) return PA_ERR_DEVICE_BOUNDS;
    if (word & kErrPlan) return PA_ERR_DEVICE_PLAN;
    return PA_OK;
}

extern "C" pa_status_t pa_selftest_wait_timeout(int64_t limit_ns, pa_stream_t stream) {
    if (limit_ns <= 0 || limit_ns > (int64_t)kWaitLimitNs) return PA_ERR_INVALID_ARG;
    unsigned int *err = device_error_word();
    if (!err) return PA_ERR_CUDA;
    selftest_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((unsigned long long)limit_ns, err);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
