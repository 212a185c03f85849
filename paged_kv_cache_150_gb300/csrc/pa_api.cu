// Library-wide pieces of the C ABI: status strings, the per-device error word
// that kernels set when they meet an index outside the pool (or a bounded wait
// runs out), and cached device queries.
#include <cuda.h>

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
std::mutex g_mu;
SymbolCache g_err_cache;
int g_sms[kMaxDevices];

// Unique id of the calling thread's current context (cuCtxGetId), or 0 when
// there is none or the driver does not offer the query.  Both driver entry
// points are resolved once.
unsigned long long current_context_id() {
    using GetCurrentFn = CUresult (*)(CUcontext *);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long *);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *a = nullptr, *b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) == cudaSuccess &&
            qa == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) == cudaSuccess &&
            qb == cudaDriverEntryPointSuccess) {
            get_current = (GetCurrentFn)a;
            get_id = (GetIdFn)b;
        }
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}
}  // namespace

void *symbol_address(SymbolCache *cache, const void *symbol) try {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    unsigned long long id = current_context_id();
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (id != 0 && cache->ctx_id[dev] == id && cache->addr[dev]) return cache->addr[dev];
    }
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess || !p) return nullptr;
    id = current_context_id();  // the lookup makes the device's primary context current
    std::lock_guard<std::mutex> lock(g_mu);
    cache->ctx_id[dev] = id;  // 0 (unknown): looked up again next time
    cache->addr[dev] = p;
    return p;
} catch (...) {
    return nullptr;
}

unsigned int *device_error_word() { return (unsigned int *)symbol_address(&g_err_cache, (const void *)&g_error_word); }

int num_sms() try {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_sms[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_sms[dev] = n;
    }
    return g_sms[dev];
} catch (...) {
    return 0;
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
