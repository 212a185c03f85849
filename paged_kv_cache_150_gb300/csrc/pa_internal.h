// Host-side helpers shared by the translation units of libpa.so.
#pragma once

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>

#include "pa.h"
#include "pa_common.cuh"

namespace pa {

inline int dtype_bytes(int32_t dtype) { return dtype == PA_F32 ? 4 : 2; }

inline pa_status_t validate_cache_desc(const pa_cache_desc_t *c) {
    if (!c) return PA_ERR_INVALID_ARG;
    if (c->num_blocks <= 0 || c->block_size <= 0 || c->num_kv_heads <= 0 || c->head_dim <= 0)
        return PA_ERR_INVALID_ARG;
    if (c->dtype != PA_F32 && c->dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    if (c->layout != PA_LAYOUT_ROW && c->layout != PA_LAYOUT_SPLIT) return PA_ERR_INVALID_ARG;
    if (c->layout == PA_LAYOUT_SPLIT && (c->head_dim * dtype_bytes(c->dtype)) % 16 != 0) return PA_ERR_INVALID_ARG;
    if ((int64_t)c->num_blocks * c->block_size >= ((int64_t)1 << 31)) return PA_ERR_INVALID_ARG;
    return PA_OK;
}

// Status of a C++ exception caught at an entry point (the C ABI never lets
// one through): PA_ERR_HOST_MEMORY for a failed host allocation, else
// PA_ERR_CUDA.  Call only inside a catch handler.
inline pa_status_t host_failure() {
    try {
        throw;
    } catch (const std::bad_alloc &) {
        return PA_ERR_HOST_MEMORY;
    } catch (...) {
        return PA_ERR_CUDA;
    }
}

// Device address of the current device's error word (nullptr on failure).
unsigned int *device_error_word();

// Cached device address of one of this library's __device__ variables, per
// device.  The address belongs to the context it was looked up in, so each
// entry keeps that context's unique id and is looked up again when the
// device's current context differs (after cudaDeviceReset, for instance).
constexpr int kMaxDevices = 64;
struct SymbolCache {
    unsigned long long ctx_id[kMaxDevices];
    void *addr[kMaxDevices];
};

// Address of `symbol` (the variable itself, as passed to cudaGetSymbolAddress)
// on the current device, from `cache` or looked up; nullptr on failure.
// Thread-safe; throws nothing.
void *symbol_address(SymbolCache *cache, const void *symbol);

// Streaming multiprocessors of the current device (0 on failure).
int num_sms();

}  // namespace pa
