// Host-side helpers shared by the translation units of libpa.so.
#pragma once

#include <algorithm>
#include <cstdint>
#include <cstring>

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

// Device address of the current device's error word (nullptr on failure).
unsigned int *device_error_word();

// Streaming multiprocessors of the current device (0 on failure).
int num_sms();

}  // namespace pa
