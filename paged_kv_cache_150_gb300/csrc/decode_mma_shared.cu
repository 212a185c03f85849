// Instantiations of the tensor-core decode kernel with a shared-prefix
// plan (the kernel itself is in decode_mma.cuh).
#include "pa_internal.h"

#include "decode_kernels.h"
#include "decode_merge.cuh"
#include "decode_mma.cuh"

namespace pa {

template <int LAYOUT>
static const void *mma_fn_shared(int D, int B) {
    if (D == 128 && B == 16) return (const void *)decode_mma_kernel<128, 16, LAYOUT, true>;
    if (D == 128 && B == 32) return (const void *)decode_mma_kernel<128, 32, LAYOUT, true>;
    if (D == 64 && B == 16) return (const void *)decode_mma_kernel<64, 16, LAYOUT, true>;
    if (D == 64 && B == 32) return (const void *)decode_mma_kernel<64, 32, LAYOUT, true>;
    return nullptr;
}

const void *mma_kernel_ptr_shared(int D, int B, int layout) {
    return layout == PA_LAYOUT_SPLIT ? mma_fn_shared<PA_LAYOUT_SPLIT>(D, B) : mma_fn_shared<PA_LAYOUT_ROW>(D, B);
}

}  // namespace pa
