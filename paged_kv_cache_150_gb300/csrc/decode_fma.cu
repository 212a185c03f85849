// Instantiations of the TMA-staged CUDA-core decode kernel (the kernel itself
// is in decode_fma.cuh).
#include "pa_internal.h"

#include "decode_kernels.h"
#include "decode_fma.cuh"

namespace pa {

template <typename T, int D>
static const void *fma_fn(int gmax) {
    if (gmax == 1) return (const void *)decode_fma_kernel<T, D, 1>;
    if (gmax == 2) return (const void *)decode_fma_kernel<T, D, 2>;
    if (gmax == 4) return (const void *)decode_fma_kernel<T, D, 4>;
    return (const void *)decode_fma_kernel<T, D, 8>;
}

const void *fma_kernel_ptr(int dtype, int D, int G) {
    const int gm = fma_gmax(G);
    if (dtype == PA_F32) {
        if (D == 64) return fma_fn<float, 64>(gm);
        if (D == 128) return fma_fn<float, 128>(gm);
    } else {
        if (D == 64) return fma_fn<__nv_bfloat16, 64>(gm);
        if (D == 128) return fma_fn<__nv_bfloat16, 128>(gm);
        if (D == 256) return fma_fn<__nv_bfloat16, 256>(gm);
    }
    return nullptr;
}

}  // namespace pa
