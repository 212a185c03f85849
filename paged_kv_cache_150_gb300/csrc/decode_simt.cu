// Instantiations of the CUDA-core decode kernel (the kernel itself is in
// decode_simt.cuh).
#include "pa_internal.h"

#include "decode_kernels.h"
#include "decode_merge.cuh"
#include "decode_simt.cuh"

namespace pa {

template <typename T, int D, int GMAX>
static const void *simt_fn(int layout) {
    return layout == PA_LAYOUT_SPLIT ? (const void *)decode_simt_kernel<T, D, GMAX, PA_LAYOUT_SPLIT>
                                     : (const void *)decode_simt_kernel<T, D, GMAX, PA_LAYOUT_ROW>;
}

const void *simt_kernel_ptr(int dtype, int D, int G, int layout) {
    const int gm = simt_gmax(G);
#define PA_SIMT_CASE(TT, DD)                                        \
    if (D == DD) {                                                  \
        if (gm == 1) return simt_fn<TT, DD, 1>(layout);             \
        if (gm == 4) return simt_fn<TT, DD, 4>(layout);             \
        return simt_fn<TT, DD, 8>(layout);                          \
    }
    if (dtype == PA_F32) {
        PA_SIMT_CASE(float, 64)
        PA_SIMT_CASE(float, 128)
    } else {
        PA_SIMT_CASE(__nv_bfloat16, 64)
        PA_SIMT_CASE(__nv_bfloat16, 128)
        PA_SIMT_CASE(__nv_bfloat16, 256)
    }
#undef PA_SIMT_CASE
    return nullptr;
}

}  // namespace pa
