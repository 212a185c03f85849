// Host handles of the decode attention kernels.  The instantiations live in
// their own translation units (decode_mma_plain.cu, decode_mma_shared.cu,
// decode_simt.cu, decode_fma.cu) so that nvcc compiles them in parallel;
// decode.cu picks one by shape and launches it through the handle.
#pragma once

namespace pa {

// Query heads per KV head rounded up to the SIMT kernel's instantiations.
inline int simt_gmax(int G) { return G <= 1 ? 1 : (G <= 4 ? 4 : 8); }

// decode_simt_kernel for (dtype, head_dim, G, layout); nullptr if none.
const void *simt_kernel_ptr(int dtype, int D, int G, int layout);

// Query heads per KV head rounded up to the TMA-staged CUDA-core kernel's
// instantiations.
inline int fma_gmax(int G) { return G <= 1 ? 1 : (G <= 2 ? 2 : (G <= 4 ? 4 : 8)); }

// decode_fma_kernel for (dtype, head_dim, G) (row layout); nullptr if none.
const void *fma_kernel_ptr(int dtype, int D, int G);

// decode_mma_kernel<D, B, layout, kShared = false / true>; nullptr if none.
const void *mma_kernel_ptr_plain(int D, int B, int layout);
const void *mma_kernel_ptr_shared(int D, int B, int layout);

}  // namespace pa
