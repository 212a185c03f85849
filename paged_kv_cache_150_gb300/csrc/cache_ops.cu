// Paged KV write (pa_reshape_and_cache) and copy-on-write block copy
// (pa_copy_blocks).  Both are bit copies bound by HBM bandwidth: every byte is
// read once and written once, in 16-byte vectors where the row allows it.
//
// Cache write: "04 · PagedAttention" (nano-vLLM Deep Dive), section 4,
// Mechanism 3 "The slot mapping" - a token's K and V go to the cache row of
// its slot.  In the [NB, B, Hk, D] layout all Hk * D elements of one token are
// contiguous at element offset slot * Hk * D, so one token is one contiguous
// row copy.
// Block copy: "PagedAttention" (tokentrails), step 4 and Code (copy_block); a
// whole block is B * Hk * D contiguous elements in both cache layouts.
#include "pa_internal.h"

namespace pa {

// Row copy by one warp: every lane issues its loads of the K and V rows
// (kUnroll vectors of each) before its stores, so a row is one memory round
// trip.
constexpr int kUnroll = 4;

template <typename V>
__device__ __forceinline__ void warp_copy_rows(V *__restrict__ kd, V *__restrict__ vd, const V *__restrict__ ks,
                                               const V *__restrict__ vs, int64_t n, int lane, bool streaming) {
    for (int64_t j0 = 0; j0 < n; j0 += 32 * kUnroll) {
        V kx[kUnroll], vx[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t j = j0 + u * 32 + lane;
            if (j < n) {
                kx[u] = streaming ? __ldcs(ks + j) : ks[j];
                vx[u] = streaming ? __ldcs(vs + j) : vs[j];
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t j = j0 + u * 32 + lane;
            if (j < n) {
                kd[j] = kx[u];
                vd[j] = vx[u];
            }
        }
    }
}

// A row is cut into NC chunks of 32 * kUnroll vectors; warp w copies chunk
// w % NC of the tokens w / NC, w / NC + NWt, w / NC + 2 NWt, ... (NWt = warps
// per chunk), 32 tokens at a time.  The 32 slots come in one load, and padding
// tokens (slot < 0, e.g. prompt positions already in the prefix cache) are
// dropped by a ballot without touching their rows.
template <typename V>
__global__ void __launch_bounds__(256, 4) reshape_and_cache_kernel(
    const V *__restrict__ k, const V *__restrict__ v, const int32_t *__restrict__ slots,
    int32_t num_tokens, V *__restrict__ k_cache, V *__restrict__ v_cache, int64_t num_slots,
    int32_t row_vecs, unsigned int *__restrict__ err) {
    grid_dependency_wait();    // launched programmatically: the previous grid's writes first
    grid_launch_dependents();  // a programmatically launched successor may get resident early
    constexpr int kChunk = 32 * kUnroll;
    const int lane = threadIdx.x & 31;
    const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int32_t NC = (row_vecs + kChunk - 1) / kChunk;
    const int64_t NWt = (((int64_t)gridDim.x * blockDim.x) >> 5) / NC;
    const int64_t wt = w / NC;
    if (wt >= NWt) return;
    const int64_t j0 = (w - wt * NC) * kChunk;
    const int64_t n = min((int64_t)kChunk, (int64_t)row_vecs - j0);
    for (int64_t t0 = wt; t0 < num_tokens; t0 += 32 * NWt) {
        const int64_t tl = t0 + (int64_t)lane * NWt;
        const int32_t sl = tl < num_tokens ? __ldg(slots + tl) : -1;
        const bool bad = (int64_t)sl >= num_slots;
        if (__any_sync(0xffffffffu, bad) && lane == 0 && j0 == 0) atomicOr(err, kErrBounds);
        unsigned int todo = __ballot_sync(0xffffffffu, sl >= 0 && !bad);
        while (todo) {
            const int b = __ffs(todo) - 1;
            todo &= todo - 1;
            const int64_t s = __shfl_sync(0xffffffffu, sl, b);
            const int64_t t = t0 + (int64_t)b * NWt;
            warp_copy_rows(k_cache + s * row_vecs + j0, v_cache + s * row_vecs + j0, k + t * row_vecs + j0,
                           v + t * row_vecs + j0, n, lane, true);
        }
    }
}

// Split layout: K [NB, Hk, D/x, B, x] receives each token's 16-byte chunks at
// their (head, chunk, offset) positions; V [NB, Hk, D, B] receives one element
// per (head, d) at stride B.
template <typename T>
__global__ void __launch_bounds__(256) reshape_and_cache_split_kernel(
    const T *__restrict__ k, const T *__restrict__ v, const int32_t *__restrict__ slots, int32_t num_tokens,
    T *__restrict__ k_cache, T *__restrict__ v_cache, int64_t num_slots, int32_t B, int32_t Hk, int32_t D,
    unsigned int *__restrict__ err) {
    grid_dependency_wait();
    grid_launch_dependents();
    constexpr int X = 16 / (int)sizeof(T);
    const int64_t per_tok = (int64_t)Hk * D;
    const int64_t total = (int64_t)num_tokens * per_tok;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int32_t t = (int32_t)(i / per_tok);
        const int32_t r = (int32_t)(i - (int64_t)t * per_tok);
        const int32_t h = r / D, d = r - h * D;
        const int32_t s = __ldg(slots + t);
        if (s < 0) continue;
        if ((int64_t)s >= num_slots) {
            if (r == 0) atomicOr(err, kErrBounds);
            continue;
        }
        const int64_t blk = s / B, off = s - blk * B;
        const int64_t head = blk * Hk + h;
        if (d % X == 0) {  // one 16-byte K chunk
            const int64_t kd = ((head * (D / X) + d / X) * B + off) * X;
            *reinterpret_cast<uint4 *>(k_cache + kd) = __ldcs(reinterpret_cast<const uint4 *>(k + i));
        }
        v_cache[(head * D + d) * B + off] = v[i];
    }
}

template <typename V>
__global__ void __launch_bounds__(256) copy_blocks_kernel(V *__restrict__ k_cache, V *__restrict__ v_cache,
                                                          const int32_t *__restrict__ pairs,
                                                          int32_t num_pairs, int32_t num_blocks,
                                                          int64_t block_vecs, int32_t chunks_per_pair,
                                                          unsigned int *__restrict__ err) {
    grid_dependency_wait();    // launched programmatically: the previous grid's writes first
    grid_launch_dependents();  // a programmatically launched successor may get resident early
    const int32_t p = blockIdx.x / chunks_per_pair;
    const int32_t chunk = blockIdx.x - p * chunks_per_pair;
    if (p >= num_pairs) return;
    const int32_t src = __ldg(pairs + 2 * p);
    const int32_t dst = __ldg(pairs + 2 * p + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (chunk == 0 && threadIdx.x == 0) atomicOr(err, kErrBounds);
        return;
    }
    const int64_t per_chunk = (block_vecs + chunks_per_pair - 1) / chunks_per_pair;
    const int64_t lo = chunk * per_chunk;
    const int64_t hi = min(block_vecs, lo + per_chunk);
    const int64_t ks = (int64_t)src * block_vecs, kd = (int64_t)dst * block_vecs;
    // The CTA's warps take consecutive 32 * kUnroll-vector pieces of the chunk.
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    for (int64_t j = lo + (int64_t)warp * 32 * kUnroll; j < hi; j += (int64_t)nwarps * 32 * kUnroll)
        warp_copy_rows(k_cache + kd + j, v_cache + kd + j, k_cache + ks + j, v_cache + ks + j,
                       min((int64_t)32 * kUnroll, hi - j), lane, false);
}

// Launch with programmatic stream serialization; the kernels wait for the
// previous grid (griddepcontrol.wait) before their first memory access, so
// only the launch and scheduling latency overlaps the previous kernel.
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kernel)(KArgs...), int grid, int block, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

static int vec_bytes_for(int64_t row_bytes, const void *a, const void *b, const void *c, const void *d) {
    const uintptr_t any = (uintptr_t)a | (uintptr_t)b | (uintptr_t)c | (uintptr_t)d;
    if (row_bytes % 16 == 0 && any % 16 == 0) return 16;
    if (row_bytes % 8 == 0 && any % 8 == 0) return 8;
    if (row_bytes % 4 == 0 && any % 4 == 0) return 4;
    return 2;
}

}  // namespace pa

using namespace pa;

extern "C" pa_status_t pa_reshape_and_cache(const void *k, const void *v, const int32_t *slot_mapping,
                                            int32_t num_tokens, void *k_cache, void *v_cache,
                                            const pa_cache_desc_t *cache, pa_stream_t stream) {
    pa_status_t st = validate_cache_desc(cache);
    if (st != PA_OK) return st;
    if (num_tokens < 0) return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID_ARG;
    unsigned int *err = device_error_word();
    if (!err) return PA_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    const int64_t num_slots = (int64_t)cache->num_blocks * cache->block_size;
    if (cache->layout == PA_LAYOUT_SPLIT) {
        if (((uintptr_t)k | (uintptr_t)k_cache) % 16 != 0) return PA_ERR_INVALID_ARG;
        const int64_t total = (int64_t)num_tokens * cache->num_kv_heads * cache->head_dim;
        const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256,
                                                                      (int64_t)std::max(num_sms(), 1) * 16));
        if (cache->dtype == PA_BF16)
            launch_pdl(reshape_and_cache_split_kernel<__nv_bfloat16>, grid, 256, s, (const __nv_bfloat16 *)k,
                       (const __nv_bfloat16 *)v, slot_mapping, num_tokens, (__nv_bfloat16 *)k_cache,
                       (__nv_bfloat16 *)v_cache, num_slots, cache->block_size, cache->num_kv_heads,
                       cache->head_dim, err);
        else
            launch_pdl(reshape_and_cache_split_kernel<float>, grid, 256, s, (const float *)k, (const float *)v,
                       slot_mapping, num_tokens, (float *)k_cache, (float *)v_cache, num_slots, cache->block_size,
                       cache->num_kv_heads, cache->head_dim, err);
        return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
    }
    const int64_t row_bytes = (int64_t)cache->num_kv_heads * cache->head_dim * dtype_bytes(cache->dtype);
    const int vb = vec_bytes_for(row_bytes, k, v, k_cache, v_cache);
    const int32_t row_vecs = (int32_t)(row_bytes / vb);
    // One warp per (token, row chunk) up to 32 warps (4 resident CTAs of 256
    // threads) per SM.
    const int threads = 256;
    const int64_t chunks = (row_vecs + 32 * kUnroll - 1) / (32 * kUnroll);
    const int64_t token_warps =
        std::min<int64_t>(num_tokens, std::max<int64_t>(1, (int64_t)std::max(num_sms(), 1) * 32 / chunks));
    const int grid = (int)std::max<int64_t>(1, (token_warps * chunks + 7) / 8);
    switch (vb) {
        case 16:
            launch_pdl(reshape_and_cache_kernel<uint4>, grid, threads, s, (const uint4 *)k, (const uint4 *)v,
                       slot_mapping, num_tokens, (uint4 *)k_cache, (uint4 *)v_cache, num_slots, row_vecs, err);
            break;
        case 8:
            launch_pdl(reshape_and_cache_kernel<uint2>, grid, threads, s, (const uint2 *)k, (const uint2 *)v,
                       slot_mapping, num_tokens, (uint2 *)k_cache, (uint2 *)v_cache, num_slots, row_vecs, err);
            break;
        case 4:
            launch_pdl(reshape_and_cache_kernel<uint32_t>, grid, threads, s, (const uint32_t *)k, (const uint32_t *)v,
                       slot_mapping, num_tokens, (uint32_t *)k_cache, (uint32_t *)v_cache, num_slots, row_vecs, err);
            break;
        default:
            launch_pdl(reshape_and_cache_kernel<uint16_t>, grid, threads, s, (const uint16_t *)k, (const uint16_t *)v,
                       slot_mapping, num_tokens, (uint16_t *)k_cache, (uint16_t *)v_cache, num_slots, row_vecs, err);
            break;
    }
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

extern "C" pa_status_t pa_copy_blocks(void *k_cache, void *v_cache, const pa_cache_desc_t *cache,
                                      const int32_t *src_dst_pairs, int32_t num_pairs,
                                      pa_stream_t stream) {
    pa_status_t st = validate_cache_desc(cache);
    if (st != PA_OK) return st;
    if (num_pairs < 0) return PA_ERR_INVALID_ARG;
    if (num_pairs == 0) return PA_OK;
    if (!k_cache || !v_cache || !src_dst_pairs) return PA_ERR_INVALID_ARG;
    unsigned int *err = device_error_word();
    if (!err) return PA_ERR_CUDA;
    const int64_t block_bytes = (int64_t)cache->block_size * cache->num_kv_heads * cache->head_dim *
                                dtype_bytes(cache->dtype);
    const int vb = vec_bytes_for(block_bytes, k_cache, v_cache, k_cache, v_cache);
    const int64_t block_vecs = block_bytes / vb;
    const int threads = 256;
    // 16 KiB of each tensor per CTA (8 warps x 32 lanes x kUnroll 16-byte
    // vectors: one round trip), at least one CTA per pair
    int32_t chunks = (int32_t)std::max<int64_t>(1, (block_vecs * vb + 16383) / 16384);
    if ((int64_t)num_pairs * chunks > INT32_MAX) chunks = INT32_MAX / num_pairs;
    const int grid = num_pairs * chunks;
    cudaStream_t s = (cudaStream_t)stream;
    switch (vb) {
        case 16:
            launch_pdl(copy_blocks_kernel<uint4>, grid, threads, s, (uint4 *)k_cache, (uint4 *)v_cache,
                       src_dst_pairs, num_pairs, cache->num_blocks, block_vecs, chunks, err);
            break;
        case 8:
            launch_pdl(copy_blocks_kernel<uint2>, grid, threads, s, (uint2 *)k_cache, (uint2 *)v_cache,
                       src_dst_pairs, num_pairs, cache->num_blocks, block_vecs, chunks, err);
            break;
        case 4:
            launch_pdl(copy_blocks_kernel<uint32_t>, grid, threads, s, (uint32_t *)k_cache, (uint32_t *)v_cache,
                       src_dst_pairs, num_pairs, cache->num_blocks, block_vecs, chunks, err);
            break;
        default:
            launch_pdl(copy_blocks_kernel<uint16_t>, grid, threads, s, (uint16_t *)k_cache, (uint16_t *)v_cache,
                       src_dst_pairs, num_pairs, cache->num_blocks, block_vecs, chunks, err);
            break;
    }
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
