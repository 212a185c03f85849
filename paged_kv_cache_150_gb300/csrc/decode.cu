// Paged decode attention (pa_decode).
//
// What is computed: for every sequence i and query head h,
//   out[i, h] = softmax_j(scale * q[i, h] . K_j) V_j   over j < seq_lens[i],
// with K_j, V_j the cache rows of slot table[i][j / B] * B + j % B
// ("10 PagedAttention" (PidokuInfra), section 4 PhysicalIndex and section 5
// "The kernel side"; "PagedAttention" (tokentrails), step 3: the same
// attention as over contiguous memory).  Query head h reads KV head
// h / (H / Hk).
//
// How (GB300 design; the pages give only a one-CTA-per-(seq, head) sketch):
// 1. decode_plan_kernel: one CTA turns seq_lens into block counts and their
//    exclusive prefix sums cu[], clamps bad lengths (recording them), zeroes
//    the merge counters and writes the zero output of empty sequences.
// 2. A persistent grid of C CTAs splits the flattened list of
//    (KV-head group, sequence, block) into Ce = min(C, W) equal contiguous
//    ranges (split_begin).  A CTA walks its range; each of its consumer warps
//    owns one KV head and all G query heads that share it, so each KV byte is
//    read from HBM once.  A range piece covering a whole sequence writes `out`
//    directly.  A piece of a longer sequence writes an unnormalised partial
//    (running max m in log2 units, sum l, accumulator) to the workspace and
//    bumps an arrival counter for its (sequence, KV head); the warp that
//    arrives last merges every piece (the split-K reduce, fused):
//      out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p,  M = max_p m_p.
//    Nothing ever waits for another CTA: the merge is done by whoever is last.
//    With the caller's host copy of the lengths showing a sequence cut into
//    kLongMergePieces or more pieces (long contexts), such (sequence, KV head)
//    pairs are merged instead by long_merge_kernel right after the launch,
//    spread over the GPU; the device decides per sequence from its own cu[].
//    Without a shared-prefix plan and with N + 1 <= kLocalCuMax, each
//    tensor-core CTA computes the same cu[] from seq_lens in its own shared
//    memory and starts on its blocks while the plan kernel still runs; it
//    waits for that kernel only before its first arrival (the counters must
//    be zeroed) and before it exits.
// 3. With a shared-prefix plan (sequences whose tables start with the same
//    physical blocks), part of the grid reads each shared block once for all
//    sharers' query heads, the rest reads each sequence's own blocks, and
//    shared_merge_kernel merges the sequences with a shared prefix.
//
// Device code: decode_merge.cuh (pieces and merges), decode_plan.cuh (plan
// kernel), decode_simt.cuh (CUDA-core kernel), decode_mma.cuh (tensor-core
// kernel).  The attention kernels are instantiated in decode_simt.cu,
// decode_mma_plain.cu and decode_mma_shared.cu (compiled in parallel); this
// file holds the plan and merge kernels, the host side and the C ABI entry
// points.
//
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "pa_internal.h"

#include "decode_kernels.h"
#include "decode_merge.cuh"
#include "decode_plan.cuh"
#include "decode_fma.cuh"  // FmaSmem, fma_lanes_per_token (host side)

namespace pa {

// ====================================================================== host
namespace {

struct DecodePlan {
    int kernel;    // PA_KERNEL_SIMT or PA_KERNEL_MMA
    bool fma;      // CUDA-core: the TMA-staged kernel (decode_fma_kernel), not the per-token one
    int stages;    // decode_fma_kernel: ring stages
    int NH;        // KV heads per CTA (consumer warps)
    int NG;        // head groups = Hk / NH
    int HPG;       // query heads per group = NH * G
    int C;         // persistent CTAs
    bool shared;   // a shared-prefix plan is used
    bool tc;       // its 64-row passes may run on tcgen05 (row layout; the CTAs' tensor memory fits an SM)
    bool local_cu; // tensor-core CTAs compute the prefix sums themselves (kLocalCuMax)
    size_t smem;   // dynamic shared memory of the attention kernel
    // workspace layout (byte offsets)
    size_t off_lens, off_cu, off_cnt, off_start, off_ml, off_acc;
    size_t off_skip, off_ctl, off_start_s, off_rowseq, off_ml_s, off_acc_s;  // shared-prefix part
    size_t total;
};

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int largest_divisor_at_most(int n, int cap) {
    for (int d = std::min(n, cap); d >= 1; --d)
        if (n % d == 0) return d;
    return 1;
}

bool mma_supported(const pa_cache_desc_t *c, int G) {
    return c->dtype == PA_BF16 && (c->head_dim == 64 || c->head_dim == 128) &&
           (c->block_size == 16 || c->block_size == 32) && G >= 1 && G <= 8;
}

bool simt_supported(const pa_cache_desc_t *c, int G) {
    const bool d_ok = c->dtype == PA_F32 ? (c->head_dim == 64 || c->head_dim == 128)
                                         : (c->head_dim == 64 || c->head_dim == 128 || c->head_dim == 256);
    return d_ok && G >= 1 && G <= 8;
}

// The TMA-staged CUDA-core kernel covers the row layout for D whose rows are
// whole 128-byte lines (fp32 64 and 128, bf16 64, 128 and 256), G <= 8 and any
// block size whose ring fits shared memory (fma_shape).
constexpr size_t kFmaStageCap = 32 * 1024;  // K + V bytes of one ring stage, NH chosen to fit
constexpr size_t kFmaRingTarget = 64 * 1024;
constexpr size_t kFmaSmemMax = 200 * 1024;

// NH (KV heads per CTA), stages and shared memory of decode_fma_kernel for
// this shape; false if its ring does not fit.
bool fma_shape(const pa_cache_desc_t *c, int G, int *NH, int *stages, size_t *smem) {
    if (c->layout != PA_LAYOUT_ROW || G < 1 || G > 8 || c->block_size > 256) return false;
    const bool d_ok = c->dtype == PA_F32 ? (c->head_dim == 64 || c->head_dim == 128)
                                         : (c->head_dim == 64 || c->head_dim == 128 || c->head_dim == 256);
    if (!d_ok) return false;
    const int eb = dtype_bytes(c->dtype), line = 128 / eb, D = c->head_dim, B = c->block_size;
    int nh = 1;
    for (int d = std::min(c->num_kv_heads, kMmaMaxHeads); d >= 1; --d) {
        if (c->num_kv_heads % d == 0 && 2 * (size_t)FmaSmem::box_bytes(d, D, B, line) <= kFmaStageCap) {
            nh = d;
            break;
        }
    }
    const size_t stage = 2 * (size_t)FmaSmem::box_bytes(nh, D, B, line);
    const int st = (int)std::max<size_t>(2, std::min<size_t>(8, kFmaRingTarget / stage));
    const int gm = fma_gmax(G);
    const size_t bytes = FmaSmem::bytes(st, nh, D, B, line, gm, fma_lanes_per_token(B));
    if (bytes > kFmaSmemMax) return false;
    *NH = nh;
    *stages = st;
    *smem = bytes;
    return true;
}

// kMmaStages stages of NH head slabs of K and of V, mbarriers after the
// tiles; with a shared-prefix plan two halves of shared_half_bytes (each the
// largest of the own-block, mma.sync and tcgen05 shared-prefix maps); 1024
// bytes to align the base.
size_t mma_smem_bytes(int D, int B, int NH, bool shared) {
    const size_t slab = (size_t)(D / 64) * B * 128;
    if (shared) return (size_t)shared_halves(D, B) * shared_half_bytes(D, B) + 1024;  // halves (NH = kPlanWarps)
    return (size_t)kMmaStages * 2 * NH * slab + 2 * (size_t)kMmaStages * sizeof(uint64_t) + 1024;
}

// Logical CTAs per CTA of the tensor-core launch (halves with a plan).
int mma_halves(int D, int B, bool shared) { return shared ? shared_halves(D, B) : 1; }
// Threads of a tensor-core attention CTA: NH consumer warps and a producer
// per half.
int mma_threads(int NH, int halves) { return (NH + 1) * 32 * halves; }

// Tensor-memory columns a tcgen05 shared-prefix CTA allocates (TcSmem::kCols).
int tc_tmem_cols(int D) { return D == 128 ? 256 : 128; }

// Pieces from which a (sequence, KV head) is merged by long_merge_kernel
// rather than by the CTA whose piece arrives last.
constexpr int32_t kLongMergePieces = 8;

// kLongMergePieces if, with these host lengths (clamped as the plan kernel
// clamps them), some sequence is cut into that many pieces; else 0.  A hint
// only: the device decides per sequence from its own seq_lens.  Two passes
// over the lengths (the total, then a running prefix): nothing is allocated.
int32_t long_merge_pieces(const int32_t *host_lens, int32_t N, int32_t B, int32_t max_len, int32_t NG, int32_t C) {
    auto blocks = [&](int32_t i) -> int64_t {
        int32_t L = host_lens[i];
        if (L < 0 || L > max_len) L = 0;
        return (L + B - 1) / B;
    };
    int64_t Wg = 0;
    for (int32_t i = 0; i < N; ++i) Wg += blocks(i);
    const int64_t W = (int64_t)NG * Wg;
    if (W == 0) return 0;
    const int64_t Ce = std::min<int64_t>(C, W);
    int64_t cu = 0;  // blocks of the sequences before i
    for (int32_t i = 0; i < N; ++i) {
        const int64_t nb = blocks(i);
        // nb blocks span at most nb * Ce / W + 2 CTAs: most sequences need no exact count
        if (nb > 0 && nb * Ce >= (int64_t)(kLongMergePieces - 2) * W) {
            for (int32_t g = 0; g < NG; ++g) {
                const int64_t x0 = g * Wg + cu;
                if (split_owner(x0 + nb - 1, W, Ce) - split_owner(x0, W, Ce) + 1 >= kLongMergePieces)
                    return kLongMergePieces;
            }
        }
        cu += nb;
    }
    return 0;
}

// The min_pieces of a call: long_merge_pieces from the host hint, for the
// tensor-core kernel without a shared-prefix plan; else 0.
int32_t call_min_pieces(const DecodePlan &p, const pa_decode_opts_t *opts, int32_t N, int32_t B, int32_t max_len) {
    if (p.kernel != PA_KERNEL_MMA || p.shared || !opts || !opts->host_seq_lens) return 0;
    return long_merge_pieces(opts->host_seq_lens, N, B, max_len, p.NG, p.C);
}

const void *mma_kernel_ptr(int D, int B, int layout, bool shared) {
    return shared ? mma_kernel_ptr_shared(D, B, layout) : mma_kernel_ptr_plain(D, B, layout);
}

// Occupancy-based default split count: one full wave of resident CTAs.  The
// answer is fixed per (device, kernel, threads, shared memory) and kept in a
// fixed table: the occupancy query costs about a microsecond of host time per
// call.  -1 on failure.
int default_ctas(const void *fn, int threads, size_t smem) {
    struct Entry {
        int dev;
        const void *fn;
        int threads;
        size_t smem;
        int ctas;
    };
    constexpr int kEntries = 256;  // distinct (device, kernel, shape) answers kept; later ones are not cached
    static std::mutex mu;
    static Entry cache[kEntries];
    static int used = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < used; ++i) {
            const Entry &e = cache[i];
            if (e.dev == dev && e.fn == fn && e.threads == threads && e.smem == smem) return e.ctas;
        }
    }
    const int sms = num_sms();
    if (sms <= 0) return -1;
    int per_sm = 0;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return -1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem) != cudaSuccess) return -1;
    const int ctas = sms * std::max(per_sm, 1);
    std::lock_guard<std::mutex> lock(mu);
    if (used < kEntries) cache[used++] = Entry{dev, fn, threads, smem, ctas};
    return ctas;
}

pa_status_t make_plan(const pa_cache_desc_t *c, int32_t N, int32_t H, const pa_decode_opts_t *opts,
                      bool need_default_splits, DecodePlan *p) {
    pa_status_t st = validate_cache_desc(c);
    if (st != PA_OK) return st;
    if (N < 0 || H <= 0 || H % c->num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    const int G = H / c->num_kv_heads;
    const int want = opts ? opts->kernel : PA_KERNEL_AUTO;
    if (want != PA_KERNEL_AUTO && want != PA_KERNEL_SIMT && want != PA_KERNEL_MMA) return PA_ERR_INVALID_ARG;
    if (opts && opts->num_splits < 0) return PA_ERR_INVALID_ARG;
    int kernel;
    if (want == PA_KERNEL_MMA || (want == PA_KERNEL_AUTO && mma_supported(c, G))) {
        if (!mma_supported(c, G)) return PA_ERR_UNSUPPORTED;
        kernel = PA_KERNEL_MMA;
    } else {
        if (!simt_supported(c, G)) return PA_ERR_UNSUPPORTED;
        kernel = PA_KERNEL_SIMT;
    }
    p->kernel = kernel;
    p->shared = false;
    p->fma = false;
    p->stages = 0;
    if (kernel == PA_KERNEL_SIMT && fma_shape(c, G, &p->NH, &p->stages, &p->smem)) {
        p->fma = true;
    } else if (kernel == PA_KERNEL_MMA) {
        p->NH = largest_divisor_at_most(c->num_kv_heads, kMmaMaxHeads);
        // Shared-prefix CTAs use 4 consumer warps: the launch shape must match.
        p->shared = opts && opts->shared_plan && p->NH == kPlanWarps;
        p->smem = mma_smem_bytes(c->head_dim, c->block_size, p->NH, p->shared);
    } else {
        p->NH = largest_divisor_at_most(c->num_kv_heads, 8);
        p->smem = 0;
    }
    p->NG = c->num_kv_heads / p->NH;
    p->HPG = p->NH * G;
    const int threads = kernel == PA_KERNEL_MMA ? mma_threads(p->NH, mma_halves(c->head_dim, c->block_size, p->shared))
                        : p->fma                ? (p->NH + 1) * 32
                                                : p->NH * 32;
    const int C_given = opts ? opts->num_splits : 0;
    int C = C_given;
    if (C == 0) {
        if (!need_default_splits) return PA_ERR_INVALID_ARG;
        const void *fn = kernel == PA_KERNEL_MMA ? mma_kernel_ptr(c->head_dim, c->block_size, c->layout, p->shared)
                         : p->fma             ? fma_kernel_ptr(c->dtype, c->head_dim, G)
                                              : simt_kernel_ptr(c->dtype, c->head_dim, G, c->layout);
        C = default_ctas(fn, threads, p->smem);
        if (C <= 0) return PA_ERR_CUDA;
        C *= kernel == PA_KERNEL_MMA ? mma_halves(c->head_dim, c->block_size, p->shared) : 1;  // logical CTAs
    }
    p->C = C;
    if (p->shared && C < 2) {  // shared prefixes need a CTA of each kind
        p->shared = false;
        p->smem = mma_smem_bytes(c->head_dim, c->block_size, p->NH, false);
    }
    // tcgen05 shared-prefix halves allocate tensor memory; both halves of
    // every CTA of the launch that can be resident on one SM must find their
    // columns (512 per SM), so that an allocation never waits on a CTA of
    // the same launch.
    p->tc = false;
    if (p->shared && c->layout == PA_LAYOUT_ROW) {
        const void *fn = mma_kernel_ptr(c->head_dim, c->block_size, c->layout, true);
        const int all = default_ctas(fn, threads, p->smem), sms = num_sms();
        const int halves = mma_halves(c->head_dim, c->block_size, true);
        if (all > 0 && sms > 0) p->tc = (all / sms) * halves * tc_tmem_cols(c->head_dim) <= 512;
    }
    // Without a plan, tensor-core CTAs keep their own prefix sums when they
    // fit and the room for them leaves as many CTAs resident per SM (checked
    // for the largest room, kLocalCuMax entries: one cached answer per shape).
    p->local_cu = false;
    if (kernel == PA_KERNEL_MMA && !p->shared && N + 1 <= kLocalCuMax) {
        const size_t extra = ((size_t)(N + 1) * sizeof(int32_t) + 15) & ~(size_t)15;
        bool fits = true;
        if (C_given == 0) {
            const void *fn = mma_kernel_ptr(c->head_dim, c->block_size, c->layout, false);
            fits = default_ctas(fn, threads, p->smem + (size_t)kLocalCuMax * sizeof(int32_t)) == C;
        }
        if (fits) {
            p->local_cu = true;
            p->smem += extra;
        }
    }
    const size_t slots = (size_t)C + (size_t)p->NG * N;
    size_t off = 0;
    p->off_lens = off;
    off = align256(off + sizeof(int32_t) * (size_t)std::max(N, 1));
    p->off_cu = off;
    off = align256(off + sizeof(int32_t) * ((size_t)N + 1));
    p->off_cnt = off;
    off = align256(off + sizeof(uint32_t) * (size_t)std::max(N, 1) * c->num_kv_heads);
    p->off_start = off;
    off = align256(off + sizeof(int32_t) * (size_t)C);
    p->off_ml = off;
    off = align256(off + sizeof(float2) * slots * p->HPG);
    p->off_acc = off;
    off = align256(off + sizeof(float) * slots * p->HPG * c->head_dim);
    p->off_skip = p->off_ctl = p->off_start_s = p->off_rowseq = p->off_ml_s = p->off_acc_s = 0;
    if (p->shared) {
        // virtual sequences V <= N (checked on the device), so at most
        // C + Hk * N shared-prefix slots of kPlanSlotRows query rows
        const size_t slots_s = (size_t)C + (size_t)c->num_kv_heads * N;
        p->off_skip = off;
        off = align256(off + sizeof(int32_t) * (size_t)std::max(N, 1));
        p->off_ctl = off;
        off = align256(off + sizeof(int32_t) * 8);
        p->off_start_s = off;
        off = align256(off + sizeof(int32_t) * (size_t)C);
        p->off_rowseq = off;  // V <= N virtual sequences of R <= kPlanSlotRows rows
        off = align256(off + sizeof(int32_t) * (size_t)std::max(N, 1) * kPlanSlotRows);
        p->off_ml_s = off;
        off = align256(off + sizeof(float2) * slots_s * kPlanSlotRows);
        p->off_acc_s = off;
        off = align256(off + sizeof(float) * slots_s * kPlanSlotRows * c->head_dim);
    }
    p->total = off;
    return PA_OK;
}

// Launch with programmatic stream serialization: the grid may be scheduled
// while the previous kernel on the stream finishes; the kernel itself calls
// griddepcontrol.wait before touching anything that kernel produced.
cudaError_t launch_pdl(const void *fn, dim3 grid, dim3 block, void **args, size_t smem, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)ptr;
    });
    return fn;
}

// 4-D maps over one cache (128-byte rows: 64 bf16 or 32 fp32 elements); NH
// heads per box (the own-block CTAs' NH, or 1 for the shared-prefix CTAs).
// The split layout is bf16 only (tensor-core kernel).
// Row layout: {64, NB*B, D/64, Hk} with byte strides {Hk*D*2, 128, D*2}, box
// {64, B, D/64, NH}, 128-byte swizzle -> shared [head][half][token][64].
// Split layout (K [NB, Hk, D/8, B, 8] or V [NB, Hk, D, B]): each (block, head)
// slab is D*B contiguous elements, viewed as {64, D*B/64, Hk, NB} with strides
// {128, D*B*2, Hk*D*B*2}, box {64, D*B/64, NH, 1}, no swizzle -> the slab's
// own byte order in shared memory.
bool encode_cache_map(CUtensorMap *map, const void *base, const pa_cache_desc_t *c, int NH, bool one_panel = false) {
    auto fn = encode_fn();
    if (!fn) return false;
    const int D = c->head_dim;
    const int B = c->block_size;
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const int eb = dtype_bytes(c->dtype), line = 128 / eb;
    const CUtensorMapDataType et = c->dtype == PA_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUresult r;
    if (c->layout == PA_LAYOUT_SPLIT) {
        cuuint64_t dims[4] = {64, (cuuint64_t)D * B / 64, (cuuint64_t)c->num_kv_heads, (cuuint64_t)c->num_blocks};
        cuuint64_t strides[3] = {128, (cuuint64_t)D * B * 2, (cuuint64_t)c->num_kv_heads * D * B * 2};
        cuuint32_t box[4] = {64, (cuuint32_t)(D * B / 64), (cuuint32_t)NH, 1};
        r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        cuuint64_t dims[4] = {(cuuint64_t)line, (cuuint64_t)c->num_blocks * B, (cuuint64_t)(D / line),
                              (cuuint64_t)c->num_kv_heads};
        cuuint64_t strides[3] = {(cuuint64_t)c->num_kv_heads * D * eb, 128, (cuuint64_t)D * eb};
        cuuint32_t box[4] = {(cuuint32_t)line, (cuuint32_t)B, one_panel ? 1u : (cuuint32_t)(D / line), (cuuint32_t)NH};
        r = fn(map, et, 4, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return r == CUDA_SUCCESS;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" size_t pa_decode_workspace_bytes(const pa_cache_desc_t *cache, int32_t num_seqs, int32_t num_heads,
                                            const pa_decode_opts_t *opts) try {
    DecodePlan p;
    if (make_plan(cache, num_seqs, num_heads, opts, true, &p) != PA_OK) return 0;
    return p.total;
} catch (...) {
    return 0;
}

extern "C" int32_t pa_decode_launch_count(const pa_cache_desc_t *cache, int32_t num_seqs, int32_t num_heads,
                                          int32_t max_blocks_per_seq, const pa_decode_opts_t *opts) try {
    DecodePlan p;
    const pa_status_t st = make_plan(cache, num_seqs, num_heads, opts, true, &p);
    if (st != PA_OK) return (int32_t)st;
    if (num_seqs == 0) return 0;
    if (max_blocks_per_seq <= 0 || (int64_t)max_blocks_per_seq * cache->block_size >= ((int64_t)1 << 31))
        return (int32_t)PA_ERR_INVALID_ARG;
    const int32_t min_pieces =
        call_min_pieces(p, opts, num_seqs, cache->block_size, max_blocks_per_seq * cache->block_size);
    return 2 + (p.shared ? 1 : 0) + (min_pieces > 0 ? 1 : 0);
} catch (...) {
    return (int32_t)host_failure();
}

extern "C" int32_t pa_decode_shared_tc(const pa_cache_desc_t *cache, int32_t num_seqs, int32_t num_heads,
                                       const pa_decode_opts_t *opts) try {
    DecodePlan p;
    const pa_status_t st = make_plan(cache, num_seqs, num_heads, opts, true, &p);
    if (st != PA_OK) return (int32_t)st;
    return p.shared && p.tc ? 1 : 0;
} catch (...) {
    return (int32_t)host_failure();
}

extern "C" int32_t pa_decode_default_splits(const pa_cache_desc_t *cache, int32_t num_heads,
                                            const pa_decode_opts_t *opts) try {
    pa_decode_opts_t o = opts ? *opts : pa_decode_opts_t{0, PA_KERNEL_AUTO, nullptr, nullptr, nullptr, nullptr};
    o.num_splits = 0;
    DecodePlan p;
    const pa_status_t st = make_plan(cache, 1, num_heads, &o, true, &p);
    return st == PA_OK ? p.C : (int32_t)st;
} catch (...) {
    return (int32_t)host_failure();
}

extern "C" void pa_split_range(int64_t total_blocks, int32_t num_splits, int32_t c, int64_t *begin,
                               int64_t *end) {
    if (begin) *begin = split_begin(c, total_blocks, num_splits);
    if (end) *end = split_begin((int64_t)c + 1, total_blocks, num_splits);
}

extern "C" int32_t pa_split_owner(int64_t total_blocks, int32_t num_splits, int64_t x) {
    return split_owner(x, total_blocks, num_splits);
}

extern "C" pa_status_t pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                                 const pa_cache_desc_t *cache, const int32_t *block_tables,
                                 int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs,
                                 int32_t num_heads, float scale, void *workspace, size_t workspace_bytes,
                                 const pa_decode_opts_t *opts, pa_stream_t stream) try {
    DecodePlan p;
    pa_status_t st = make_plan(cache, num_seqs, num_heads, opts, true, &p);
    if (st != PA_OK) return st;
    if (num_seqs == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens || !workspace)
        return PA_ERR_INVALID_ARG;
    if (max_blocks_per_seq <= 0 || (int64_t)num_seqs * max_blocks_per_seq >= ((int64_t)1 << 31) ||
        (int64_t)max_blocks_per_seq * cache->block_size >= ((int64_t)1 << 31))
        return PA_ERR_INVALID_ARG;
    if (!(scale == scale)) return PA_ERR_INVALID_ARG;
    if (((uintptr_t)workspace & 255) != 0) return PA_ERR_INVALID_ARG;
    if (workspace_bytes < p.total) return PA_ERR_WORKSPACE;
    const int eb = dtype_bytes(cache->dtype);
    if (((uintptr_t)q | (uintptr_t)out) % (size_t)(eb * 2) != 0) return PA_ERR_INVALID_ARG;
    if (p.shared && (uintptr_t)q % 16 != 0) {  // shared-prefix warps read q rows in 16-byte pieces
        p.shared = false;
        p.tc = false;
        p.smem = mma_smem_bytes(cache->head_dim, cache->block_size, p.NH, false);
    }
    unsigned int *err = device_error_word();
    if (!err) return PA_ERR_CUDA;

    uint8_t *ws = (uint8_t *)workspace;
    int32_t *lens_ws = (int32_t *)(ws + p.off_lens);
    int32_t *cu = (int32_t *)(ws + p.off_cu);
    unsigned int *cnt = (unsigned int *)(ws + p.off_cnt);
    int32_t *start_seq = (int32_t *)(ws + p.off_start);
    float2 *ml = (float2 *)(ws + p.off_ml);
    float *acc = (float *)(ws + p.off_acc);
    const int G = num_heads / cache->num_kv_heads;
    const float scale_log2 = scale * 1.4426950408889634f;
    const int32_t max_len = max_blocks_per_seq * cache->block_size;
    cudaStream_t s = (cudaStream_t)stream;
    cudaGetLastError();  // clear a stale launch error so the checks below are ours

    const int32_t HD = num_heads * cache->head_dim;
    const int32_t ncnt = num_seqs * cache->num_kv_heads;
    SharedArgs sh{};
    if (p.shared) {
        sh.plan = opts->shared_plan;
        sh.skip = (const int32_t *)(ws + p.off_skip);
        sh.ctl = (const int32_t *)(ws + p.off_ctl);
        sh.start_s = (const int32_t *)(ws + p.off_start_s);
        sh.rowseq = (const int32_t *)(ws + p.off_rowseq);
        sh.ml_s = (float2 *)(ws + p.off_ml_s);
        sh.acc_s = (float *)(ws + p.off_acc_s);
        sh.tc = p.tc ? 1 : 0;
    }
    {
        int32_t Nv = num_seqs, Bv = cache->block_size, ml_v = max_len, HDv = HD, nc = ncnt, NGv = p.NG, Cv = p.C;
        int32_t Gv = G, Hkv = cache->num_kv_heads, NHv = p.NH, tcv = sh.tc;
        void *outp = out;
        const int32_t *planp = sh.plan;
        int32_t *skipp = (int32_t *)sh.skip, *ctlp = (int32_t *)sh.ctl, *start_sp = (int32_t *)sh.start_s;
        int32_t *rowseqp = (int32_t *)sh.rowseq;
        // the plan's words in shared memory when they fit (at most 96 KiB)
        const size_t plan_bytes = sizeof(int32_t) * (7 * (size_t)num_seqs + 16);
        int32_t in_smem = p.shared && plan_bytes <= 96 * 1024 ? 1 : 0;
        const void *pfn = cache->dtype == PA_BF16 ? (const void *)decode_plan_kernel<__nv_bfloat16>
                                                  : (const void *)decode_plan_kernel<float>;
        const size_t psmem = in_smem ? plan_bytes : 0;
        if (psmem > 48 * 1024 &&
            cudaFuncSetAttribute(pfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)psmem) != cudaSuccess)
            return PA_ERR_CUDA;
        void *pargs[] = {&seq_lens, &Nv, &Bv, &ml_v, &HDv, &lens_ws, &cu, &cnt, &nc, &outp, &NGv, &Cv, &start_seq,
                         &err, &planp, &Gv, &Hkv, &NHv, &skipp, &ctlp, &start_sp, &rowseqp, &in_smem, &tcv};
        if (launch_pdl(pfn, dim3(1), dim3(1024), pargs, psmem, s) != cudaSuccess) return PA_ERR_CUDA;
    }

    if (opts && opts->ev_partial_begin && cudaEventRecord((cudaEvent_t)opts->ev_partial_begin, s) != cudaSuccess)
        return PA_ERR_CUDA;
    if (p.kernel == PA_KERNEL_MMA) {
        if (((uintptr_t)k_cache | (uintptr_t)v_cache) % 16 != 0) return PA_ERR_INVALID_ARG;
        // NH-head boxes; one-head boxes for the mma.sync shared-prefix CTAs;
        // one-head, one-panel boxes for the tcgen05 ones
        CUtensorMap tmk, tmv, tmk1, tmv1, tmkp, tmvp;
        if (!encode_cache_map(&tmk, k_cache, cache, p.NH) || !encode_cache_map(&tmv, v_cache, cache, p.NH))
            return PA_ERR_CUDA;
        if (p.shared) {
            if (!encode_cache_map(&tmk1, k_cache, cache, 1) || !encode_cache_map(&tmv1, v_cache, cache, 1))
                return PA_ERR_CUDA;
        } else {
            tmk1 = tmk;
            tmv1 = tmv;
        }
        if (p.tc) {
            if (!encode_cache_map(&tmkp, k_cache, cache, 1, true) || !encode_cache_map(&tmvp, v_cache, cache, 1, true))
                return PA_ERR_CUDA;
        } else {
            tmkp = tmk1;
            tmvp = tmv1;
        }
        const void *fn = mma_kernel_ptr(cache->head_dim, cache->block_size, cache->layout, p.shared);
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem) != cudaSuccess)
            return PA_ERR_CUDA;
        // with a plan, shared_halves logical CTAs (halves) per CTA
        const int halves = mma_halves(cache->head_dim, cache->block_size, p.shared);
        const dim3 grid((p.C + halves - 1) / halves), block(mma_threads(p.NH, halves));
        const __nv_bfloat16 *qb = (const __nv_bfloat16 *)q;
        __nv_bfloat16 *ob = (__nv_bfloat16 *)out;
        int32_t NB = cache->num_blocks, Hk = cache->num_kv_heads, NHv = p.NH, Cv = p.C;
        int32_t Nv = num_seqs, Hv = num_heads, Gv = G, mb = max_blocks_per_seq;
        float sl = scale_log2;
        int32_t local_cu = p.local_cu ? 1 : 0;
        int32_t min_pieces = call_min_pieces(p, opts, num_seqs, cache->block_size, max_len);
        void *args[] = {&tmk, &tmv, &tmk1, &tmv1, &tmkp, &tmvp, &qb, &ob, &block_tables, &mb, &lens_ws, &cu, &Nv, &Hv, &Hk,
                        &Gv, &NB, &NHv, &sl, &Cv, &ml, &acc, &cnt, &start_seq, &err, &sh, &seq_lens, &local_cu,
                        &min_pieces};
        if (launch_pdl(fn, grid, block, args, p.smem, s) != cudaSuccess) return PA_ERR_CUDA;
        if (min_pieces > 0) {
            // one CTA per SM takes the long (sequence, KV head) merges in turn
            const int64_t tasks = (int64_t)num_seqs * Hk;
            const dim3 lgrid((unsigned)std::min<int64_t>(tasks, std::max(num_sms(), 1))), lblock(256);
            void *largs[] = {&ob, &cu, &Nv, &Hv, &Hk, &Gv, &NHv, &Cv, &ml, &acc, &min_pieces};
            const void *lfn = cache->head_dim == 128 ? (const void *)long_merge_kernel<128>
                                                     : (const void *)long_merge_kernel<64>;
            if (launch_pdl(lfn, lgrid, lblock, largs, 0, s) != cudaSuccess) return PA_ERR_CUDA;
        }
        if (p.shared) {
            // one warp per (sequence, KV head) bound: members <= N
            const int64_t warps = (int64_t)num_seqs * Hk;
            const dim3 mgrid((unsigned)((warps + 7) / 8)), mblock(256);
            void *margs[] = {&ob, &cu, &Nv, &Hv, &Hk, &Gv, &NHv, &Cv, &ml, &acc, &sh};
            const void *mfn = cache->head_dim == 128 ? (const void *)shared_merge_kernel<128>
                                                     : (const void *)shared_merge_kernel<64>;
            if (launch_pdl(mfn, mgrid, mblock, margs, 0, s) != cudaSuccess) return PA_ERR_CUDA;
        }
    } else if (p.fma) {
        if (((uintptr_t)k_cache | (uintptr_t)v_cache) % 16 != 0) return PA_ERR_INVALID_ARG;
        CUtensorMap tmk, tmv;
        if (!encode_cache_map(&tmk, k_cache, cache, p.NH) || !encode_cache_map(&tmv, v_cache, cache, p.NH))
            return PA_ERR_CUDA;
        const void *fn = fma_kernel_ptr(cache->dtype, cache->head_dim, G);
        if (!fn) return PA_ERR_UNSUPPORTED;
        if (p.smem > 48 * 1024 &&
            cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem) != cudaSuccess)
            return PA_ERR_CUDA;
        const dim3 grid(p.C), block((p.NH + 1) * 32);
        int32_t NB = cache->num_blocks, Hk = cache->num_kv_heads, NHv = p.NH, Cv = p.C, St = p.stages;
        int32_t Nv = num_seqs, Hv = num_heads, Gv = G, mb = max_blocks_per_seq, Bv = cache->block_size;
        float sl = scale_log2;
        void *args[] = {&tmk, &tmv, &q, &out, &block_tables, &mb, &lens_ws, &cu, &Nv, &Hv, &Hk, &Gv, &Bv, &NB,
                        &NHv, &St, &sl, &Cv, &ml, &acc, &cnt, &start_seq, &err};
        if (launch_pdl(fn, grid, block, args, p.smem, s) != cudaSuccess) return PA_ERR_CUDA;
    } else {
        const void *fn = simt_kernel_ptr(cache->dtype, cache->head_dim, G, cache->layout);
        if (!fn) return PA_ERR_UNSUPPORTED;
        const dim3 grid(p.C), block(p.NH * 32);
        int32_t NB = cache->num_blocks, Hk = cache->num_kv_heads, NHv = p.NH, Cv = p.C;
        int32_t Nv = num_seqs, Hv = num_heads, Gv = G, mb = max_blocks_per_seq, Bv = cache->block_size;
        float sl = scale_log2;
        void *args[] = {&q, &out, &k_cache, &v_cache, &block_tables, &mb, &lens_ws, &cu, &Nv, &Hv, &Hk,
                        &Gv, &Bv, &NB, &NHv, &sl, &Cv, &ml, &acc, &cnt, &start_seq, &err};
        if (launch_pdl(fn, grid, block, args, 0, s) != cudaSuccess) return PA_ERR_CUDA;
    }
    if (opts && opts->ev_partial_end && cudaEventRecord((cudaEvent_t)opts->ev_partial_end, s) != cudaSuccess)
        return PA_ERR_CUDA;

    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
} catch (...) {
    return host_failure();
}

// ------------------------------------------------------------ no-alloc entry
// Scratch of pa_decode_no_alloc: a fixed array in the library's device image
// (one per GPU that loads the library, alive until exit).  Host code must not
// pass `g_decode_scratch` itself to a kernel: on the host that name is only a
// stand-in, so its device address is looked up per device (symbol_address).
static __device__ __align__(256) unsigned char g_decode_scratch[PA_NO_ALLOC_SCRATCH_BYTES];

namespace {
SymbolCache g_scratch_cache;
}  // namespace

extern "C" pa_status_t pa_decode_no_alloc(void *out, const void *q, const void *k_cache, const void *v_cache,
                                          const pa_cache_desc_t *cache, const int32_t *block_tables,
                                          int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs,
                                          int32_t num_heads, float scale, const pa_decode_opts_t *opts,
                                          pa_stream_t stream) try {
    DecodePlan p;
    const pa_status_t st = make_plan(cache, num_seqs, num_heads, opts, true, &p);
    if (st != PA_OK) return st;
    if (p.total > (size_t)PA_NO_ALLOC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
    // Looked up once per device (and again if the device's context changes),
    // with that device current; host code never hands g_decode_scratch itself
    // to a kernel.
    void *scratch = symbol_address(&g_scratch_cache, (const void *)&g_decode_scratch);
    if (!scratch) return PA_ERR_CUDA;
    return pa_decode(out, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                     num_heads, scale, scratch, (size_t)PA_NO_ALLOC_SCRATCH_BYTES, opts, stream);
} catch (...) {
    return host_failure();
}
