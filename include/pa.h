/*
 * pa.h - C ABI of libpa.so: paged-KV decode attention for NVIDIA GB300 (sm_103a).
 *
 * Sources, cited by page title and section:
 *   [nano-vLLM ch.04]  "04 · PagedAttention", nano-vLLM Deep Dive
 *   [PidokuInfra 10]   "10 PagedAttention", PidokuInfra inference engineering
 *   [tokentrails]      "PagedAttention", tokentrails.org serving notes
 *
 * Conventions shared by every call
 * --------------------------------
 * - KV cache layout: pa_cache_desc_t.layout, PA_LAYOUT_ROW by default:
 *   [num_blocks, block_size, num_kv_heads, head_dim] for both K and V,
 *   row-major, head_dim contiguous ([PidokuInfra 10] section 5 "The kernel
 *   side", comment on k_cache).  Token slot s of the pool is block s / B,
 *   offset s % B.  PA_LAYOUT_SPLIT is the vLLM layout (see pa_layout_t).
 * - Element types: PA_F32 (IEEE fp32) or PA_BF16 (bfloat16).  q, k, v, out
 *   and both caches share the cache's element type.  Arithmetic is fp32.
 * - Pointers named "device" must be CUDA device memory (or managed memory)
 *   of the current device; "host" pointers are ordinary host memory.  The
 *   caller owns every buffer.  The library never allocates device memory and
 *   keeps no pointer after a call returns.
 * - Work is enqueued on the caller's stream (NULL = legacy default stream).
 *   No call synchronises, except pa_get_device_error.
 * - Every call checks what the host can see (null pointers, shapes, sizes,
 *   alignment, supported combinations) and returns a status without
 *   launching anything when a check fails.  Nothing aborts the process.
 *   Index errors that only the device can see (a slot or table entry outside
 *   the pool, a length beyond the table) are skipped by the kernels and
 *   recorded in a per-device error word read by pa_get_device_error.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* same type as cudaStream_t / CUstream */
struct CUevent_st;  /* same type as cudaEvent_t / CUevent */
typedef struct CUstream_st *pa_stream_t;
typedef struct CUevent_st *pa_event_t;

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = -1,    /* null pointer, bad shape or size */
    PA_ERR_UNSUPPORTED = -2,    /* valid request with no compiled kernel variant */
    PA_ERR_CUDA = -3,           /* a CUDA runtime/driver call failed */
    PA_ERR_NO_BLOCKS = -4,      /* block manager: the free list cannot satisfy the request */
    PA_ERR_DEVICE_BOUNDS = -5,  /* a kernel met an index outside the pool or the table */
    PA_ERR_DEVICE_TIMEOUT = -6, /* a kernel's bounded wait on an mbarrier ran out */
    PA_ERR_WORKSPACE = -7,      /* the decode workspace is smaller than required */
    PA_ERR_DEVICE_PLAN = -8,    /* a shared-prefix plan does not match its decode call */
    PA_ERR_HOST_MEMORY = -9     /* a host allocation failed (no C++ exception ever leaves a call) */
} pa_status_t;

typedef enum pa_dtype { PA_F32 = 0, PA_BF16 = 1 } pa_dtype_t;

/* Cache layouts.  Both keep each physical block contiguous (B * Hk * D
 * elements per tensor), so block copies and the block-table walk are the same.
 *   PA_LAYOUT_ROW    K and V [NB, B, Hk, D]: one token's Hk * D elements
 *                    contiguous ([PidokuInfra 10] section 5 "The kernel side").
 *   PA_LAYOUT_SPLIT  K [NB, Hk, D/x, B, x] and V [NB, Hk, D, B], x = 16 /
 *                    element bytes (8 for bf16, 4 for fp32): the layout of
 *                    [PidokuInfra 10] section 5 "The layout, more precisely",
 *                    where 16-byte K chunks of consecutive tokens are adjacent
 *                    and V is stored token-minor.  Needs (D * element bytes)
 *                    % 16 == 0. */
typedef enum pa_layout { PA_LAYOUT_ROW = 0, PA_LAYOUT_SPLIT = 1 } pa_layout_t;

/* Shape of the paged KV pool (host struct, read during the call only). */
typedef struct pa_cache_desc {
    int32_t num_blocks;   /* NB: physical blocks in the pool */
    int32_t block_size;   /* B: tokens per block */
    int32_t num_kv_heads; /* Hk */
    int32_t head_dim;     /* D */
    int32_t dtype;        /* pa_dtype_t */
    int32_t layout;       /* pa_layout_t (0 = PA_LAYOUT_ROW) */
} pa_cache_desc_t;

/* Human-readable name of a status code (static string). */
const char *pa_status_string(pa_status_t status);

/* Library version string (static). */
const char *pa_version(void);

/* ------------------------------------------------------------------------
 * pa_reshape_and_cache - paged KV write.
 *
 * For every new token t with slot s = slot_mapping[t]:
 *     k_cache[s / B, s % B, h, :] = k[t, h, :]   and the same for v,
 * for every KV head h, as bit copies (in PA_LAYOUT_SPLIT the same elements
 * go to their split-layout positions).  The slot is the one the block manager
 * gives (physical_block * B + offset; [nano-vLLM ch.04] section 4,
 * Mechanism 3 "The slot mapping"; [tokentrails] Code).
 *
 * k, v          device, [num_tokens, Hk, D], cache element type, contiguous.
 * slot_mapping  device int32 [num_tokens].  A negative slot is padding and is
 *               skipped.  A slot >= NB * B is skipped and recorded as
 *               PA_ERR_DEVICE_BOUNDS.
 * k_cache, v_cache  device, in the descriptor's layout; written in place.
 * Slots must be distinct (two tokens with one slot race).
 * num_tokens == 0 is a no-op.  Pointers must be 16-byte aligned when a
 * token row (Hk * D elements) is a multiple of 16 bytes.
 * ---------------------------------------------------------------------- */
pa_status_t pa_reshape_and_cache(const void *k, const void *v, const int32_t *slot_mapping,
                                 int32_t num_tokens, void *k_cache, void *v_cache,
                                 const pa_cache_desc_t *cache, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_copy_blocks - copy-on-write block copy.
 *
 * For every pair p: block dst = src_dst_pairs[2p + 1] of both caches becomes a
 * bit copy of block src = src_dst_pairs[2p] (all B * Hk * D elements).  This is
 * the copy made before a write into a block whose refcount is above one
 * ([nano-vLLM ch.04] section 6 "Copy-on-write block sharing";
 * [tokentrails] step 4 and Code; [PidokuInfra 10] section 5 "Copy-on-write
 * sharing").
 *
 * src_dst_pairs  device int32 [num_pairs, 2].  Destinations must be distinct
 *                and no destination may also be a source in the same call;
 *                the result then does not depend on pair order.  The host
 *                block manager only emits such pairs.  An id outside [0, NB)
 *                skips the pair and is recorded as PA_ERR_DEVICE_BOUNDS.
 * num_pairs == 0 is a no-op.
 * ---------------------------------------------------------------------- */
pa_status_t pa_copy_blocks(void *k_cache, void *v_cache, const pa_cache_desc_t *cache,
                           const int32_t *src_dst_pairs, int32_t num_pairs, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_decode - single-query decode attention through block tables.
 *
 * For every sequence i and query head h (kv head kh = h / (H / Hk)):
 *     out[i, h, :] = sum_j softmax_j(scale * q[i, h, :] . K_j) V_j,
 * over positions j < seq_lens[i], where K_j, V_j are the cache rows of slot
 * block_tables[i, j / B] * B + j % B ([PidokuInfra 10] section 4
 * PhysicalIndex and section 5 "The kernel side"; [tokentrails] step 3: the
 * same attention as over contiguous memory).  A sequence of length 0 gives
 * an all-zero output.
 *
 * The work is split over a grid of persistent CTAs that share the flattened
 * list of (KV-head group, sequence, block) evenly; a sequence cut between
 * CTAs is merged by a rescaling reduce (running max and sum), done by the CTA
 * whose piece arrives last or, for sequences cut into many pieces when the
 * options carry host_seq_lens, by a second kernel spread over the GPU.  The
 * split depends only on the lengths and the split count, so the same call
 * gives the same bits every time.  A call launches 2 to 3 kernels
 * (pa_decode_launch_count), all on `stream`.
 *
 * out           device [num_seqs, H, D] (written).
 * q             device [num_seqs, H, D].
 * block_tables  device int32 [num_seqs, max_blocks_per_seq]; entries past
 *               ceil(seq_lens[i] / B) are never read.  An entry outside
 *               [0, NB) reads zeros and is recorded as PA_ERR_DEVICE_BOUNDS.
 * seq_lens      device int32 [num_seqs], each in [0, max_blocks_per_seq * B];
 *               an out-of-range length counts as 0 and is recorded.
 * scale         multiplies q . k before the softmax (commonly 1/sqrt(D)).
 * workspace     device scratch of at least pa_decode_workspace_bytes(...)
 *               bytes with the same options, 256-byte aligned; its contents
 *               need no initialisation and are garbage afterwards.  Calls that
 *               share a workspace must be ordered on one stream.
 * opts          optional (NULL = defaults), see pa_decode_opts_t.
 * Requirements: H % Hk == 0, H / Hk <= 8, D in {64, 128, 256} (f32: {64, 128}),
 *               num_seqs * max_blocks_per_seq < 2^31.
 * ---------------------------------------------------------------------- */
typedef enum pa_kernel {
    PA_KERNEL_AUTO = 0, /* tensor-core kernel when it applies, else the CUDA-core one */
    PA_KERNEL_SIMT = 1, /* CUDA-core kernel (fp32 and bf16): blocks staged by TMA in the row layout
                           when the ring fits (D 64/128, bf16 also 256, block sizes up to 256),
                           else one token at a time */
    PA_KERNEL_MMA = 2   /* TMA + tensor-core kernel (bf16, D 64 or 128, B 16 or 32) */
} pa_kernel_t;

typedef struct pa_decode_opts {
    int32_t num_splits; /* persistent CTAs sharing the work; 0 = one wave on this device */
    int32_t kernel;     /* pa_kernel_t */
    pa_event_t ev_partial_begin; /* optional: recorded just before the attention kernel */
    pa_event_t ev_partial_end;   /* optional: recorded just after the attention kernel */
    const int32_t *shared_plan;  /* optional device copy of a pa_shared_plan_build plan (NULL = none) */
    /* Optional HOST copy of seq_lens (num_seqs entries; NULL = none), a hint
     * read on the host during the call.  With it, when some sequence is cut
     * into 8 or more pieces (long contexts), those sequences are merged by a
     * second kernel that spreads their merges over the GPU instead of
     * leaving each to the CTA that finishes last.  The hint only chooses the
     * merge path; the device decides per sequence from seq_lens itself, so a
     * missing or wrong hint never gives a wrong result.  The two paths fold
     * the pieces in different batches (the running maximum is rescaled at
     * different points), so for sequences cut into 8 or more pieces the
     * outputs with and without the hint agree to rounding, not bit for bit;
     * every other output is the same bits either way.  A given call (same
     * arguments, hint included) always gives the same bits. */
    const int32_t *host_seq_lens;
} pa_decode_opts_t;

size_t pa_decode_workspace_bytes(const pa_cache_desc_t *cache, int32_t num_seqs, int32_t num_heads,
                                 const pa_decode_opts_t *opts);

pa_status_t pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                      const pa_cache_desc_t *cache, const int32_t *block_tables,
                      int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs,
                      int32_t num_heads, float scale, void *workspace, size_t workspace_bytes,
                      const pa_decode_opts_t *opts, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_decode_no_alloc - pa_decode for callers that cannot allocate device
 * memory.  (The pages have no counterpart; this is a library convenience.)
 *
 * Some callers have no way to hand pa_decode a workspace: a serving process
 * that reserved nearly all device memory for its KV pool at startup has none
 * left for per-call scratch, a plugin that runs inside a host framework may
 * be forbidden to call cudaMalloc because the framework owns the allocator,
 * and a latency-critical loop cannot afford the device-wide synchronisation
 * that cudaMalloc/cudaFree can imply.  This call takes the same arguments as
 * pa_decode minus the workspace and allocates nothing: its scratch is a
 * fixed array of PA_NO_ALLOC_SCRATCH_BYTES bytes compiled into the library,
 * one copy per GPU that loads it, held until the process exits.
 *
 * - The first call on a device looks up that array's device address (once,
 *   with that device current) and caches it; make this first call before
 *   any stream capture.  The cached address belongs to the device's current
 *   context: if that context changes (after cudaDeviceReset, say), the next
 *   call looks the address up again.
 * - A shape whose workspace (pa_decode_workspace_bytes with the same
 *   options) exceeds PA_NO_ALLOC_SCRATCH_BYTES returns PA_ERR_WORKSPACE and
 *   launches nothing.
 * - Every call on a device shares the one array, and the array keeps the
 *   last call's contents; each call zeroes what it needs zeroed (its arrival
 *   counters) before use.  Calls that can overlap on the GPU (for example
 *   on two streams with no ordering between them) race on the array: order
 *   them on one stream.
 * - No cudaMalloc, cudaFree or allocating library routine is called.
 * ---------------------------------------------------------------------- */
#define PA_NO_ALLOC_SCRATCH_BYTES (16u << 20)

pa_status_t pa_decode_no_alloc(void *out, const void *q, const void *k_cache, const void *v_cache,
                               const pa_cache_desc_t *cache, const int32_t *block_tables,
                               int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs,
                               int32_t num_heads, float scale, const pa_decode_opts_t *opts,
                               pa_stream_t stream);

/* ------------------------------------------------------------------------
 * Shared-prefix decode plan.
 *
 * Sequences forked from one prompt (parallel sampling, beam search) or
 * matched in the prefix cache point at the same physical blocks
 * ([PidokuInfra 10] section 5 "Copy-on-write sharing": one copy of the
 * prompt's blocks with refcount n, and "The relationship to prefix caching";
 * [tokentrails] step 4: shared blocks with reference counts).  Attention over a shared block is the same K and V for every
 * sharer, only the queries differ.  With a plan, pa_decode reads each shared
 * block once and applies it to the query heads of all sharers; each
 * sequence's own blocks are read as before, and the two kinds of partial
 * result are merged by the same rescaling reduce.  The output is the same
 * attention (within the tolerance of a different summation order).
 *
 * pa_shared_plan_build works on the HOST copies of one batch's block tables
 * and lengths (the ones that will be passed to pa_decode).  A group is two or
 * more sequences whose tables start with the same physical block; its shared
 * prefix is the longest run of leading blocks that every member has in
 * common, cut so that every member keeps at least one position of its own
 * after it (P * B < seq_lens[i]).  Groups with P < min_shared_blocks are
 * dropped.  Sharing needs H / Hk in {1, 2, 4, 8}; for other ratios the plan
 * holds no group (info->num_groups = 0) and pa_decode runs as without one.
 *
 * plan       host int32 buffer of at least pa_shared_plan_ints(num_seqs)
 *            elements (written).  Copy it to the device unchanged and pass
 *            its device address in pa_decode_opts_t.shared_plan, with the
 *            same tables, lengths and head counts.  The device checks the
 *            plan's header (sizes, heads per KV head, block size) and that
 *            every member keeps a position of its own; a mismatch records
 *            PA_ERR_DEVICE_PLAN and the affected sequences (or, for a bad
 *            header, all of them) are computed without sharing.  Whether the
 *            members' table entries really are equal is NOT re-checked on the
 *            device: a plan built from other tables gives wrong results.
 * info       optional (NULL allowed): groups, member sequences, shared blocks.
 * Returns PA_ERR_INVALID_ARG for bad sizes or null pointers, or when a
 * length is outside [0, max_blocks_per_seq * B], and PA_ERR_HOST_MEMORY when
 * its host scratch cannot be allocated.
 * The tensor-core kernel uses the plan when Hk is a multiple of 4, the launch
 * has at least 2 CTAs and q is 16-byte aligned; otherwise (and in the
 * CUDA-core kernel) the plan is ignored and the call runs without sharing.
 * In the row layout, plans of 64 query rows per pass (groups of more than 32
 * rows) run their shared blocks as tcgen05 MMAs with the accumulators in
 * tensor memory; such a call's attention CTAs each hold two halves of the
 * usual size (a kernel with tcgen05 instructions is resident once per SM).
 * ---------------------------------------------------------------------- */
typedef struct pa_shared_plan_info {
    int32_t num_groups;    /* groups of >= 2 sequences sharing a prefix */
    int32_t num_members;   /* sequences in groups */
    int64_t shared_blocks; /* sum over groups of their shared prefix blocks */
    int64_t saved_blocks;  /* block reads (per KV head) saved per decode: sum of (members - passes) * P */
} pa_shared_plan_info_t;

size_t pa_shared_plan_ints(int32_t num_seqs);

pa_status_t pa_shared_plan_build(const int32_t *block_tables, int32_t max_blocks_per_seq,
                                 const int32_t *seq_lens, int32_t num_seqs, int32_t block_size,
                                 int32_t num_heads, int32_t num_kv_heads, int32_t min_shared_blocks,
                                 int32_t *plan, size_t plan_ints, pa_shared_plan_info_t *info);

/* Number of CTAs a default (num_splits = 0) decode launch uses on the current
 * device for this shape, or a negative pa_status_t. */
int32_t pa_decode_default_splits(const pa_cache_desc_t *cache, int32_t num_heads,
                                 const pa_decode_opts_t *opts);

/* 1 when a pa_decode call with these arguments (opts->shared_plan set) runs
 * the passes of 64 query rows of its shared prefixes as tcgen05 MMAs with the
 * accumulators in tensor memory, 0 when it would run them on mma.sync (no
 * plan, the split layout, or a tensor-memory budget that does not fit an
 * SM), or a negative pa_status_t.  Plans of 16 or 32 rows per pass always
 * run on mma.sync; the plan's rows per pass are read on the device, so this
 * host-only query does not look at them ("10 PagedAttention" (PidokuInfra),
 * section 5 "The relationship to prefix caching").  Launches nothing. */
int32_t pa_decode_shared_tc(const pa_cache_desc_t *cache, int32_t num_seqs, int32_t num_heads,
                            const pa_decode_opts_t *opts);

/* Kernels that one pa_decode call with these arguments launches on the
 * current device (its plan kernel, the attention kernel and the merge
 * kernels its options bring in), assuming q is 16-byte aligned; or a
 * negative pa_status_t.  Host-only: launches nothing, reads only host memory
 * (opts->host_seq_lens when given). */
int32_t pa_decode_launch_count(const pa_cache_desc_t *cache, int32_t num_seqs, int32_t num_heads,
                               int32_t max_blocks_per_seq, const pa_decode_opts_t *opts);

/* Host mirror of the decode work split (the kernels use the same integer
 * formulas): CTA c of num_splits owns flattened blocks [begin, end) of
 * total_blocks; pa_split_owner gives the CTA that owns block x. */
void pa_split_range(int64_t total_blocks, int32_t num_splits, int32_t c, int64_t *begin,
                    int64_t *end);
int32_t pa_split_owner(int64_t total_blocks, int32_t num_splits, int64_t x);

/* ------------------------------------------------------------------------
 * pa_get_device_error - synchronise `stream`, then read and clear the error
 * word of the current device.  Returns PA_OK, PA_ERR_DEVICE_BOUNDS,
 * PA_ERR_DEVICE_TIMEOUT or PA_ERR_CUDA.
 * ---------------------------------------------------------------------- */
pa_status_t pa_get_device_error(pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_selftest_wait_timeout - check of the kernels' bounded waits.  Launches
 * one thread that waits on a shared-memory mbarrier that nothing arrives at,
 * through the same bounded-wait routine the attention kernel uses, with a
 * limit of limit_ns nanoseconds (0 < limit_ns <= 2e9).  The wait runs out, the
 * kernel records a timeout in the error word and returns; the context stays
 * usable, and the next pa_get_device_error returns PA_ERR_DEVICE_TIMEOUT.
 * (Library self-test; the pages have no counterpart.)
 * ---------------------------------------------------------------------- */
pa_status_t pa_selftest_wait_timeout(int64_t limit_ns, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * Host block manager (all host memory; not thread-safe per handle).
 *
 * A stack of free block ids, a refcount per block and a block table per
 * sequence ([PidokuInfra 10] section 4 "Tiny example"; [nano-vLLM ch.04]
 * sections 4 and 7):
 * - allocation takes the top n ids of the stack in stack order and sets
 *   their refcount to 1; a request the stack cannot meet returns
 *   PA_ERR_NO_BLOCKS and changes nothing;
 * - freeing decrements refcounts and pushes a block back only at 0;
 * - fork copies a table and increments every refcount;
 * - appending a token at position pos allocates a block when pos % B == 0;
 *   otherwise, if the block holding pos has refcount > 1, it is copied first
 *   (copy-on-write: a fresh block replaces it in this table, the old block's
 *   refcount drops by one, and the (src, dst) pair is returned for
 *   pa_copy_blocks), so a shared block is never written in place;
 * - the slot of a token is table[pos / B] * B + pos % B (PhysicalIndex).
 * Sequence ids are assigned 0, 1, 2, ... in creation order.  A call that
 * runs out of host memory returns PA_ERR_HOST_MEMORY; it is the one failure
 * that may leave a partial change behind, so the handle should then be
 * destroyed.
 * ---------------------------------------------------------------------- */
typedef struct pa_bm pa_bm_t;

/* free_order (host, nullable): the initial stack, bottom first, a permutation
 * of [0, num_blocks); the last entry is popped first.  NULL gives the stack
 * num_blocks-1, ..., 1, 0 (block 0 on top).  Returns NULL on bad arguments or
 * when num_blocks * block_size >= 2^31. */
pa_bm_t *pa_bm_create(int32_t num_blocks, int32_t block_size, const int32_t *free_order);
void pa_bm_destroy(pa_bm_t *bm);

pa_status_t pa_bm_new_seq(pa_bm_t *bm, int32_t num_tokens, int32_t *seq_out);
pa_status_t pa_bm_fork(pa_bm_t *bm, int32_t parent, int32_t *child_out);
pa_status_t pa_bm_free_seq(pa_bm_t *bm, int32_t seq);

/* Make room for the next token of seq.  slot_out receives its slot; cow_src /
 * cow_dst receive the copy-on-write pair or -1 when no copy is needed. */
pa_status_t pa_bm_append_token(pa_bm_t *bm, int32_t seq, int32_t *slot_out, int32_t *cow_src,
                               int32_t *cow_dst);

/* Append `count` tokens at once: all or nothing (PA_ERR_NO_BLOCKS leaves the
 * state unchanged).  slots_out [count]; cow_pairs_out [2] receives at most one
 * pair (only the first written block can be shared); *num_pairs_out is 0 or 1. */
pa_status_t pa_bm_append_tokens(pa_bm_t *bm, int32_t seq, int32_t count, int32_t *slots_out,
                                int32_t *cow_pairs_out, int32_t *num_pairs_out);

pa_status_t pa_bm_seq_len(const pa_bm_t *bm, int32_t seq, int32_t *len_out,
                          int32_t *num_blocks_out);
pa_status_t pa_bm_block_table(const pa_bm_t *bm, int32_t seq, int32_t *out, int32_t capacity,
                              int32_t *len_out);
pa_status_t pa_bm_physical_index(const pa_bm_t *bm, int32_t seq, int32_t pos, int32_t *slot_out);
pa_status_t pa_bm_refcount(const pa_bm_t *bm, int32_t block, int32_t *ref_out);
pa_status_t pa_bm_stats(const pa_bm_t *bm, int32_t *free_out, int32_t *used_out,
                        int32_t *shared_out);

/* Prefix caching ([PidokuInfra 10] section 5 "The relationship to prefix
 * caching"; [nano-vLLM ch.04] section 7, hash_to_block).  Creates a sequence
 * for a prompt of num_tokens token ids (host), reusing the blocks of the
 * longest cached prefix made of full blocks (refcount + 1); the other blocks
 * are allocated, and its full blocks are registered.  A block's key is a
 * chained hash: 64-bit FNV-1a over the parent block's key (8 bytes
 * little-endian; 0 for the first block) and the block's token ids (4 bytes
 * little-endian each); a hit also compares the ids.  *num_cached_tokens_out
 * receives the number of leading positions whose K/V already sit in the cache
 * (a multiple of B): the caller writes only positions from there on.  A block
 * leaves the cache when its refcount reaches 0.  PA_ERR_NO_BLOCKS changes
 * nothing.  Only prompt blocks are registered; tokens appended later are not. */
pa_status_t pa_bm_new_seq_cached(pa_bm_t *bm, const int32_t *token_ids, int32_t num_tokens, int32_t *seq_out,
                                 int32_t *num_cached_tokens_out);

/* Slots of positions [first_pos, first_pos + count) of seq (host slots_out). */
pa_status_t pa_bm_slots(const pa_bm_t *bm, int32_t seq, int32_t first_pos, int32_t count, int32_t *slots_out);

/* Prefix-cache counters: registered blocks (evictable ones included), block
 * hits, block lookups. */
pa_status_t pa_bm_cache_stats(const pa_bm_t *bm, int32_t *cached_blocks_out, int64_t *hits_out,
                              int64_t *lookups_out);

/* Retention of prefix-cached blocks (off by default; the eviction of the
 * hands-on exercise of "10 PagedAttention" (PidokuInfra), section 10 A).  On:
 * a registered block whose refcount reaches 0 stays registered as evictable
 * instead of returning to the free list; a later prompt that hits it revives
 * it; an allocation takes free blocks first and then evicts the least
 * recently released evictable blocks, one at a time onto the free stack (the
 * hash entry is dropped).  The blocks one pa_bm_free_seq releases count as
 * released from the sequence's last block to its first, so a prompt loses
 * its tail before its head (prefix matching stops at the first miss).
 * Evictable blocks count as free in pa_bm_stats.  Off: evictable blocks
 * become free, oldest first.  Never fails for a valid bm. */
pa_status_t pa_bm_set_prefix_retention(pa_bm_t *bm, int32_t on);

/* Number of evictable (retained, refcount 0) blocks. */
pa_status_t pa_bm_evictable(const pa_bm_t *bm, int32_t *count_out);

/* Export tables for a decode batch: tables_out [n, max_blocks] (host) padded
 * with -1, lens_out [n]; PA_ERR_INVALID_ARG if a table is longer than
 * max_blocks. */
pa_status_t pa_bm_export(const pa_bm_t *bm, const int32_t *seqs, int32_t n, int32_t max_blocks,
                         int32_t *tables_out, int32_t *lens_out);

/* ------------------------------------------------------------------------
 * Allocation simulator (host only): contiguous max-length reservation
 * against paged blocks under one request stream ([PidokuInfra 10] section 10,
 * exercises B and C; the utilisation contrast of section 2).  One decode step
 * at a time: arrivals join a FIFO queue; the queue head is admitted while it
 * fits (contiguous: prompt + max_new_tokens slots in one interval, first fit;
 * paged: ceil(prompt / B) blocks of the host block manager); every running
 * request (oldest admission first) generates one token, a paged request
 * taking a block when its new token starts one, or, if none is free, being
 * preempted (blocks freed, progress lost, back to the queue front); finished
 * requests free their memory; the step adds held slots (reservations, or
 * blocks x B), used slots (tokens stored) and running requests to the totals.
 * utilization = sum_used / sum_held.
 * arrival_step must be non-decreasing; lengths >= 1; for the contiguous
 * policy output_len <= max_new_tokens.
 * ---------------------------------------------------------------------- */
typedef enum pa_sim_policy { PA_SIM_CONTIGUOUS = 0, PA_SIM_PAGED = 1 } pa_sim_policy_t;

typedef struct pa_sim_config {
    int32_t policy;          /* pa_sim_policy_t */
    int32_t block_size;      /* paged: tokens per block */
    int32_t max_new_tokens;  /* contiguous: reservation = prompt + max_new_tokens */
    int32_t max_steps;       /* step limit */
    int64_t total_slots;     /* token capacity of the pool */
} pa_sim_config_t;

typedef struct pa_sim_result {
    int64_t steps, admitted, completed, preemptions, blocked_steps, peak_running;
    int64_t sum_used, sum_held, sum_running;
    double utilization;      /* sum_used / sum_held */
} pa_sim_result_t;

/* Returns PA_ERR_INVALID_ARG for arguments outside the rules above and
 * PA_ERR_HOST_MEMORY when its host state cannot be allocated. */
pa_status_t pa_sim_run(const pa_sim_config_t *cfg, const int32_t *arrival_step, const int32_t *prompt_len,
                       const int32_t *output_len, int32_t num_requests, pa_sim_result_t *out);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
