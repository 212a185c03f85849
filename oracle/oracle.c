/*
 * Plain CPU oracle for the paged-KV decode path.
 *
 * Sources, cited by page title and section:
 *   [nano-vLLM ch.04]  "04 · PagedAttention", nano-vLLM Deep Dive
 *   [PidokuInfra 10]   "10 PagedAttention", PidokuInfra inference engineering
 *   [tokentrails]      "PagedAttention", tokentrails.org serving notes
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes
 * or calls this file; only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark load it.  It shares no code, header, table
 * or constant with the CUDA path.
 *
 * Every routine is the definition written out with plain loops, in the order
 * the pages state it, with no blocking, fusion or reordering:
 *
 *   - physical index   [PidokuInfra 10] section 4 "Tiny example", PhysicalIndex:
 *                      slot = table[pos / B] * B + pos % B; the same rule as
 *                      [nano-vLLM ch.04] section 4, Mechanism 3 "The slot
 *                      mapping" (physical_block_id * block_size + offset).
 *   - cache write      [nano-vLLM ch.04] section 4, Mechanism 3: each new
 *                      token's K and V go to the cache row named by its slot;
 *                      [tokentrails] Code: the token is stored at
 *                      (block, t mod BLOCK).
 *   - block copy       [tokentrails] step 4 and Code (copy_block);
 *                      [nano-vLLM ch.04] section 6 "Copy-on-write block
 *                      sharing": the whole shared block is duplicated.
 *   - decode attention [PidokuInfra 10] section 5 "The kernel side" (walk of
 *                      ceil(ctx / B) blocks through the table, cache layout
 *                      [num_blocks, block_size, num_kv_heads, head_dim]) and
 *                      [tokentrails] step 3 "Attention across blocks": the
 *                      same attention as over contiguous memory, i.e.
 *                      out = softmax(scale * q K^T) V, computed in fp64.
 *
 * Readings where the pages are silent:
 *   - grouped-query heads: query head h reads KV head h / (H / Hk);
 *   - a sequence of length 0 yields an all-zero output;
 *   - a negative slot in the slot mapping is padding and is skipped;
 *   - the softmax subtracts the maximum score before exponentiating (the
 *     result is the same softmax, this only keeps exp() in range).
 *
 * Element types: 0 = IEEE fp32, 1 = bfloat16 (upper 16 bits of an fp32).
 * bfloat16 values are widened exactly (bits << 16) before any arithmetic.
 *
 * Cache layouts (the element of token slot blk * B + off, KV head h, dim d):
 *   0  block rows  K and V [num_blocks, B, Hk, D]   ([PidokuInfra 10]
 *                  section 5 "The kernel side", comment on k_cache)
 *   1  split       K [num_blocks, Hk, D/x, B, x], V [num_blocks, Hk, D, B],
 *                  x = 16 / element bytes ([PidokuInfra 10] section 5
 *                  "The layout, more precisely")
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1

static int elem_bytes(int dtype) { return dtype == ORC_F32 ? 4 : 2; }

/* Exact widening of one stored element to double. */
static double load_as_double(const void *base, int dtype, int64_t index) {
    float f;
    if (dtype == ORC_F32) {
        memcpy(&f, (const char *)base + index * 4, 4);
    } else {
        uint16_t h;
        uint32_t u;
        memcpy(&h, (const char *)base + index * 2, 2);
        u = ((uint32_t)h) << 16;
        memcpy(&f, &u, 4);
    }
    return (double)f;
}

/* Element offsets of (blk, off, h, d) in the K and the V cache. */
static int64_t k_offset(int layout, int64_t blk, int64_t off, int64_t h, int64_t d, int64_t B, int64_t Hk,
                        int64_t D, int64_t x) {
    if (layout == 1) return (((blk * Hk + h) * (D / x) + d / x) * B + off) * x + d % x;
    return ((blk * B + off) * Hk + h) * D + d;
}

static int64_t v_offset(int layout, int64_t blk, int64_t off, int64_t h, int64_t d, int64_t B, int64_t Hk,
                        int64_t D) {
    if (layout == 1) return ((blk * Hk + h) * D + d) * B + off;
    return ((blk * B + off) * Hk + h) * D + d;
}

/* PhysicalIndex: where token `pos` of a sequence lives in the pool. */
int64_t orc_physical_index(const int32_t *table, int32_t block_size, int64_t pos) {
    int64_t logical_block = pos / block_size;
    int64_t offset = pos % block_size;
    return (int64_t)table[logical_block] * block_size + offset;
}

/* Slot mapping for a batch of new tokens: token t belongs to sequence
 * seq_ids[t] at position positions[t].  Tables are [num_seqs, max_blocks]. */
void orc_slot_mapping(const int32_t *tables, int32_t max_blocks, const int32_t *seq_ids,
                      const int32_t *positions, int32_t num_tokens, int32_t block_size,
                      int64_t *slots_out) {
    for (int32_t t = 0; t < num_tokens; ++t) {
        const int32_t *table = tables + (int64_t)seq_ids[t] * max_blocks;
        slots_out[t] = orc_physical_index(table, block_size, positions[t]);
    }
}

/* Cache write: k_cache[s / B, s % B, h, :] = k[t, h, :] (and the same for v)
 * for every token t whose slot s is not negative.  Returns the number of
 * tokens whose slot lay beyond the pool (those are skipped). */
int32_t orc_reshape_and_cache(const void *k, const void *v, const int64_t *slots,
                              int32_t num_tokens, void *k_cache, void *v_cache,
                              int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                              int32_t head_dim, int32_t dtype, int32_t layout) {
    int32_t out_of_range = 0;
    int64_t eb = elem_bytes(dtype);
    int64_t x = 16 / eb;
    for (int32_t t = 0; t < num_tokens; ++t) {
        int64_t s = slots[t];
        if (s < 0) continue;
        if (s >= (int64_t)num_blocks * block_size) {
            out_of_range++;
            continue;
        }
        int64_t blk = s / block_size;
        int64_t off = s % block_size;
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            for (int32_t d = 0; d < head_dim; ++d) {
                int64_t src = ((int64_t)t * num_kv_heads + h) * head_dim + d;
                int64_t kd = k_offset(layout, blk, off, h, d, block_size, num_kv_heads, head_dim, x);
                int64_t vd = v_offset(layout, blk, off, h, d, block_size, num_kv_heads, head_dim);
                memcpy((char *)k_cache + kd * eb, (const char *)k + src * eb, eb);
                memcpy((char *)v_cache + vd * eb, (const char *)v + src * eb, eb);
            }
        }
    }
    return out_of_range;
}

/* Copy-on-write block copy: for each pair (src, dst) the whole physical block
 * dst becomes a byte copy of block src, in K and in V. */
void orc_copy_blocks(void *k_cache, void *v_cache, int64_t block_bytes, const int32_t *pairs,
                     int32_t num_pairs) {
    for (int32_t p = 0; p < num_pairs; ++p) {
        int64_t src = pairs[2 * p];
        int64_t dst = pairs[2 * p + 1];
        memcpy((char *)k_cache + dst * block_bytes, (const char *)k_cache + src * block_bytes,
               block_bytes);
        memcpy((char *)v_cache + dst * block_bytes, (const char *)v_cache + src * block_bytes,
               block_bytes);
    }
}

typedef struct {
    double *out;
    int dtype;
    const void *q, *k_cache, *v_cache;
    int32_t num_blocks, block_size, num_kv_heads, head_dim, layout;
    const int32_t *tables;
    int32_t max_blocks;
    const int32_t *seq_lens;
    int32_t num_seqs, num_heads;
    double scale;
    const int32_t *pairs; /* [n, 2] of (seq, head), or NULL for every pair */
    int32_t num_pairs;
    int32_t stride, first;
    int32_t status;
} decode_job;

/* One (sequence, query head): out = softmax(scale * q K^T) V over the
 * sequence's tokens, each token found through the block table. */
static int32_t decode_one(const decode_job *j, int32_t seq, int32_t head, double *scores) {
    const int32_t D = j->head_dim;
    const int32_t group = j->num_heads / j->num_kv_heads;
    const int32_t kv_head = head / group;
    const int32_t L = j->seq_lens[seq];
    const int32_t *table = j->tables + (int64_t)seq * j->max_blocks;
    double *o = j->out + ((int64_t)seq * j->num_heads + head) * D;
    int64_t qbase = ((int64_t)seq * j->num_heads + head) * D;

    for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
    if (L == 0) return 0;
    if (L < 0 || L > (int64_t)j->max_blocks * j->block_size) return -1;

    /* scores s_j = scale * sum_d q[d] * K_j[d] */
    for (int32_t pos = 0; pos < L; ++pos) {
        int64_t blk_id = table[pos / j->block_size];
        if (blk_id < 0 || blk_id >= j->num_blocks) return -1;
        int64_t slot = orc_physical_index(table, j->block_size, pos);
        int64_t blk = slot / j->block_size;
        int64_t off = slot % j->block_size;
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d)
            dot += load_as_double(j->q, j->dtype, qbase + d) *
                   load_as_double(j->k_cache, j->dtype,
                                  k_offset(j->layout, blk, off, kv_head, d, j->block_size,
                                           j->num_kv_heads, D, 16 / elem_bytes(j->dtype)));
        scores[pos] = j->scale * dot;
    }
    /* softmax weights */
    double m = scores[0];
    for (int32_t pos = 1; pos < L; ++pos)
        if (scores[pos] > m) m = scores[pos];
    double z = 0.0;
    for (int32_t pos = 0; pos < L; ++pos) {
        scores[pos] = exp(scores[pos] - m);
        z += scores[pos];
    }
    /* out = sum_j w_j V_j */
    for (int32_t pos = 0; pos < L; ++pos) {
        int64_t slot = orc_physical_index(table, j->block_size, pos);
        int64_t blk = slot / j->block_size;
        int64_t off = slot % j->block_size;
        double w = scores[pos] / z;
        for (int32_t d = 0; d < D; ++d)
            o[d] += w * load_as_double(j->v_cache, j->dtype,
                                       v_offset(j->layout, blk, off, kv_head, d, j->block_size,
                                                j->num_kv_heads, D));
    }
    return 0;
}

static void *decode_worker(void *arg) {
    decode_job *j = (decode_job *)arg;
    int32_t total = j->pairs ? j->num_pairs : j->num_seqs * j->num_heads;
    double *scores = (double *)malloc(sizeof(double) * ((size_t)j->max_blocks * j->block_size + 1));
    if (!scores) {
        j->status = -2;
        return NULL;
    }
    for (int32_t idx = j->first; idx < total; idx += j->stride) {
        int32_t seq, head;
        if (j->pairs) {
            seq = j->pairs[2 * idx];
            head = j->pairs[2 * idx + 1];
        } else {
            seq = idx / j->num_heads;
            head = idx % j->num_heads;
        }
        if (decode_one(j, seq, head, scores) != 0) j->status = -1;
    }
    free(scores);
    return NULL;
}

/* Decode attention for the listed (seq, head) pairs (all pairs when `pairs`
 * is NULL), split over `num_threads` POSIX threads.  out is fp64
 * [num_seqs, num_heads, head_dim]; entries of unlisted pairs are untouched.
 * Returns 0, or -1 when a length or a table entry is out of range. */
int32_t orc_decode(double *out, int32_t dtype, const void *q, const void *k_cache,
                   const void *v_cache, int32_t num_blocks, int32_t block_size,
                   int32_t num_kv_heads, int32_t head_dim, const int32_t *tables,
                   int32_t max_blocks, const int32_t *seq_lens, int32_t num_seqs,
                   int32_t num_heads, double scale, const int32_t *pairs, int32_t num_pairs,
                   int32_t num_threads, int32_t layout) {
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return -1;
    if (layout == 1 && head_dim % (16 / elem_bytes(dtype)) != 0) return -1;
    if (num_threads < 1) num_threads = 1;
    decode_job base;
    base.out = out;
    base.dtype = dtype;
    base.q = q;
    base.k_cache = k_cache;
    base.v_cache = v_cache;
    base.num_blocks = num_blocks;
    base.block_size = block_size;
    base.num_kv_heads = num_kv_heads;
    base.head_dim = head_dim;
    base.layout = layout;
    base.tables = tables;
    base.max_blocks = max_blocks;
    base.seq_lens = seq_lens;
    base.num_seqs = num_seqs;
    base.num_heads = num_heads;
    base.scale = scale;
    base.pairs = pairs;
    base.num_pairs = num_pairs;
    base.stride = num_threads;
    base.status = 0;

    decode_job *jobs = (decode_job *)malloc(sizeof(decode_job) * num_threads);
    pthread_t *threads = (pthread_t *)malloc(sizeof(pthread_t) * num_threads);
    if (!jobs || !threads) {
        free(jobs);
        free(threads);
        return -2;
    }
    for (int32_t t = 0; t < num_threads; ++t) {
        jobs[t] = base;
        jobs[t].first = t;
    }
    for (int32_t t = 1; t < num_threads; ++t) pthread_create(&threads[t], NULL, decode_worker, &jobs[t]);
    decode_worker(&jobs[0]);
    for (int32_t t = 1; t < num_threads; ++t) pthread_join(threads[t], NULL);
    int32_t status = 0;
    for (int32_t t = 0; t < num_threads; ++t)
        if (jobs[t].status != 0) status = jobs[t].status;
    free(jobs);
    free(threads);
    return status;
}
