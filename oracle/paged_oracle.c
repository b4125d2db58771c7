/*
 * Paged-KV decode oracle: plain, slow, obviously correct CPU code in fp64.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header or constant
 * with the CUDA library: it takes the same raw arrays (pools, block tables,
 * context lengths, slot mapping, q) and computes the textbook definition.
 *
 * Sources (the xserv compare pages):
 *  - "xserv compare phase10...cf1e9e4", crates/xserv-kernels/src/attention.rs,
 *    doc comments of `reshape_and_cache_bf16`, `reshape_and_cache_batched_bf16`
 *    and `paged_decode_attention`: the pool layout
 *    [num_blocks_total, num_kv_heads, block_size, head_dim], the block table
 *    [batch, max_blocks_per_seq] (int32), context lengths [batch] (int32) that
 *    count the token written in this step, scale = 1/sqrt(head_dim), output
 *    [batch, num_q_heads, 1, head_dim].
 *  - "xserv compare phase5...phase9", docs/09-kv-cache.md, section
 *    "After (with cache)": a decode step appends the new K/V to the cache and
 *    attends with one query over all S+1 cached tokens (softmax(q K^T) V).
 *  - "xserv compare phase8...phase13", crates/xserv-model/src/qwen3.rs,
 *    `repeat_kv`: query head h reads KV head h / (num_q_heads/num_kv_heads).
 *
 * Precision: inputs are widened exactly (bf16 -> fp32 -> fp64 by bit shift);
 * every sum, the max, exp and the division run in fp64.  Output is fp64.
 *
 * Functions return 0 on success and a negative code on invalid input; the
 * oracle never clamps anything.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F32 0
#define ORACLE_BF16 1

#define ORACLE_OK 0
#define ORACLE_EINVAL -1
#define ORACLE_ETABLE -2 /* a position beyond the block table's width   */
#define ORACLE_EBLOCK -3 /* a physical block id outside [0, num_blocks)  */
#define ORACLE_ENOMEM -4

/* Exact widening of element idx of a bf16 or fp32 array to double. */
static double widen(const void *base, int64_t idx, int dtype) {
    if (dtype == ORACLE_F32) return (double)((const float *)base)[idx];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static int elem_bytes(int dtype) {
    if (dtype == ORACLE_F32) return 4;
    if (dtype == ORACLE_BF16) return 2;
    return 0;
}

/*
 * Slot resolution for one decode step.  context_lens[b] already counts the
 * token being written (the batched append of reshape_and_cache_batched_bf16
 * takes the length after the step), so the new token's logical position is
 * p = context_lens[b] - 1 and it lives at
 *     slot = block_tables[b][p / block_size] * block_size + p % block_size.
 * A sequence with context_lens[b] <= 0 writes nothing: slot -1.
 */
int oracle_slot_mapping(const int32_t *block_tables, int max_blocks_per_seq,
                        const int32_t *context_lens, int B, int block_size,
                        int64_t num_blocks, int64_t *slot_mapping) {
    if (B < 0 || block_size <= 0 || max_blocks_per_seq < 0) return ORACLE_EINVAL;
    for (int b = 0; b < B; ++b) {
        int32_t n = context_lens[b];
        if (n <= 0) {
            slot_mapping[b] = -1;
            continue;
        }
        int64_t p = (int64_t)n - 1;
        int64_t logical_block = p / block_size;
        if (logical_block >= max_blocks_per_seq) return ORACLE_ETABLE;
        int32_t blk = block_tables[(int64_t)b * max_blocks_per_seq + logical_block];
        if (blk < 0 || blk >= num_blocks) return ORACLE_EBLOCK;
        slot_mapping[b] = (int64_t)blk * block_size + p % block_size;
    }
    return ORACLE_OK;
}

/*
 * KV append: for every token t with slot s = slot_mapping[t] >= 0, copy the
 * head_dim elements of k_new[t, h, :] into k_cache[s / bs, h, s % bs, :]
 * (same for V), for every KV head h.  A pure byte copy.
 * k_new, v_new: [T, Hkv, D]; pools: [num_blocks, Hkv, bs, D].
 */
int oracle_kv_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                     const int64_t *slot_mapping, int T, int Hkv, int D, int block_size,
                     int64_t num_blocks, int dtype) {
    int eb = elem_bytes(dtype);
    if (!eb || T < 0 || Hkv <= 0 || D <= 0 || block_size <= 0) return ORACLE_EINVAL;
    size_t row = (size_t)D * eb;
    for (int t = 0; t < T; ++t) {
        int64_t s = slot_mapping[t];
        if (s < 0) continue;
        int64_t blk = s / block_size, off = s % block_size;
        if (blk >= num_blocks) return ORACLE_EBLOCK;
        for (int h = 0; h < Hkv; ++h) {
            size_t dst = (size_t)(((blk * Hkv + h) * block_size + off) * D) * eb;
            size_t src = (size_t)(((int64_t)t * Hkv + h) * D) * eb;
            memcpy((char *)k_cache + dst, (const char *)k_new + src, row);
            memcpy((char *)v_cache + dst, (const char *)v_new + src, row);
        }
    }
    return ORACLE_OK;
}

/*
 * Paged decode attention, one query token per sequence.
 *
 * For sequence b, query head h, KV head g = h / (Hq / Hkv) and each token
 * t < N = context_lens[b], the key row is found through the block table:
 *     blk = block_tables[b][t / bs],  K_t = k_cache[blk, g, t % bs, :].
 * logit_t = scale * sum_d q[b, h, d] * K_t[d]
 * w_t     = exp(logit_t - max_t' logit_t')
 * out[b, h, :] = sum_t w_t V_t / sum_t w_t
 * A sequence with N <= 0 attends to nothing and its output is zero.
 * q: [B, Hq, D]; out: [B, Hq, D] fp64.
 */
int oracle_paged_decode(const void *q, const void *k_cache, const void *v_cache,
                        const int32_t *block_tables, int max_blocks_per_seq,
                        const int32_t *context_lens, int B, int Hq, int Hkv, int D,
                        int block_size, int64_t num_blocks, double scale, int dtype,
                        double *out, int nthreads) {
    if (!elem_bytes(dtype) || B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || block_size <= 0)
        return ORACLE_EINVAL;
    if (Hq % Hkv != 0) return ORACLE_EINVAL;
    const int group = Hq / Hkv;

    /* Validate every block id that will be read before doing any work. */
    for (int b = 0; b < B; ++b) {
        int32_t n = context_lens[b];
        if (n <= 0) continue;
        int64_t nblk = ((int64_t)n + block_size - 1) / block_size;
        if (nblk > max_blocks_per_seq) return ORACLE_ETABLE;
        for (int64_t i = 0; i < nblk; ++i) {
            int32_t blk = block_tables[(int64_t)b * max_blocks_per_seq + i];
            if (blk < 0 || blk >= num_blocks) return ORACLE_EBLOCK;
        }
    }

    int status = ORACLE_OK;
    if (nthreads <= 0) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int64_t bh = 0; bh < (int64_t)B * Hq; ++bh) {
        int b = (int)(bh / Hq), h = (int)(bh % Hq);
        int g = h / group;
        int32_t n = context_lens[b];
        double *o = out + bh * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (n <= 0) continue;
        double *logit = (double *)malloc(sizeof(double) * (size_t)n);
        if (!logit) {
#pragma omp atomic write
            status = ORACLE_ENOMEM;
            continue;
        }
        const int64_t qbase = bh * D;
        for (int32_t t = 0; t < n; ++t) {
            int64_t blk = block_tables[(int64_t)b * max_blocks_per_seq + t / block_size];
            int64_t kbase = ((blk * Hkv + g) * block_size + t % block_size) * D;
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += widen(q, qbase + d, dtype) * widen(k_cache, kbase + d, dtype);
            logit[t] = scale * dot;
        }
        double mx = logit[0];
        for (int32_t t = 1; t < n; ++t)
            if (logit[t] > mx) mx = logit[t];
        double den = 0.0;
        for (int32_t t = 0; t < n; ++t) {
            double w = exp(logit[t] - mx);
            den += w;
            int64_t blk = block_tables[(int64_t)b * max_blocks_per_seq + t / block_size];
            int64_t vbase = ((blk * Hkv + g) * block_size + t % block_size) * D;
            for (int d = 0; d < D; ++d) o[d] += w * widen(v_cache, vbase + d, dtype);
        }
        for (int d = 0; d < D; ++d) o[d] /= den;
        free(logit);
    }
    return status;
}

/*
 * Paged decode attention with attention sinks and a sliding window (the
 * gpt-oss variant: "xserv compare phase10...cf1e9e4",
 * crates/xserv-kernels/src/attention.rs, paged_decode_attention_sinks and
 * flash_attention_sinks doc comments: a per-query-head sink value folded
 * into the softmax denominator; window_size 0 = full attention, > 0 =
 * sliding window).
 *
 * Readings: the sink s_h is one more logit, in the same units as
 * scale * q.K, that has no value row; a window W > 0 keeps the W most
 * recent tokens, t in [max(0, N - W), N).  sinks may be NULL (no sink);
 * otherwise it holds Hq values of the q dtype.
 *     m   = max(max_t logit_t, s_h)
 *     den = sum_t exp(logit_t - m) + exp(s_h - m)
 *     out[b, h, :] = sum_t exp(logit_t - m) V_t / den
 */
int oracle_paged_decode_sinks(const void *q, const void *k_cache, const void *v_cache,
                              const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *context_lens, int B, int Hq, int Hkv, int D,
                              int block_size, int64_t num_blocks, double scale,
                              const void *sinks, int window, int dtype, double *out,
                              int nthreads) {
    if (!elem_bytes(dtype) || B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || block_size <= 0 ||
        window < 0)
        return ORACLE_EINVAL;
    if (Hq % Hkv != 0) return ORACLE_EINVAL;
    const int group = Hq / Hkv;
    for (int b = 0; b < B; ++b) {
        int32_t n = context_lens[b];
        if (n <= 0) continue;
        int64_t nblk = ((int64_t)n + block_size - 1) / block_size;
        if (nblk > max_blocks_per_seq) return ORACLE_ETABLE;
        for (int64_t i = 0; i < nblk; ++i) {
            int32_t blk = block_tables[(int64_t)b * max_blocks_per_seq + i];
            if (blk < 0 || blk >= num_blocks) return ORACLE_EBLOCK;
        }
    }
    int status = ORACLE_OK;
    if (nthreads <= 0) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int64_t bh = 0; bh < (int64_t)B * Hq; ++bh) {
        int b = (int)(bh / Hq), h = (int)(bh % Hq);
        int kv_head = h / group;
        int32_t n = context_lens[b];
        double *o = out + bh * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (n <= 0) continue;
        int32_t first = (window > 0 && n > window) ? n - window : 0;
        double *lg = (double *)malloc(sizeof(double) * (size_t)(n - first));
        if (!lg) {
#pragma omp atomic write
            status = ORACLE_ENOMEM;
            continue;
        }
        for (int32_t t = first; t < n; ++t) {
            int64_t blk = block_tables[(int64_t)b * max_blocks_per_seq + t / block_size];
            int64_t krow = ((blk * Hkv + kv_head) * block_size + t % block_size) * D;
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += widen(q, bh * D + d, dtype) * widen(k_cache, krow + d, dtype);
            lg[t - first] = scale * dot;
        }
        double top = lg[0];
        for (int32_t i = 1; i < n - first; ++i)
            if (lg[i] > top) top = lg[i];
        double sink = 0.0;
        if (sinks) {
            sink = widen(sinks, h, dtype);
            if (sink > top) top = sink;
        }
        double den = sinks ? exp(sink - top) : 0.0;
        for (int32_t t = first; t < n; ++t) {
            double wt = exp(lg[t - first] - top);
            den += wt;
            int64_t blk = block_tables[(int64_t)b * max_blocks_per_seq + t / block_size];
            int64_t vrow = ((blk * Hkv + kv_head) * block_size + t % block_size) * D;
            for (int d = 0; d < D; ++d) o[d] += wt * widen(v_cache, vrow + d, dtype);
        }
        for (int d = 0; d < D; ++d) o[d] /= den;
        free(lg);
    }
    return status;
}

/*
 * KV swap: copy whole KV blocks between two pools (the pages' CPU swap-out /
 * swap-in of paged KV blocks to pinned host memory: "xserv compare
 * phase10...cf1e9e4", README, --swap-space-gb).  For every pair
 * i < n of mapping ([n][2] int64: source block, destination block) with both
 * ids >= 0, the block_bytes bytes of source block s in src_k (and src_v) are
 * copied to destination block d of dst_k (and dst_v).  A pair with a
 * negative id is skipped; an id at or past its pool's size is an error.
 * Destinations are expected to be distinct.
 */
int oracle_kv_swap(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                   const int64_t *mapping, int n, int64_t block_bytes, int64_t src_blocks,
                   int64_t dst_blocks) {
    if (n < 0 || block_bytes <= 0) return ORACLE_EINVAL;
    for (int i = 0; i < n; ++i) {
        int64_t s = mapping[2 * i], d = mapping[2 * i + 1];
        if (s < 0 || d < 0) continue;
        if (s >= src_blocks || d >= dst_blocks) return ORACLE_EBLOCK;
        memcpy((char *)dst_k + d * block_bytes, (const char *)src_k + s * block_bytes,
               (size_t)block_bytes);
        memcpy((char *)dst_v + d * block_bytes, (const char *)src_v + s * block_bytes,
               (size_t)block_bytes);
    }
    return ORACLE_OK;
}

/*
 * Block allocation for one decode step (the pages' PagedKVCache hands each
 * sequence a new physical block when its next token starts a page:
 * "xserv compare phase10...cf1e9e4", bench-qwen3.rs / gpt-oss drivers,
 * PagedKVCache::new_tp(.., total_blocks, .., max_blocks_per_seq, ..),
 * register_sequence, free_sequence, seq_len; the struct's body is not on the
 * pages).  Reading: a free list is a stack of block ids free_stack[0, top).
 * For every active sequence b (context_lens[b] >= 0; -1 = no sequence):
 * the new token's position is p = context_lens[b]; if p % bs == 0 it starts
 * page p / bs, which takes the block on top of the stack.  Then
 * context_lens[b] = p + 1.  A sequence whose page would lie past the table
 * (failed[b] = 2) or that finds the stack empty (failed[b] = 1) is left
 * unchanged.  Sequences are served in index order; the device kernel may
 * hand the popped blocks out in another order.
 */
int oracle_block_alloc_decode(int32_t *block_tables, int max_blocks_per_seq, int32_t *context_lens,
                              int B, int block_size, const int32_t *free_stack, int32_t *free_top,
                              int32_t *failed) {
    if (B < 0 || block_size <= 0 || max_blocks_per_seq < 0 || *free_top < 0) return ORACLE_EINVAL;
    for (int b = 0; b < B; ++b) {
        failed[b] = 0;
        int32_t p = context_lens[b];
        if (p < 0) continue;
        int32_t page = p / block_size;
        if (page >= max_blocks_per_seq) {
            failed[b] = 2;
            continue;
        }
        if (p % block_size == 0) {
            if (*free_top == 0) {
                failed[b] = 1;
                continue;
            }
            *free_top -= 1;
            block_tables[(int64_t)b * max_blocks_per_seq + page] = free_stack[*free_top];
        }
        context_lens[b] = p + 1;
    }
    return ORACLE_OK;
}

/*
 * Release sequences (PagedKVCache::free_sequence): every block of the listed
 * sequences, pages 0 .. ceil(len / bs) - 1 in order, is pushed on the free
 * stack; their table rows become -1 and their lengths -1 (no sequence).
 */
int oracle_block_free(const int32_t *seq_ids, int n, int32_t *block_tables, int max_blocks_per_seq,
                      int32_t *context_lens, int block_size, int32_t *free_stack,
                      int32_t *free_top, int64_t stack_capacity) {
    if (n < 0 || block_size <= 0) return ORACLE_EINVAL;
    for (int i = 0; i < n; ++i) {
        int32_t b = seq_ids[i];
        int32_t len = context_lens[b];
        int32_t pages = len > 0 ? (len + block_size - 1) / block_size : 0;
        if (pages > max_blocks_per_seq) return ORACLE_ETABLE;
        for (int32_t pg = 0; pg < pages; ++pg) {
            if (*free_top >= stack_capacity) return ORACLE_EINVAL;
            free_stack[*free_top] = block_tables[(int64_t)b * max_blocks_per_seq + pg];
            *free_top += 1;
        }
        for (int32_t pg = 0; pg < max_blocks_per_seq; ++pg)
            block_tables[(int64_t)b * max_blocks_per_seq + pg] = -1;
        context_lens[b] = -1;
    }
    return ORACLE_OK;
}

/*
 * Prefill append for one sequence ("xserv compare phase10...cf1e9e4",
 * attention.rs, reshape_and_cache_bf16: k_src/v_src are [num_kv_heads,
 * num_tokens, head_dim]; token i goes to position start_pos + i of the
 * sequence whose block list is block_ids, which must hold at least
 * ceil((start_pos + num_tokens) / block_size) ids):
 *     pool[block_ids[(start + i) / bs], h, (start + i) % bs, :] = src[h, i, :]
 */
int oracle_prefill_append(const void *k_src, const void *v_src, void *k_cache, void *v_cache,
                          const int32_t *block_ids, int n_ids, int T, int Hkv, int D,
                          int block_size, int64_t num_blocks, int start_pos, int dtype) {
    int eb = elem_bytes(dtype);
    if (!eb || T < 0 || Hkv <= 0 || D <= 0 || block_size <= 0 || start_pos < 0)
        return ORACLE_EINVAL;
    size_t row = (size_t)D * eb;
    for (int i = 0; i < T; ++i) {
        int64_t pos = (int64_t)start_pos + i;
        if (pos / block_size >= n_ids) return ORACLE_ETABLE;
        int64_t blk = block_ids[pos / block_size];
        if (blk < 0 || blk >= num_blocks) return ORACLE_EBLOCK;
        for (int h = 0; h < Hkv; ++h) {
            size_t dst = (size_t)(((blk * Hkv + h) * block_size + pos % block_size) * D) * eb;
            size_t src = (size_t)(((int64_t)h * T + i) * D) * eb;
            memcpy((char *)k_cache + dst, (const char *)k_src + src, row);
            memcpy((char *)v_cache + dst, (const char *)v_src + src, row);
        }
    }
    return ORACLE_OK;
}

/*
 * Chunked prefill attention over the paged cache for one sequence: query
 * token i (q[i, h, :], q is [T, Hq, D]) sits at position start_pos + i and
 * attends causally to every cached token t <= start_pos + i, keys and values
 * gathered through block_ids, query head h reading KV head h / (Hq / Hkv)
 * (the naive attention with a causal mask offset by the cached prefix:
 * "xserv compare phase10...cf1e9e4", attention.rs, attention /
 * apply_causal_mask(offset); flash_attention for q_len > 1).
 *     out[i, h, :] = sum_{t <= start+i} softmax_t(scale q[i,h,:].K_t) V_t
 */
int oracle_paged_prefill(const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_ids, int n_ids, int T, int start_pos, int Hq,
                         int Hkv, int D, int block_size, int64_t num_blocks, double scale,
                         int dtype, double *out, int nthreads) {
    if (!elem_bytes(dtype) || T < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || block_size <= 0 ||
        start_pos < 0 || Hq % Hkv != 0)
        return ORACLE_EINVAL;
    const int group = Hq / Hkv;
    const int64_t total = (int64_t)start_pos + T;
    const int64_t pages = (total + block_size - 1) / block_size;
    if (pages > n_ids) return ORACLE_ETABLE;
    for (int64_t i = 0; i < pages; ++i)
        if (block_ids[i] < 0 || block_ids[i] >= num_blocks) return ORACLE_EBLOCK;
    int status = ORACLE_OK;
    if (nthreads <= 0) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int64_t ih = 0; ih < (int64_t)T * Hq; ++ih) {
        int i = (int)(ih / Hq), h = (int)(ih % Hq);
        int kvh = h / group;
        int64_t last = (int64_t)start_pos + i;  /* attends to tokens 0..last */
        double *o = out + ih * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        double *sc = (double *)malloc(sizeof(double) * (size_t)(last + 1));
        if (!sc) {
#pragma omp atomic write
            status = ORACLE_ENOMEM;
            continue;
        }
        for (int64_t t = 0; t <= last; ++t) {
            int64_t blk = block_ids[t / block_size];
            int64_t kr = ((blk * Hkv + kvh) * block_size + t % block_size) * D;
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += widen(q, ih * D + d, dtype) * widen(k_cache, kr + d, dtype);
            sc[t] = scale * acc;
        }
        double mval = sc[0];
        for (int64_t t = 1; t <= last; ++t) mval = sc[t] > mval ? sc[t] : mval;
        double z = 0.0;
        for (int64_t t = 0; t <= last; ++t) {
            double e = exp(sc[t] - mval);
            z += e;
            int64_t blk = block_ids[t / block_size];
            int64_t vr = ((blk * Hkv + kvh) * block_size + t % block_size) * D;
            for (int d = 0; d < D; ++d) o[d] += e * widen(v_cache, vr + d, dtype);
        }
        for (int d = 0; d < D; ++d) o[d] /= z;
        free(sc);
    }
    return status;
}

/* Number of threads an OpenMP parallel region would use (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
