/*
 * xs_paged.h - C ABI of libxs_paged, the GB300 (sm_103a) decode step over a
 * paged KV cache: write each running sequence's new K/V token into its page,
 * then attend with that sequence's single query token over all of its pages.
 *
 * The operations follow the xserv inference engine's description of its
 * paged KV cache ("xserv compare phase10...cf1e9e4",
 * crates/xserv-kernels/src/attention.rs, the doc comments and extern
 * signatures of reshape_and_cache_bf16, reshape_and_cache_batched_bf16 and
 * paged_decode_attention) and of decode attention over a cache
 * ("xserv compare phase5...phase9", docs/09-kv-cache.md, "After (with
 * cache)").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every array argument is a DEVICE pointer owned by the caller.  The
 *    library never allocates or frees memory; scratch space (split-K
 *    partials) is passed in by the caller, except for
 *    xs_paged_decode_noalloc, which uses one fixed array the library
 *    reserves on each device when it is loaded.
 *  - Work is enqueued asynchronously on the caller's stream; a call returns
 *    once the launch is queued.  Nothing synchronises the device.
 *  - Return value: XS_OK (0) or a negative XS_E* code.  Host-visible
 *    argument errors are detected before anything is launched.  A launch
 *    failure reports XS_ELAUNCH (the CUDA error is left for
 *    cudaGetLastError/cudaPeekAtLastError to inspect).
 *  - Device-side problems (a block id outside the pool, a context length
 *    beyond the block table) are never trapped: the kernel redirects the
 *    access to a valid address or skips it, and ORs an XS_FLAG_* bit into
 *    *err_flag when err_flag is not NULL.  Results are then unspecified for
 *    the affected sequence only.
 *  - Layouts (all row-major, contiguous):
 *      KV pool      [num_blocks, Hkv, block_size, D]   element (blk,h,o,d) at
 *                   ((blk*Hkv + h)*block_size + o)*D + d
 *      block_tables int32 [B, max_blocks_per_seq]; row b lists sequence b's
 *                   physical blocks in logical order; entries past the last
 *                   page the sequence uses are never read
 *      context_lens int32 [B]; number of tokens of sequence b INCLUDING the
 *                   token written this step (the same meaning as the
 *                   per-sequence lengths of the pages' batched append)
 *      q, out       [B, Hq, D] (the pages' [batch, num_q_heads, 1, head_dim])
 *      k_new, v_new [T, Hkv, D], one row per written token
 *  - Query head h reads KV head h / (Hq/Hkv) ("xserv compare
 *    phase8...phase13", crates/xserv-model/src/qwen3.rs, repeat_kv).
 *  - dtype: XS_F32 or XS_BF16; q, k_new, v_new, pools and out share it.
 *    Arithmetic is fp32; bf16 outputs are rounded to nearest-even.
 *  - Supported: block_size 16, D in {64, 128}, Hq/Hkv in {1, 2, 4, 8}.
 *    Pointers to pools, q, k_new, v_new, out and partials must be 16-byte
 *    aligned.
 */
#ifndef XS_PAGED_H
#define XS_PAGED_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* dtype codes */
#define XS_F32 0
#define XS_BF16 1

/* return codes */
#define XS_OK 0
#define XS_ENULL -1        /* a required pointer is NULL                      */
#define XS_ESHAPE -2       /* a size is negative, zero where it must not be,
                              Hq % Hkv != 0, or sizes are inconsistent        */
#define XS_EDTYPE -3       /* dtype is not XS_F32 / XS_BF16                   */
#define XS_EALIGN -4       /* a pointer is not 16-byte aligned                */
#define XS_EUNSUPPORTED -5 /* block_size != 16, D not in {64,128},
                              Hq/Hkv not in {1,2,4,8}                         */
#define XS_EWORKSPACE -6   /* partials missing or too small for the split    */
#define XS_ELAUNCH -7      /* a kernel launch failed                          */
#define XS_EDEVICE -8      /* querying the current device failed              */
#define XS_ESCRATCH -9     /* the split needs more than the library's fixed
                              scratch array holds (xs_paged_decode_noalloc)   */

/* bits ORed into *err_flag by the kernels */
#define XS_FLAG_BAD_BLOCK 1 /* a block id outside [0, num_blocks) was met;
                               block 0 was read instead / the write skipped  */
#define XS_FLAG_BAD_LEN 2   /* context_lens[b] > max_blocks_per_seq*block_size;
                               the length was clamped to that bound          */
#define XS_FLAG_BAD_SLOT 4  /* slot_mapping[t] beyond the pool; write skipped */
#define XS_FLAG_TIMEOUT 8   /* a bounded wait for staged data gave up; the
                               kernel drained its copies and returned        */
#define XS_FLAG_CONFIG 16   /* internal: a launch got less shared memory than
                               its batch needs; the kernel did nothing       */
#define XS_FLAG_POOL_EMPTY 32 /* the free-block stack was empty (allocation)
                                 or full (release); that sequence was left
                                 as it was                                    */
#define XS_FLAG_BOUNDS 64   /* only in the debug build (libxs_paged_debug.so,
                               compiled with -DXS_DEBUG_BOUNDS): a computed
                               global-memory index fell outside its buffer;
                               the access was skipped.  Release builds never
                               set it (the checks compile away).              */

/*
 * xs_slot_mapping - where each sequence's new token goes (one decode step).
 *
 * For every b with n = context_lens[b] > 0 the new token's logical position
 * is p = n - 1 and its slot is
 *     slot_mapping[b] = block_tables[b][p / block_size] * block_size
 *                       + p % block_size;
 * sequences with n <= 0 get -1 (nothing to write).  The pages pass
 * block_tables + kv_lens to their batched append
 * ("xserv compare phase10...cf1e9e4", attention.rs,
 * reshape_and_cache_batched_bf16); this call exposes that address step.
 *
 * block_tables int32 [B, max_blocks_per_seq]; context_lens int32 [B];
 * slot_mapping int64 [B] (output).  A position beyond the table width sets
 * XS_FLAG_BAD_LEN and a block id outside [0, num_blocks) sets
 * XS_FLAG_BAD_BLOCK; both write slot -1.
 */
int xs_slot_mapping(const int32_t *block_tables, int max_blocks_per_seq,
                    const int32_t *context_lens, int B, int block_size, int64_t num_blocks,
                    int64_t *slot_mapping, int *err_flag, cudaStream_t stream);

/*
 * xs_kv_append - scatter T new K/V rows into their pool slots.
 *
 *     k_cache[s / bs, h, s % bs, :] = k_new[t, h, :]   (same for V)
 * for every t < T with s = slot_mapping[t] >= 0 and every KV head h; the
 * copy is bit-exact.  Follows the pool layout and scatter of
 * reshape_and_cache_bf16 / reshape_and_cache_batched_bf16
 * ("xserv compare phase10...cf1e9e4", attention.rs); here the destination
 * comes from a precomputed slot_mapping so one call serves any token mix.
 *
 * k_new, v_new [T, Hkv, D]; k_cache, v_cache [num_blocks, Hkv, bs, D];
 * slot_mapping int64 [T].  Slots at or beyond num_blocks*bs set
 * XS_FLAG_BAD_SLOT and are skipped.  Tokens must have distinct slots.
 */
int xs_kv_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                 const int64_t *slot_mapping, int T, int Hkv, int D, int block_size,
                 int64_t num_blocks, int dtype, int *err_flag, cudaStream_t stream);

/*
 * xs_kv_append_paged - the decode-step append with slot resolution fused in:
 * writes k_new[b] / v_new[b] ([B, Hkv, D]) at position context_lens[b] - 1
 * of sequence b, located through block_tables exactly as xs_slot_mapping
 * does.  This is the pages' reshape_and_cache_batched_bf16 ("xserv compare
 * phase10...cf1e9e4", attention.rs), which reads the very block table the
 * attention call reads.  Errors as xs_slot_mapping; bad entries are skipped.
 */
int xs_kv_append_paged(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                       const int32_t *block_tables, int max_blocks_per_seq,
                       const int32_t *context_lens, int B, int Hkv, int D, int block_size,
                       int64_t num_blocks, int dtype, int *err_flag, cudaStream_t stream);

/*
 * xs_prefill_append - write a prefill chunk into one sequence's pages (the
 * pages' reshape_and_cache_bf16, "xserv compare phase10...cf1e9e4",
 * attention.rs): k_src, v_src are [Hkv, T, D] (the pages' layout); row i
 * goes to position start_pos + i, i.e. block block_ids[(start_pos + i) / bs],
 * offset (start_pos + i) % bs.  block_ids (int32 [n_ids], device) is the
 * sequence's block list.  Positions past n_ids*bs set XS_FLAG_BAD_LEN, ids
 * outside [0, num_blocks) XS_FLAG_BAD_BLOCK; both are skipped.  Bit-exact.
 */
int xs_prefill_append(const void *k_src, const void *v_src, void *k_cache, void *v_cache,
                      const int32_t *block_ids, int n_ids, int T, int Hkv, int D, int block_size,
                      int64_t num_blocks, int start_pos, int dtype, int *err_flag,
                      cudaStream_t stream);

/*
 * XS_PREFILL_OVERLAP - lets the launches of a chunked prefill overlap: chunk
 * c + 1's append and attention may start while chunk c's attention is still
 * running, on the SMs it leaves idle.
 *
 * xs_prefill_append_ex with this flag is launched programmatically dependent
 * on the previous kernel on the stream and does not wait for it: the caller
 * promises that kernel (if still running) writes none of k_src, v_src and
 * block_ids, and reads or writes none of the rows this launch appends - true
 * when it is the attention of the previous chunk of the same sequence, which
 * reads positions before start_pos only.
 *
 * xs_paged_prefill_tc_ex with this flag is launched programmatically
 * dependent on the previous kernel and reads q, block_ids and the K/V rows
 * of positions before start_pos (key tiles that end before it) before
 * waiting for that kernel; the rows from start_pos on, and every write, wait
 * for it.  The caller promises the previous kernel writes none of what is
 * read early - true when it is this chunk's append (which writes positions
 * from start_pos on) launched with the same flag behind the previous chunk's
 * attention.  Its successor may start once that wait has returned, so a
 * chain append(c), attention(c), append(c + 1), ... never lets a launch read
 * rows whose append has not completed: each attention's wait covers its own
 * chunk's append, which started only after the previous attention's wait
 * covered the append before it.
 *
 * flags 0 is xs_prefill_append / xs_paged_prefill_tc; unknown bits are
 * XS_EUNSUPPORTED.
 */
#define XS_PREFILL_OVERLAP 1
int xs_prefill_append_ex(const void *k_src, const void *v_src, void *k_cache, void *v_cache,
                         const int32_t *block_ids, int n_ids, int T, int Hkv, int D,
                         int block_size, int64_t num_blocks, int start_pos, int flags, int dtype,
                         int *err_flag, cudaStream_t stream);

/*
 * xs_paged_prefill_attn / xs_paged_prefill_reduce / xs_paged_prefill -
 * causal attention of a T-token prefill chunk over one sequence's paged
 * cache (the chunk already appended): query token i (q [T, Hq, D], out
 * [T, Hq, D]) sits at position start_pos + i and attends to every cached
 * token t <= start_pos + i through block_ids (the pages' attention with a
 * causal mask offset by the cached prefix, "xserv compare phase10...cf1e9e4",
 * attention.rs, attention / apply_causal_mask / flash_attention).
 * start_pos + T must not exceed n_ids * block_size (XS_ESHAPE).  Split-K and
 * workspace as xs_paged_decode_attn with B = T and max_blocks_per_seq =
 * n_ids: partials [T, Hq, max_partitions, D].  Row i equals the decode
 * attention of the token at position start_pos + i.
 */
int xs_paged_prefill_attn(void *out, float *part_o, float *part_m, float *part_l, const void *q,
                          const void *k_cache, const void *v_cache, const int32_t *block_ids,
                          int n_ids, int T, int start_pos, int Hq, int Hkv, int D,
                          int block_size, int64_t num_blocks, float scale, int partition_tokens,
                          int max_partitions, int dtype, int *err_flag, int *work_counters,
                          cudaStream_t stream);
int xs_paged_prefill_reduce(void *out, const float *part_o, const float *part_m,
                            const float *part_l, int T, int start_pos, int Hq, int D,
                            int partition_tokens, int max_partitions, int dtype,
                            cudaStream_t stream);
int xs_paged_prefill(void *out, float *part_o, float *part_m, float *part_l, const void *q,
                     const void *k_cache, const void *v_cache, const int32_t *block_ids,
                     int n_ids, int T, int start_pos, int Hq, int Hkv, int D, int block_size,
                     int64_t num_blocks, float scale, int partition_tokens, int max_partitions,
                     int dtype, int *err_flag, int *work_counters, cudaStream_t stream);

/*
 * xs_paged_prefill_tc - the same causal chunk attention as xs_paged_prefill
 * (q [T, Hq, D], out [T, Hq, D], block_ids [n_ids], row i at position
 * start_pos + i over the cached prefix and the chunk), on the tensor cores,
 * in one launch with no workspace: CTAs of two tiles of 128 (query token,
 * query head) rows of one KV group stream 128-key K/V tiles through shared
 * memory with TMA and compute Q K^T and P V with tcgen05.mma into TMEM (bf16
 * operands, fp32 accumulation; the softmax weights P enter P V rounded to
 * bf16).  bf16 only (XS_F32 is
 * XS_EUNSUPPORTED); D in {64, 128}; G = Hq / Hkv in {1, 2, 4, 8};
 * num_blocks * Hkv * 16 + 16 < 2^31 (TMA row coordinates).  A block id
 * outside the pool reads as zeros and raises XS_FLAG_BAD_BLOCK.  Errors
 * otherwise as xs_paged_prefill; XS_EDEVICE if the driver's tensor-map
 * encoder cannot be found.
 */
int xs_paged_prefill_tc(void *out, const void *q, const void *k_cache, const void *v_cache,
                        const int32_t *block_ids, int n_ids, int T, int start_pos, int Hq,
                        int Hkv, int D, int block_size, int64_t num_blocks, float scale,
                        int dtype, int *err_flag, cudaStream_t stream);
/* xs_paged_prefill_tc with launch flags (XS_PREFILL_OVERLAP, above). */
int xs_paged_prefill_tc_ex(void *out, const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *block_ids, int n_ids, int T, int start_pos, int Hq,
                           int Hkv, int D, int block_size, int64_t num_blocks, float scale,
                           int flags, int dtype, int *err_flag, cudaStream_t stream);

/*
 * xs_block_alloc_decode - the page allocation of one decode step, on the
 * device (the pages' PagedKVCache gives a sequence a new physical block when
 * its next token starts a page; "xserv compare phase10...cf1e9e4", the
 * bench-qwen3 and gpt-oss drivers: PagedKVCache::new_tp(.., total_blocks,
 * .., max_blocks_per_seq, ..), register_sequence, free_sequence, seq_len).
 *
 * free_stack int32 [capacity] holds free block ids in [0, *free_top);
 * free_top is one int32 on the device.  For every b with context_lens[b] >=
 * 0 (a slot with -1 holds no sequence): the token this step writes sits at
 * p = context_lens[b]; if p % block_size == 0 it starts page p / block_size,
 * which gets the block popped from the stack; then context_lens[b] = p + 1,
 * so the lengths mean what xs_kv_append_paged and xs_paged_decode_attn
 * expect.  A page past the table sets XS_FLAG_BAD_LEN, an empty stack
 * XS_FLAG_POOL_EMPTY; that sequence is left unchanged.  Which sequence gets
 * which popped block depends on the order of atomic operations.
 * Everything is device state, so the call can sit in a captured step.
 */
int xs_block_alloc_decode(int32_t *block_tables, int max_blocks_per_seq, int32_t *context_lens,
                          int B, int block_size, const int32_t *free_stack, int32_t *free_top,
                          int *err_flag, cudaStream_t stream);

/*
 * xs_block_free - release sequences (PagedKVCache::free_sequence): all blocks
 * of each listed slot (seq_ids int32 [n], distinct, on the device) are pushed
 * on the free stack, the slot's table row is set to -1 and its length to -1
 * (no sequence; write 0 to register a new, empty one).  A full stack sets
 * XS_FLAG_POOL_EMPTY; an id outside [0, B) sets XS_FLAG_BAD_SLOT.
 */
int xs_block_free(const int32_t *seq_ids, int n, int32_t *block_tables, int max_blocks_per_seq,
                  int32_t *context_lens, int B, int block_size, int32_t *free_stack,
                  int32_t *free_top, int64_t stack_capacity, int *err_flag, cudaStream_t stream);

/*
 * xs_kv_swap - copy whole KV blocks from one pool to another, e.g. from the
 * device pool to a swap pool in pinned host memory (swap-out) or back
 * (swap-in): the pages' CPU swap of paged KV blocks ("xserv compare
 * phase10...cf1e9e4", README, --swap-space-gb, KV swapped out to pinned CPU
 * memory).
 *
 * For every i < n with s = block_mapping[2i] >= 0 and d = block_mapping[2i+1]
 * >= 0, the block_bytes bytes of block s of src_k (and src_v) are copied to
 * block d of dst_k (and dst_v); a block is [Hkv, block_size, D] of the pool
 * layout, so block_bytes = Hkv * block_size * D * element size (a multiple of
 * 16).  Any pool may live in device memory or in pinned host memory the GPU
 * can address (GB300 reaches it over NVLink-C2C); block_mapping (int64
 * [n, 2]) must be device-accessible too.  Destinations must be distinct.
 * Ids at or past src_blocks / dst_blocks set XS_FLAG_BAD_BLOCK and are
 * skipped; pairs with a negative id are skipped silently.  Bit-exact.
 * Every pointer is checked first (cudaPointerGetAttributes): pinned host
 * memory is used through its device alias, pageable host memory only where
 * the device can access pageable memory; anything else returns
 * XS_EUNSUPPORTED without launching.
 */
int xs_kv_swap(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
               const int64_t *block_mapping, int n, int64_t block_bytes, int64_t src_blocks,
               int64_t dst_blocks, int *err_flag, cudaStream_t stream);

/*
 * xs_paged_decode_partition_tokens - host-only heuristic for the split-K
 * partition size (tokens, a multiple of 16) of xs_paged_decode_attn.
 *
 * Each sequence's context is cut into partitions of this many tokens; one
 * work item is (sequence, KV head, partition).  The heuristic picks the
 * power of two in [64, 2048] that minimises a simple cost model: items per
 * resident CTA (2 per SM) plus one, times the time of one item (its pages
 * spread over 4 consumer warps plus a fixed per-item cost for staging q,
 * merging and the partials).  total_context_tokens = sum of context_lens
 * (pass <= 0 if unknown: B * max_context_len is used).  Returns the
 * partition size, or a negative XS_E* code.
 */
int xs_paged_decode_partition_tokens(int B, int Hkv, int64_t total_context_tokens,
                                     int max_context_len, int num_sms);

/*
 * xs_paged_decode_max_partitions - partitions a sequence can need: the
 * ceiling of max_blocks_per_seq*block_size / partition_tokens.
 */
int xs_paged_decode_max_partitions(int max_blocks_per_seq, int block_size, int partition_tokens);

/*
 * xs_paged_decode_num_splits - the split-K factor of the longest sequence:
 * how many partitions of xs_paged_decode_partition_tokens(B, Hkv,
 * B * max_context_len, max_context_len, sm_count) tokens a context of
 * max_context_len tokens is cut into (1 = no split, no reduce needed).  The
 * split is chosen from the batch, the KV heads, the context length and the
 * SM count so that the work items fill the resident CTAs (2 per SM).  Host
 * only.  Returns the count (>= 1), or XS_ESHAPE (B < 0, Hkv <= 0,
 * max_context_len < 0, sm_count <= 0).
 */
int xs_paged_decode_num_splits(int B, int Hkv, int max_context_len, int sm_count);

/*
 * xs_paged_decode_workspace_bytes - bytes of fp32 partials for the split:
 * part_o [B, Hq, max_partitions, D], part_m and part_l [B, Hq,
 * max_partitions], each rounded up to 256 bytes (the caller may carve one
 * buffer: part_o at 0, part_m and part_l after it).
 */
size_t xs_paged_decode_workspace_bytes(int B, int Hq, int D, int max_partitions);

/*
 * xs_paged_decode_attn - paged decode attention, split-K partition pass.
 *
 * For sequence b, query head h, KV head g = h / (Hq/Hkv), tokens
 * t < N = context_lens[b] gathered through the page table
 * (K_t = k_cache[block_tables[b][t / bs], g, t % bs, :]):
 *     out[b, h, :] = sum_t softmax_t(scale * q[b, h, :] . K_t) V_t
 * ("xserv compare phase10...cf1e9e4", attention.rs, paged_decode_attention
 * and its launch_paged_decode_attention_bf16 signature; the softmax over all
 * cached tokens from "xserv compare phase5...phase9", docs/09-kv-cache.md).
 *
 * Work split: every (b, g, partition p) covers tokens
 * [p*P, min(N, (p+1)*P)) with P = partition_tokens (a multiple of 16) and
 * computes all Hq/Hkv query heads of group g from one read of each page.
 *  - A sequence with one partition (N <= P) gets its final out[b] written
 *    here.
 *  - A sequence with more partitions gets fp32 partials instead:
 *      part_o[b, h, p, :] = sum_t w_t V_t / l,  part_l[b, h, p] = l = sum_t w_t,
 *      part_m[b, h, p] = max_t logit_t * log2(e)  (w_t = 2^(logit_t*log2 e - m));
 *    xs_paged_decode_reduce then writes out[b].
 *  - A sequence with N <= 0 gets out[b] = 0.
 * max_partitions must be >= xs_paged_decode_max_partitions(...); part_* may
 * be NULL only when max_partitions == 1.
 *
 * Scheduling: a persistent grid (resident CTAs on every SM) takes the work
 * items.  With work_counters == NULL, CTA c takes items c, c + grid, ...
 * With work_counters (2 ints on the device, zero before the first launch
 * that uses them), CTAs take the next item from work_counters[0] as they
 * finish, which balances ragged batches; the last CTA of every launch sets
 * both ints back to zero.  Launches sharing one work_counters buffer must be
 * ordered (one stream); if a launch is abandoned, zero the buffer before the
 * next one.
 *
 * q [B, Hq, D]; out [B, Hq, D]; k_cache, v_cache [num_blocks, Hkv, bs, D];
 * block_tables int32 [B, max_blocks_per_seq]; context_lens int32 [B].
 * Device-side errors: XS_FLAG_BAD_BLOCK, XS_FLAG_BAD_LEN, XS_FLAG_TIMEOUT.
 */
int xs_paged_decode_attn(void *out, float *part_o, float *part_m, float *part_l,
                         const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *context_lens, int B, int Hq, int Hkv, int D,
                         int block_size, int64_t num_blocks, float scale,
                         int partition_tokens, int max_partitions, int dtype, int *err_flag,
                         int *work_counters, cudaStream_t stream);

/*
 * xs_paged_decode_reduce - split-K combine.  For every sequence with more
 * than one partition and every query head, merges the partials by their
 * log-sum-exp weights:
 *     M = max_i m_i,  L = sum_i l_i 2^(m_i - M),
 *     out = sum_i l_i 2^(m_i - M) o_i / L
 * and writes out[b, h, :] in dtype.  Sequences with one partition or none
 * are left as xs_paged_decode_attn wrote them.  Arguments as in
 * xs_paged_decode_attn; partials are read only.
 */
int xs_paged_decode_reduce(void *out, const float *part_o, const float *part_m,
                           const float *part_l, const int32_t *context_lens, int B, int Hq,
                           int D, int partition_tokens, int max_partitions, int dtype,
                           cudaStream_t stream);

/*
 * xs_paged_decode_attn_splits, xs_paged_decode_reduce_splits - the two
 * passes with the split given as a count, as in the survey's sketch of this
 * boundary: num_splits >= 1 partitions of
 *     P = round_up(ceil(max_blocks_per_seq * block_size / num_splits), 16)
 * tokens cover the longest sequence the table can hold, so partials sized by
 * xs_paged_decode_workspace_bytes(B, Hq, D, num_splits) hold every split.
 * They are xs_paged_decode_attn / xs_paged_decode_reduce with
 * partition_tokens = P and max_partitions = num_splits (and no work
 * counters); a sequence shorter than P still gets its out[b] from the first
 * pass, so out is required in both.  With num_splits == 1 every sequence is
 * one partition, out is final after the first pass and the partials may be
 * NULL; the second pass then does nothing.  The reduce takes
 * max_blocks_per_seq and block_size to derive the same P.  XS_ESHAPE for
 * num_splits <= 0; other arguments and errors as the two passes.
 */
int xs_paged_decode_attn_splits(void *out, float *part_o, float *part_m, float *part_l,
                                const void *q, const void *k_cache, const void *v_cache,
                                const int32_t *block_tables, int max_blocks_per_seq,
                                const int32_t *context_lens, int B, int Hq, int Hkv, int D,
                                int block_size, int64_t num_blocks, float scale, int num_splits,
                                int dtype, int *err_flag, cudaStream_t stream);
int xs_paged_decode_reduce_splits(void *out, const float *part_o, const float *part_m,
                                  const float *part_l, const int32_t *context_lens,
                                  int max_blocks_per_seq, int B, int Hq, int D, int block_size,
                                  int num_splits, int dtype, cudaStream_t stream);

/*
 * xs_paged_decode - xs_paged_decode_attn followed, when max_partitions > 1,
 * by xs_paged_decode_reduce on the same stream.
 */
int xs_paged_decode(void *out, float *part_o, float *part_m, float *part_l, const void *q,
                    const void *k_cache, const void *v_cache, const int32_t *block_tables,
                    int max_blocks_per_seq, const int32_t *context_lens, int B, int Hq, int Hkv,
                    int D, int block_size, int64_t num_blocks, float scale, int partition_tokens,
                    int max_partitions, int dtype, int *err_flag, int *work_counters,
                    cudaStream_t stream);

/*
 * xs_paged_decode_attn_sinks / xs_paged_decode_reduce_sinks /
 * xs_paged_decode_sinks - the gpt-oss variant of the three calls above
 * ("xserv compare phase10...cf1e9e4", attention.rs,
 * paged_decode_attention_sinks and launch_paged_decode_attention_sinks_bf16):
 *  - sinks: NULL or [Hq] values of the q dtype, one per query head.  A sink
 *    is one more logit, in the same units as scale * q.K, with no value row:
 *    it only adds exp(sink - max) to the softmax denominator.
 *  - window: 0 = attend to every cached token; W > 0 = a sliding window,
 *    only the W most recent tokens [max(0, N - W), N) of each sequence.
 * The split covers the windowed range; the reduce must get the same sinks
 * and window as the attention pass.  Arguments and errors otherwise as
 * xs_paged_decode_attn / xs_paged_decode_reduce / xs_paged_decode; a
 * negative window is XS_ESHAPE.
 */
int xs_paged_decode_attn_sinks(void *out, float *part_o, float *part_m, float *part_l,
                               const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *block_tables, int max_blocks_per_seq,
                               const int32_t *context_lens, const void *sinks, int window, int B,
                               int Hq, int Hkv, int D, int block_size, int64_t num_blocks,
                               float scale, int partition_tokens, int max_partitions, int dtype,
                               int *err_flag, int *work_counters, cudaStream_t stream);
int xs_paged_decode_reduce_sinks(void *out, const float *part_o, const float *part_m,
                                 const float *part_l, const int32_t *context_lens,
                                 const void *sinks, int window, int B, int Hq, int D,
                                 int partition_tokens, int max_partitions, int dtype,
                                 cudaStream_t stream);
int xs_paged_decode_sinks(void *out, float *part_o, float *part_m, float *part_l, const void *q,
                          const void *k_cache, const void *v_cache, const int32_t *block_tables,
                          int max_blocks_per_seq, const int32_t *context_lens, const void *sinks,
                          int window, int B, int Hq, int Hkv, int D, int block_size,
                          int64_t num_blocks, float scale, int partition_tokens,
                          int max_partitions, int dtype, int *err_flag, int *work_counters,
                          cudaStream_t stream);

/*
 * xs_paged_decode_step - one whole decode step in ONE launch: the KV append
 * of xs_kv_append_paged, the attention of xs_paged_decode_attn_sinks and the
 * split-K combine of xs_paged_decode_reduce_sinks ("xserv compare
 * phase10...cf1e9e4", attention.rs: reshape_and_cache_batched_bf16, then
 * paged_decode_attention / paged_decode_attention_sinks).  The result equals
 * those three calls in that order.
 *
 * How the launch does it:
 *  - append: the work item that covers sequence b's last page for KV head g
 *    writes k_new[b, g, :] and v_new[b, g, :] into slot
 *    block_tables[b][(N-1)/16] * 16 + (N-1) % 16 (N = context_lens[b]) and
 *    then loads that page, so the new token is attended to.  N <= 0 appends
 *    nothing; N beyond the table appends nothing and raises XS_FLAG_BAD_LEN;
 *    an out-of-pool block id appends nothing and raises XS_FLAG_BAD_BLOCK.
 *    k_new and v_new are both NULL (attention only) or both [B, Hkv, D] in
 *    dtype.  No other sequence may attend to a row written in the same step
 *    (true of any block table where the block a sequence appends to is its
 *    own, e.g. shared prefixes copied on write).
 *  - combine: each item of a split (sequence, KV head) writes its partials,
 *    then counts itself in; the item that completes the group merges the
 *    group's partials for the G query heads into out.
 *  - small launches (xs_paged_decode_step_cluster_size > 0: bf16, every
 *    (sequence, KV head) group in one wave of thread-block clusters)
 *    run one cluster per group instead: its CTAs split the group's tokens
 *    into their own partitions (partition_tokens is not used), and the
 *    split-K combine reads the CTAs' partials from distributed shared
 *    memory, so part_o/part_m/part_l and the counters are not touched (they
 *    must still be valid).  The result is the same up to the order of the
 *    fp32 sums.
 *
 * counters: int32 on the device, xs_paged_decode_step_counters(B, Hkv) of
 * them (2 + B * Hkv: the work-item counters, then one arrival count per
 * sequence and KV head), zero before the first launch; every completed
 * launch leaves them zero.  Launches sharing counters must be ordered (one
 * stream, or one CUDA graph).  After a launch that raised XS_FLAG_TIMEOUT,
 * zero them before the next launch.  NULL counters is XS_EWORKSPACE.
 *
 * Other arguments, layouts, workspace rules and errors as
 * xs_paged_decode_attn_sinks (sinks NULL and window 0 give the plain step).
 * k_cache and v_cache are written (the new rows only).
 */
int xs_paged_decode_step(void *out, const void *q, const void *k_new, const void *v_new,
                         void *k_cache, void *v_cache, const int32_t *block_tables,
                         int max_blocks_per_seq, const int32_t *context_lens, const void *sinks,
                         int window, int B, int Hq, int Hkv, int D, int block_size,
                         int64_t num_blocks, float scale, int partition_tokens,
                         int max_partitions, float *part_o, float *part_m, float *part_l,
                         int *counters, int dtype, int *err_flag, cudaStream_t stream);

/*
 * xs_paged_decode_step_ex - xs_paged_decode_step with launch flags (flags 0
 * is xs_paged_decode_step; XS_STEP_EARLY_READS and XS_STEP_PERSISTENT may be
 * combined).  Unknown flag bits are XS_EUNSUPPORTED.
 *
 * XS_STEP_EARLY_READS: the launch is made programmatically dependent on the
 * previous kernel on the stream (as every launch of this library is), and
 * reads context_lens, block_tables and the first pages of each CTA's first
 * work item BEFORE waiting for that kernel to complete, overlapping that
 * start-up (lengths -> item tables -> block ids -> pages: dependent memory
 * round trips) with the previous kernel's tail.  In a launch of at most 16
 * rounds of work items (a round: one item per resident CTA), each CTA also
 * prefetches the next 16 pages of its first item into L2 at that point (a
 * cache hint: L2 is coherent, so nothing stale can be read through it).
 * q, k_new/v_new, the counters and every write wait for it as usual; a page
 * that receives this launch's appended row is not read early.  The caller
 * promises that the
 * kernel launched just before this one on the stream (if it is still
 * running) writes none of context_lens, block_tables, or the pages of
 * k_cache/v_cache this launch attends to (other than the rows it appends
 * itself), and neither does any earlier kernel that kernel lets run beside
 * it - true, for instance, when the previous kernel is a projection GEMM or
 * the attention step of another layer.  (No launch of this library lets its
 * successor start before its own wait has returned, so behind one of them
 * only that launch can still be running.)
 */
#define XS_STEP_EARLY_READS 1
/*
 * XS_STEP_PERSISTENT: run the persistent grid (partials in part_o/part_m/
 * part_l, counted through the counters) even where the launch would run as
 * clusters (xs_paged_decode_step_cluster_size > 0).  Same result up to the
 * order of the fp32 sums.
 */
#define XS_STEP_PERSISTENT 2
int xs_paged_decode_step_ex(void *out, const void *q, const void *k_new, const void *v_new,
                            void *k_cache, void *v_cache, const int32_t *block_tables,
                            int max_blocks_per_seq, const int32_t *context_lens, const void *sinks,
                            int window, int B, int Hq, int Hkv, int D, int block_size,
                            int64_t num_blocks, float scale, int partition_tokens,
                            int max_partitions, float *part_o, float *part_m, float *part_l,
                            int *counters, int flags, int dtype, int *err_flag,
                            cudaStream_t stream);

/*
 * xs_paged_decode_step_partition_tokens - partition length P for
 * xs_paged_decode_step: the cost model of xs_paged_decode_partition_tokens
 * fitted to one-launch step times, with whole rounds of the grid when every
 * sequence has the same length (total_context_tokens = B * max_context_len)
 * and a cost per partition of the longest sequence for its split-K combine,
 * searched over multiples of 64 in [64, 2048] (64, 128, ..., 576, 640, 768,
 * 896, 1024, 1280, 1536, 2048) so that a batch's item count can land just
 * under a whole number of rounds of the grid.  Same arguments plus Hq;
 * XS_ESHAPE also when Hq % Hkv != 0.
 */
int xs_paged_decode_step_partition_tokens(int B, int Hq, int Hkv, int64_t total_context_tokens,
                                          int max_context_len, int num_sms);

/*
 * xs_paged_decode_step_cluster_size - the cluster size (2..16) with which
 * xs_paged_decode_step / _ex runs a launch of this shape on the current
 * device, or 0 when it runs the persistent grid.  Clusters are used for bf16
 * (D = 64 or 128) when the tokens a sequence can hold (max_blocks_per_seq * 16, or
 * the window when smaller) split into at most 16 partitions of at most 192
 * pages (191 with a window) and all B * Hkv clusters fit the device at once;
 * the largest such size is taken (at most one CTA per 64 tokens), except
 * that a launch of short partitions (at most 32 pages) which would fill
 * every cluster slot takes the largest smaller size that leaves a slot free
 * (so the next launch can start early), if that adds at most half again to
 * the pages of a CTA.  Only the
 * shape decides: B, Hq, Hkv, D, max_blocks_per_seq, window and dtype are
 * those of the step.  XS_ESHAPE for a negative size, Hq % Hkv != 0.
 */
int xs_paged_decode_step_cluster_size(int B, int Hq, int Hkv, int D, int max_blocks_per_seq,
                                      int window, int dtype);

/*
 * xs_paged_decode_step_counters - how many int32 counters
 * xs_paged_decode_step needs for B sequences and Hkv KV heads (2 + B * Hkv),
 * or XS_ESHAPE (B < 0, Hkv <= 0).
 */
int64_t xs_paged_decode_step_counters(int B, int Hkv);

/*
 * xs_paged_decode_noalloc - xs_paged_decode for callers that cannot allocate
 * device memory.  The paper has no counterpart of this entry point: it is a
 * service of this library.
 *
 * Who needs it: code that must not call cudaMalloc/cudaFree (or any
 * allocating library routine) on its decode path - for example an engine
 * that has already handed all free device memory to its own KV pool, a
 * plugin whose host application owns every allocation, or a serving loop
 * where an allocation could stall the device (cudaFree synchronises) or fail
 * under memory pressure in the middle of a step.  Such callers still pass
 * q, the pools, the tables and out, but not the split-K partials.
 *
 * The partials live in one array that the library defines at file scope in
 * device memory, XS_NOALLOC_SCRATCH_BYTES (64 MiB) in size.  Every GPU that
 * loads the library reserves that array until the process exits.  The call
 * allocates nothing: on every call it looks up the array's device address for
 * the current device and context with cudaGetSymbolAddress (nothing is
 * cached, so a cudaDeviceReset or another current context cannot leave a
 * stale address).  The first call on a device may load the library's device
 * code there (lazy module loading), so make that first call on each device -
 * any call that passes the argument checks - before any stream capture.
 *
 * Arguments as xs_paged_decode, without part_o/part_m/part_l and
 * max_partitions (derived as xs_paged_decode_max_partitions(
 * max_blocks_per_seq, block_size, partition_tokens)).  partition_tokens <= 0
 * picks the size with xs_paged_decode_partition_tokens for the current
 * device, taking B * max_blocks_per_seq * block_size as the token count.
 * Returns XS_ESCRATCH, before launching anything, when
 * xs_paged_decode_workspace_bytes(B, Hq, D, max_partitions) exceeds
 * XS_NOALLOC_SCRATCH_BYTES (choose a larger partition_tokens or a smaller
 * batch).
 *
 * All calls share the one array and it keeps whatever the last call left
 * there.  Nothing in it needs clearing: every partial the reduce reads is
 * written by the attention pass of the same call first.  Two calls whose
 * work overlaps on the GPU (different streams, or different host threads)
 * race on the array and corrupt each other's results; order them on one
 * stream or serialise them.
 */
#define XS_NOALLOC_SCRATCH_BYTES (64ull << 20)
int xs_paged_decode_noalloc(void *out, const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *context_lens, int B, int Hq, int Hkv, int D,
                            int block_size, int64_t num_blocks, float scale,
                            int partition_tokens, int dtype, int *err_flag,
                            cudaStream_t stream);

/*
 * xs_version - library version as MAJOR*10000 + MINOR*100 + PATCH.
 */
int xs_version(void);

/*
 * xs_debug_bounds_failures - in the debug library (libxs_paged_debug.so,
 * the same sources compiled with -DXS_DEBUG_BOUNDS), the number of in-kernel
 * bounds checks that failed on the current device since the last reset
 * (reset != 0 clears the count after reading it).  Every global-memory index
 * the kernels compute is checked there against its buffer's extent before
 * the access; a failure skips the access and raises XS_FLAG_BOUNDS.  The
 * paper has no counterpart of this entry point: the checks are a test aid
 * standing in for a device memory checker.  Synchronous (it copies the
 * counters).
 * Returns XS_EUNSUPPORTED in the release library, XS_EDEVICE if the copy
 * failed.
 */
int xs_debug_bounds_failures(int reset);

/*
 * xs_debug_wait_injection - in the debug library only, a way to make the
 * decode kernel's bounded waits run out on purpose, so the recovery path can
 * be exercised without a device fault.  The paper has no counterpart of this
 * entry point: it is a test aid.
 *
 * wait_limit_ns (> 0) becomes the limit of every bounded wait of the decode
 * kernel (default 4e9, i.e. 4 s).  skip_page >= 0 makes CTA 0's producer skip
 * issuing the copies of its page number skip_page (its pages counted from 0
 * in the order it issues them) in every later launch: nothing is in flight
 * for that page, the consumer's wait for it runs out, the launch raises
 * XS_FLAG_TIMEOUT, drains the copies it did issue and returns; -1 issues
 * every page.  Both settings hold on the current device until changed.
 * After a launch that raised XS_FLAG_TIMEOUT the outputs of the affected
 * sequences are unspecified and the step's counters must be zeroed (see
 * xs_paged_decode_step).  Synchronous.  Returns XS_OK, XS_ESHAPE
 * (wait_limit_ns <= 0 or skip_page < -1), XS_EDEVICE if the copy failed, and
 * XS_EUNSUPPORTED in the release library.
 */
int xs_debug_wait_injection(int64_t wait_limit_ns, int skip_page);

#ifdef __cplusplus
}
#endif

#endif /* XS_PAGED_H */
