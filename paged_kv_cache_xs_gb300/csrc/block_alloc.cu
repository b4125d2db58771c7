// Device-side page allocator for the decode step: a free stack of physical
// block ids in device memory; every sequence whose next token starts a page
// pops a block into its block-table row, and its length advances by one.
// With it, every step of a decode loop - allocate, append, attend, reduce -
// runs from device-resident state, so a whole step can be one CUDA graph.
//
// The pages' PagedKVCache (used by the bench-qwen3 / gpt-oss drivers,
// "xserv compare phase10...cf1e9e4": new_tp(.., total_blocks, ..,
// max_blocks_per_seq, ..), register_sequence, free_sequence, seq_len) hands
// out blocks on the host; its body is not on the pages.
#include "xs_common.cuh"

namespace xs {
namespace {

__global__ void block_alloc_decode_kernel(int32_t *__restrict__ block_tables, int max_blocks,
                                          int32_t *__restrict__ lens, int B, int bs,
                                          const int32_t *__restrict__ free_stack,
                                          int32_t *__restrict__ free_top, int *err_flag) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int32_t p = lens[b];
    if (p < 0) return;  // no sequence in this slot
    const int32_t page = p / bs;
    if (page >= max_blocks) {
        raise_flag(err_flag, XS_FLAG_BAD_LEN);
        return;
    }
    if (p % bs == 0) {
        const int32_t idx = atomicSub(free_top, 1) - 1;
        if (idx < 0) {  // the stack ran dry: give the slot back, leave the sequence as is
            atomicAdd(free_top, 1);
            raise_flag(err_flag, XS_FLAG_POOL_EMPTY);
            return;
        }
        block_tables[static_cast<int64_t>(b) * max_blocks + page] = free_stack[idx];
    }
    lens[b] = p + 1;
}

// One CTA per released sequence: read its length once, push its blocks,
// then clear its row and mark the slot empty.
__global__ void block_free_kernel(const int32_t *__restrict__ seq_ids, int B,
                                  int32_t *__restrict__ block_tables, int max_blocks,
                                  int32_t *__restrict__ lens, int bs,
                                  int32_t *__restrict__ free_stack, int32_t *__restrict__ free_top,
                                  int64_t capacity, int *err_flag) {
    const int32_t b = seq_ids[blockIdx.x];
    if (b < 0 || b >= B) {
        if (threadIdx.x == 0) raise_flag(err_flag, XS_FLAG_BAD_SLOT);
        return;
    }
    __shared__ int32_t pages;
    if (threadIdx.x == 0) {
        const int32_t n = lens[b];
        pages = n > 0 ? min((n + bs - 1) / bs, max_blocks) : 0;
    }
    __syncthreads();
    int32_t *row = block_tables + static_cast<int64_t>(b) * max_blocks;
    for (int pg = threadIdx.x; pg < pages; pg += blockDim.x) {
        const int32_t blk = row[pg];
        const int32_t idx = atomicAdd(free_top, 1);
        if (idx >= capacity) {
            atomicSub(free_top, 1);
            raise_flag(err_flag, XS_FLAG_POOL_EMPTY);
        } else {
            free_stack[idx] = blk;
        }
    }
    __syncthreads();
    for (int pg = threadIdx.x; pg < max_blocks; pg += blockDim.x) row[pg] = -1;
    if (threadIdx.x == 0) lens[b] = -1;
}

}  // namespace
}  // namespace xs

extern "C" int xs_block_alloc_decode(int32_t *block_tables, int max_blocks_per_seq,
                                     int32_t *context_lens, int B, int block_size,
                                     const int32_t *free_stack, int32_t *free_top, int *err_flag,
                                     cudaStream_t stream) {
    if (!block_tables || !context_lens || !free_stack || !free_top) return XS_ENULL;
    if (B < 0 || max_blocks_per_seq < 0 || block_size <= 0) return XS_ESHAPE;
    if (B == 0) return XS_OK;
    const int threads = 128;
    xs::block_alloc_decode_kernel<<<(B + threads - 1) / threads, threads, 0, stream>>>(
        block_tables, max_blocks_per_seq, context_lens, B, block_size, free_stack, free_top,
        err_flag);
    return xs::launch_status();
}

extern "C" int xs_block_free(const int32_t *seq_ids, int n, int32_t *block_tables,
                             int max_blocks_per_seq, int32_t *context_lens, int B, int block_size,
                             int32_t *free_stack, int32_t *free_top, int64_t stack_capacity,
                             int *err_flag, cudaStream_t stream) {
    if (!seq_ids || !block_tables || !context_lens || !free_stack || !free_top) return XS_ENULL;
    if (n < 0 || B < 0 || max_blocks_per_seq < 0 || block_size <= 0 || stack_capacity < 0)
        return XS_ESHAPE;
    if (n == 0) return XS_OK;
    xs::block_free_kernel<<<n, 128, 0, stream>>>(seq_ids, B, block_tables, max_blocks_per_seq,
                                                 context_lens, block_size, free_stack, free_top,
                                                 stack_capacity, err_flag);
    return xs::launch_status();
}
