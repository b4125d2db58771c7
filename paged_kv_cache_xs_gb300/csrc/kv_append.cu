// KV append for the paged decode step: slot resolution and the 16-byte
// vectorised scatter of new K/V rows into their pool pages.
//
// Pool layout [num_blocks, Hkv, block_size, D] and the meaning of the
// lengths (they already count the token written in this step) follow the xserv pages
// ("xserv compare phase10...cf1e9e4", crates/xserv-kernels/src/attention.rs,
// reshape_and_cache_bf16 / reshape_and_cache_batched_bf16).
#include "xs_common.cuh"

namespace xs {
namespace {

constexpr int kAppendThreads = 256;

// Resolve the slot of the token sequence b writes this step; -1 if none or
// if the table entry is invalid (flagged).
__device__ __forceinline__ int64_t resolve_slot(const int32_t *__restrict__ block_tables,
                                                int max_blocks, const int32_t *__restrict__ lens,
                                                int b, int bs, int64_t num_blocks, int *err_flag) {
    const int32_t n = lens[b];
    if (n <= 0) return -1;
    const int64_t p = static_cast<int64_t>(n) - 1;
    const int64_t lb = p / bs;
    if (lb >= max_blocks) {
        raise_flag(err_flag, XS_FLAG_BAD_LEN);
        return -1;
    }
    const int32_t blk = block_tables[static_cast<int64_t>(b) * max_blocks + lb];
    if (blk < 0 || blk >= num_blocks) {
        raise_flag(err_flag, XS_FLAG_BAD_BLOCK);
        return -1;
    }
    return static_cast<int64_t>(blk) * bs + p % bs;
}

__global__ void slot_mapping_kernel(const int32_t *__restrict__ block_tables, int max_blocks,
                                    const int32_t *__restrict__ lens, int B, int bs,
                                    int64_t num_blocks, int64_t *__restrict__ slots,
                                    int *err_flag) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B) slots[b] = resolve_slot(block_tables, max_blocks, lens, b, bs, num_blocks, err_flag);
}

// One thread moves one 16-byte chunk of one row (token t, K or V, head h).
// Threads of a warp cover consecutive chunks of consecutive heads, so both
// the read of k_new/v_new and the write of each destination row coalesce.
// A slot of -1 (from the table form) or < 0 (given) is skipped.
template <bool kFromTable>
__global__ void __launch_bounds__(kAppendThreads)
    kv_append_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                     uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                     const int64_t *__restrict__ slot_mapping,
                     const int32_t *__restrict__ block_tables, int max_blocks,
                     const int32_t *__restrict__ lens, int T, int Hkv, int chunks_per_row, int bs,
                     int64_t num_blocks, int *err_flag) {
    const int64_t per_token = static_cast<int64_t>(Hkv) * chunks_per_row;
    const int64_t total = static_cast<int64_t>(T) * 2 * per_token;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / (2 * per_token);
        const int64_t r = i - t * 2 * per_token;
        const bool is_v = r >= per_token;
        const int64_t hc = is_v ? r - per_token : r;  // head * chunks + chunk
        int64_t slot;
        if (kFromTable) {
            // Only the first chunk of the token reports table problems.
            slot = resolve_slot(block_tables, max_blocks, lens, static_cast<int>(t), bs, num_blocks,
                                (r == 0) ? err_flag : nullptr);
        } else {
            slot = slot_mapping[t];
            if (slot >= num_blocks * bs) {
                if (r == 0) raise_flag(err_flag, XS_FLAG_BAD_SLOT);
                slot = -1;
            }
        }
        if (slot < 0) continue;
        const int64_t h = hc / chunks_per_row;
        const int64_t c = hc - h * chunks_per_row;
        const int64_t blk = slot / bs, off = slot - (slot / bs) * bs;
        const int64_t dst = ((blk * Hkv + h) * bs + off) * chunks_per_row + c;
        const int64_t src = t * per_token + hc;
        if (!XS_BOUNDS(dst >= 0 && dst < num_blocks * Hkv * bs * chunks_per_row, err_flag))
            continue;
        if (is_v)
            v_cache[dst] = v_new[src];
        else
            k_cache[dst] = k_new[src];
    }
}

// Prefill append: chunk rows src[h, i, :] ([Hkv, T, D], the pages' layout)
// to position start + i of one sequence.  One thread per 16-byte chunk.
__global__ void __launch_bounds__(kAppendThreads)
    prefill_append_kernel(const uint4 *__restrict__ k_src, const uint4 *__restrict__ v_src,
                          uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                          const int32_t *__restrict__ block_ids, int n_ids, int T, int Hkv,
                          int chunks_per_row, int bs, int64_t num_blocks, int start,
                          int *err_flag) {
    // Launched programmatically dependent on the previous kernel only when
    // the caller promised it does not wait for it (XS_PREFILL_OVERLAP): then
    // the next launch (this chunk's attention) may be placed at once.  (A
    // no-op in a launch made without the attribute.)
    griddep_launch_dependents();
    const int64_t per_token = static_cast<int64_t>(Hkv) * chunks_per_row;
    const int64_t total = static_cast<int64_t>(T) * 2 * per_token;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / (2 * per_token);
        const int64_t r = i - t * 2 * per_token;
        const bool is_v = r >= per_token;
        const int64_t hc = is_v ? r - per_token : r;
        const int64_t h = hc / chunks_per_row, c = hc - h * chunks_per_row;
        const int64_t pos = start + t;
        const int64_t page = pos / bs;
        if (page >= n_ids) {
            if (r == 0) raise_flag(err_flag, XS_FLAG_BAD_LEN);
            continue;
        }
        const int32_t blk = block_ids[page];
        if (blk < 0 || blk >= num_blocks) {
            if (r == 0) raise_flag(err_flag, XS_FLAG_BAD_BLOCK);
            continue;
        }
        const int64_t dst = ((static_cast<int64_t>(blk) * Hkv + h) * bs + pos % bs) *
                                chunks_per_row + c;
        const int64_t src = (h * T + t) * chunks_per_row + c;
        if (!XS_BOUNDS(dst >= 0 && dst < num_blocks * Hkv * bs * chunks_per_row, err_flag))
            continue;
        if (is_v)
            v_cache[dst] = v_src[src];
        else
            k_cache[dst] = k_src[src];
    }
}

int launch_append(bool from_table, const void *k_new, const void *v_new, void *k_cache,
                  void *v_cache, const int64_t *slot_mapping, const int32_t *block_tables,
                  int max_blocks, const int32_t *lens, int T, int Hkv, int D, int bs,
                  int64_t num_blocks, int dtype, int *err_flag, cudaStream_t stream) {
    if (!k_new || !v_new || !k_cache || !v_cache) return XS_ENULL;
    if (from_table ? (!block_tables || !lens) : !slot_mapping) return XS_ENULL;
    const int eb = elem_bytes(dtype);
    if (!eb) return XS_EDTYPE;
    if (T < 0 || Hkv <= 0 || D <= 0 || bs <= 0 || num_blocks < 0 || (from_table && max_blocks < 0))
        return XS_ESHAPE;
    if ((static_cast<int64_t>(D) * eb) % 16 != 0) return XS_EUNSUPPORTED;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return XS_EALIGN;
    if (T == 0) return XS_OK;
    const int chunks = D * eb / 16;
    const int64_t total = static_cast<int64_t>(T) * 2 * Hkv * chunks;
    const int64_t blocks64 = (total + kAppendThreads - 1) / kAppendThreads;
    const int grid = static_cast<int>(blocks64 < (1 << 20) ? blocks64 : (1 << 20));
    auto kn = static_cast<const uint4 *>(k_new);
    auto vn = static_cast<const uint4 *>(v_new);
    auto kc = static_cast<uint4 *>(k_cache);
    auto vc = static_cast<uint4 *>(v_cache);
    if (from_table)
        kv_append_kernel<true><<<grid, kAppendThreads, 0, stream>>>(
            kn, vn, kc, vc, nullptr, block_tables, max_blocks, lens, T, Hkv, chunks, bs, num_blocks,
            err_flag);
    else
        kv_append_kernel<false><<<grid, kAppendThreads, 0, stream>>>(
            kn, vn, kc, vc, slot_mapping, nullptr, 0, nullptr, T, Hkv, chunks, bs, num_blocks,
            err_flag);
    return launch_status();
}

}  // namespace
XS_DEFINE_BOUNDS_COUNTER(bounds_failures_append)

}  // namespace xs

extern "C" int xs_slot_mapping(const int32_t *block_tables, int max_blocks_per_seq,
                               const int32_t *context_lens, int B, int block_size,
                               int64_t num_blocks, int64_t *slot_mapping, int *err_flag,
                               cudaStream_t stream) {
    if (!block_tables || !context_lens || !slot_mapping) return XS_ENULL;
    if (B < 0 || block_size <= 0 || max_blocks_per_seq < 0 || num_blocks < 0) return XS_ESHAPE;
    if (B == 0) return XS_OK;
    const int threads = 128;
    xs::slot_mapping_kernel<<<(B + threads - 1) / threads, threads, 0, stream>>>(
        block_tables, max_blocks_per_seq, context_lens, B, block_size, num_blocks, slot_mapping,
        err_flag);
    return xs::launch_status();
}

extern "C" int xs_kv_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                            const int64_t *slot_mapping, int T, int Hkv, int D, int block_size,
                            int64_t num_blocks, int dtype, int *err_flag, cudaStream_t stream) {
    return xs::launch_append(false, k_new, v_new, k_cache, v_cache, slot_mapping, nullptr, 0,
                             nullptr, T, Hkv, D, block_size, num_blocks, dtype, err_flag, stream);
}

extern "C" int xs_kv_append_paged(const void *k_new, const void *v_new, void *k_cache,
                                  void *v_cache, const int32_t *block_tables,
                                  int max_blocks_per_seq, const int32_t *context_lens, int B,
                                  int Hkv, int D, int block_size, int64_t num_blocks, int dtype,
                                  int *err_flag, cudaStream_t stream) {
    return xs::launch_append(true, k_new, v_new, k_cache, v_cache, nullptr, block_tables,
                             max_blocks_per_seq, context_lens, B, Hkv, D, block_size, num_blocks,
                             dtype, err_flag, stream);
}

extern "C" int xs_prefill_append(const void *k_src, const void *v_src, void *k_cache,
                                 void *v_cache, const int32_t *block_ids, int n_ids, int T,
                                 int Hkv, int D, int block_size, int64_t num_blocks, int start_pos,
                                 int dtype, int *err_flag, cudaStream_t stream) {
    return xs_prefill_append_ex(k_src, v_src, k_cache, v_cache, block_ids, n_ids, T, Hkv, D,
                                block_size, num_blocks, start_pos, 0, dtype, err_flag, stream);
}

extern "C" int xs_prefill_append_ex(const void *k_src, const void *v_src, void *k_cache,
                                    void *v_cache, const int32_t *block_ids, int n_ids, int T,
                                    int Hkv, int D, int block_size, int64_t num_blocks,
                                    int start_pos, int flags, int dtype, int *err_flag,
                                    cudaStream_t stream) {
    if (flags & ~XS_PREFILL_OVERLAP) return XS_EUNSUPPORTED;
    if (!k_src || !v_src || !k_cache || !v_cache || !block_ids) return XS_ENULL;
    const int eb = xs::elem_bytes(dtype);
    if (!eb) return XS_EDTYPE;
    if (T < 0 || Hkv <= 0 || D <= 0 || block_size <= 0 || n_ids < 0 || start_pos < 0 ||
        num_blocks < 0)
        return XS_ESHAPE;
    if ((static_cast<int64_t>(D) * eb) % 16 != 0) return XS_EUNSUPPORTED;
    if (!xs::aligned16(k_src) || !xs::aligned16(v_src) || !xs::aligned16(k_cache) ||
        !xs::aligned16(v_cache))
        return XS_EALIGN;
    if (T == 0) return XS_OK;
    const int chunks = D * eb / 16;
    const int64_t total = static_cast<int64_t>(T) * 2 * Hkv * chunks;
    const int64_t blocks64 = (total + xs::kAppendThreads - 1) / xs::kAppendThreads;
    const int grid = static_cast<int>(blocks64 < (1 << 20) ? blocks64 : (1 << 20));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(xs::kAppendThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    if (flags & XS_PREFILL_OVERLAP) {  // (the kernel never waits: the caller's promise)
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    if (cudaLaunchKernelEx(&cfg, xs::prefill_append_kernel, static_cast<const uint4 *>(k_src),
                           static_cast<const uint4 *>(v_src), static_cast<uint4 *>(k_cache),
                           static_cast<uint4 *>(v_cache), block_ids, n_ids, T, Hkv, chunks,
                           block_size, num_blocks, start_pos, err_flag) != cudaSuccess) {
        cudaGetLastError();
        return XS_ELAUNCH;
    }
    return xs::launch_status();
}
