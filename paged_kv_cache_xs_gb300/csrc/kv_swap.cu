// KV swap: whole-block copies between two paged pools - the device pool and a
// swap pool in pinned host memory, either direction - so KV blocks can be
// moved out of HBM and back ("xserv compare phase10...cf1e9e4", README: the
// paged KV cache swaps blocks out to pinned CPU memory, --swap-space-gb).
//
// One launch moves every mapped block: each thread keeps several 16-byte
// loads in flight before storing them, because on GB300 the GPU reaches the
// pinned host pool directly over NVLink-C2C, where latency is high.
#include <algorithm>

#include "xs_common.cuh"

namespace xs {
namespace {

constexpr int kSwapThreads = 256;
constexpr int kSwapUnroll = 4;

__global__ void __launch_bounds__(kSwapThreads)
    kv_swap_kernel(const uint4 *__restrict__ src_k, const uint4 *__restrict__ src_v,
                   uint4 *__restrict__ dst_k, uint4 *__restrict__ dst_v,
                   const int64_t *__restrict__ mapping, int n, int64_t chunks_per_block,
                   int64_t src_blocks, int64_t dst_blocks, int *err_flag) {
    const int64_t per_pair = 2 * chunks_per_block;
    const int64_t total = static_cast<int64_t>(n) * per_pair;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x * kSwapUnroll + threadIdx.x;
         base < total; base += stride * kSwapUnroll) {
        uint4 v[kSwapUnroll];
        int64_t dst_idx[kSwapUnroll];
        bool is_v[kSwapUnroll];
#pragma unroll
        for (int u = 0; u < kSwapUnroll; ++u) {
            dst_idx[u] = -1;
            const int64_t i = base + static_cast<int64_t>(u) * blockDim.x;
            if (i >= total) continue;
            const int64_t pair = i / per_pair;
            const int64_t r = i - pair * per_pair;
            is_v[u] = r >= chunks_per_block;
            const int64_t c = is_v[u] ? r - chunks_per_block : r;
            const int64_t s = mapping[2 * pair], d = mapping[2 * pair + 1];
            if (s < 0 || d < 0) continue;
            if (s >= src_blocks || d >= dst_blocks) {
                if (r == 0) raise_flag(err_flag, XS_FLAG_BAD_BLOCK);
                continue;
            }
            v[u] = is_v[u] ? src_v[s * chunks_per_block + c] : src_k[s * chunks_per_block + c];
            dst_idx[u] = d * chunks_per_block + c;
        }
#pragma unroll
        for (int u = 0; u < kSwapUnroll; ++u) {
            if (dst_idx[u] < 0) continue;
            if (is_v[u])
                dst_v[dst_idx[u]] = v[u];
            else
                dst_k[dst_idx[u]] = v[u];
        }
    }
}

// The address the device uses for p: device and managed memory as is, pinned
// host memory through its mapped alias, pageable host memory only where the
// device can read pageable memory (e.g. over NVLink-C2C with address
// translation).  nullptr when the device cannot reach p.
const void *device_view(const void *p, int dev) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    switch (a.type) {
        case cudaMemoryTypeDevice:
        case cudaMemoryTypeManaged:
            return a.devicePointer ? a.devicePointer : p;
        case cudaMemoryTypeHost:
            return a.devicePointer;
        default: {
            int pageable = 0;
            if (cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev) !=
                cudaSuccess)
                return nullptr;
            return pageable ? p : nullptr;
        }
    }
}

}  // namespace
}  // namespace xs

extern "C" int xs_kv_swap(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                          const int64_t *block_mapping, int n, int64_t block_bytes,
                          int64_t src_blocks, int64_t dst_blocks, int *err_flag,
                          cudaStream_t stream) {
    if (!src_k || !src_v || !dst_k || !dst_v || !block_mapping) return XS_ENULL;
    if (n < 0 || block_bytes <= 0 || src_blocks < 0 || dst_blocks < 0) return XS_ESHAPE;
    if (block_bytes % 16 != 0) return XS_EUNSUPPORTED;
    if (!xs::aligned16(src_k) || !xs::aligned16(src_v) || !xs::aligned16(dst_k) ||
        !xs::aligned16(dst_v))
        return XS_EALIGN;
    if (n == 0) return XS_OK;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return XS_EDEVICE;
    const void *sk = xs::device_view(src_k, dev), *sv = xs::device_view(src_v, dev);
    const void *dk = xs::device_view(dst_k, dev), *dv = xs::device_view(dst_v, dev);
    const void *mp = xs::device_view(block_mapping, dev);
    if (!sk || !sv || !dk || !dv || !mp) return XS_EUNSUPPORTED;  // not device-accessible
    const int64_t chunks = block_bytes / 16;
    const int64_t total = static_cast<int64_t>(n) * 2 * chunks;
    const int64_t per_cta = static_cast<int64_t>(xs::kSwapThreads) * xs::kSwapUnroll;
    const int64_t want = (total + per_cta - 1) / per_cta;
    const int grid = static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(sms) * 8));
    xs::kv_swap_kernel<<<grid, xs::kSwapThreads, 0, stream>>>(
        static_cast<const uint4 *>(sk), static_cast<const uint4 *>(sv),
        static_cast<uint4 *>(const_cast<void *>(dk)), static_cast<uint4 *>(const_cast<void *>(dv)),
        static_cast<const int64_t *>(mp), n, chunks, src_blocks, dst_blocks, err_flag);
    return xs::launch_status();
}
