// Chunked-prefill attention on the tensor cores: a T-token chunk at positions
// start_pos .. start_pos + T - 1 attends causally to every cached token of
// its sequence, gathered through the chunk's block list ("xserv compare
// phase10...cf1e9e4", attention.rs, attention / apply_causal_mask /
// flash_attention: softmax(scale * Q K^T + causal mask) V with the mask
// offset by the cached prefix).
//
// Design (flash-attention style, one pass, no split):
//  * CTA = (64 query rows, KV head g).  A row is a (query token, query head)
//    pair: the CTA takes 64 / G tokens x the G query heads of the group, so
//    every K/V byte a CTA stages serves all G heads.  Four consumer warps own
//    16 rows each; a fifth warp is the producer.
//  * K and V go through shared memory in tiles of 64 keys (4 pages), a
//    3-stage ring filled by TMA tensor copies: one 3-D copy per page, box
//    [64 elements, 16 rows, D/64 halves] of a tensor map over the pool, with
//    128-byte swizzle.  The layout that lands in shared memory is [half][row]
//    of 128-byte lines, so the 8 rows of every 8x8 ldmatrix block sit in 8
//    different bank groups.  Pages past the chunk's last key are requested at
//    a row beyond the pool: TMA fills them with zeros.
//  * S = Q K^T and O += P V with mma.sync m16n8k16 (bf16 in, fp32 accumulate);
//    Q stays in registers as A fragments, K and V fragments come from
//    ldmatrix (V transposed), and the S accumulators of two 8-key tiles are
//    repacked in registers as the A fragment of P (bf16) for P V.
//  * Online softmax in base 2 per row, causal mask per (row, key); the row
//    sum is kept per lane and reduced over the quad at the end.
#include <cuda.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "xs_common.cuh"

namespace xs {
namespace pftc {

constexpr int kBlock = 16;
constexpr int kConsumers = 4;
constexpr int kThreads = 32 * (kConsumers + 1);
constexpr int kKeys = 64;  // keys per tile
constexpr int kPagesPerTile = kKeys / kBlock;
constexpr int kStages = 3;
constexpr int kRows = 16 * kConsumers;  // query rows per CTA
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kWaitLimitNs = 4000000000ull;

template <int D>
struct TCfg {
    static constexpr int kHalves = D / 64;
    static constexpr int kPageBytes = kBlock * D * 2;  // bf16
    static constexpr int kTileBytes = kPagesPerTile * kPageBytes;
    static constexpr int kStageBytes = 2 * kTileBytes;  // K tile, then V tile
    static constexpr int kRingBytes = kStages * kStageBytes;
    // ring (1024-aligned for the 128-byte swizzle) + barriers + alignment slack
    static constexpr int kSmemBytes = kRingBytes + 2 * kStages * 8 + 1024;
};

struct PParams {
    __nv_bfloat16 *out;            // [T, Hq, D]
    const __nv_bfloat16 *q;        // [T, Hq, D]
    const int32_t *block_ids;      // [n_ids]
    int n_ids, T, start, Hq, Hkv;
    int64_t num_blocks;
    int oob_row;                   // a row coordinate past the pool: zero-filled pages
    float qscale;                  // scale * log2(e)
    int *err_flag;
};

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                            uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                                  uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// d = a (16x16, row) * b (16x8, col) + d; bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *tm, int x, int y,
                                            int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

// Shared-memory address of (key, dims d .. d+7) in a tile staged by TMA:
// page key/16, line (d/64) * 16 + key%16 of 128 bytes, 16-byte chunk
// (d%64)/8 stored at chunk ^ (line % 8) (the 128-byte swizzle; tile bases are
// 1024-byte aligned, so the line index is the address's swizzle phase).
template <int D>
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int key, int d) {
    const int line = (d >> 6) * kBlock + (key & 15);
    return base + (key >> 4) * TCfg<D>::kPageBytes + line * 128 +
           ((((d & 63) >> 3) ^ (line & 7)) << 4);
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 2)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const PParams p) {
    using C = TCfg<D>;
    constexpr int kTq = kRows / G;  // query tokens per CTA
    extern __shared__ unsigned char smem_raw[];
    unsigned char *ring = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + C::kRingBytes);
    uint64_t *empty = full + kStages;
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = blockIdx.y;
    const int tok0 = blockIdx.x * kTq;
    const int ntok = min(kTq, p.T - tok0);
    const int kmax = p.start + tok0 + ntok;  // keys [0, kmax) are read
    const int ntiles = (kmax + kKeys - 1) / kKeys;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumers);
        }
        mbar_fence_init();
        s_abort = 0;
    }
    __syncthreads();

    if (warp == kConsumers) {
        // ============================================================ producer
        const int npages = (kmax + kBlock - 1) / kBlock;
        int issued = 0;
        for (int kt = 0; kt < ntiles; ++kt) {
            const int s = kt % kStages;
            const uint32_t ph = (kt / kStages) & 1;
            int row = p.oob_row;
            const int pg = kt * kPagesPerTile + lane;
            if (lane < kPagesPerTile && pg < npages) {
                const int32_t blk = p.block_ids[pg];
                if (blk < 0 || blk >= p.num_blocks)
                    raise_flag(p.err_flag, XS_FLAG_BAD_BLOCK);  // read as zeros
                else
                    row = (blk * p.Hkv + g) * kBlock;
            }
            bool ok = true;
            if (lane == 0) {
                ok = mbar_wait_bounded(&empty[s], ph ^ 1, kWaitLimitNs);
                if (ok) mbar_arrive_expect_tx(&full[s], C::kStageBytes);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) {
                    raise_flag(p.err_flag, XS_FLAG_TIMEOUT);
                    atomicExch(&s_abort, 1);
                }
                break;
            }
            if (lane < kPagesPerTile) {
                const uint32_t kdst = smem_addr(ring + s * C::kStageBytes + lane * C::kPageBytes);
                tma_load_3d(kdst, &tmk, 0, row, 0, &full[s]);
                tma_load_3d(kdst + C::kTileBytes, &tmv, 0, row, 0, &full[s]);
            }
            ++issued;
        }
        // Let every copy this CTA issued land before it can exit.
        if (lane == 0) {
            for (int kt = max(0, issued - kStages); kt < issued; ++kt)
                mbar_wait_bounded(&full[kt % kStages], (kt / kStages) & 1, kWaitLimitNs);
        }
        return;
    }

    // ================================================================ consumers
    const int group = lane >> 2, tq = lane & 3;
    const int r0 = 16 * warp + group, r1 = r0 + 8;  // this lane's two rows
    const int i0 = r0 % kTq, j0 = r0 / kTq, i1 = r1 % kTq, j1 = r1 / kTq;
    const bool v0 = i0 < ntok, v1 = i1 < ntok;
    const int qpos0 = p.start + tok0 + i0, qpos1 = p.start + tok0 + i1;
    const __nv_bfloat16 *q0 =
        p.q + (static_cast<int64_t>(tok0 + (v0 ? i0 : 0)) * p.Hq + g * G + j0) * D;
    const __nv_bfloat16 *q1 =
        p.q + (static_cast<int64_t>(tok0 + (v1 ? i1 : 0)) * p.Hq + g * G + j1) * D;

    uint32_t qa[D / 16][4];
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const int d = 16 * ks + 2 * tq;
        qa[ks][0] = v0 ? *reinterpret_cast<const uint32_t *>(q0 + d) : 0u;
        qa[ks][1] = v1 ? *reinterpret_cast<const uint32_t *>(q1 + d) : 0u;
        qa[ks][2] = v0 ? *reinterpret_cast<const uint32_t *>(q0 + d + 8) : 0u;
        qa[ks][3] = v1 ? *reinterpret_cast<const uint32_t *>(q1 + d + 8) : 0u;
    }
    float oacc[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
#pragma unroll
        for (int c = 0; c < 4; ++c) oacc[n][c] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    // ldmatrix lane roles: matrix mi = lane / 8, row ri = lane % 8 of it.
    const int mi = lane >> 3, ri = lane & 7;
    bool ok = true;
    for (int kt = 0; kt < ntiles; ++kt) {
        const int s = kt % kStages;
        if (!__all_sync(0xffffffffu,
                        mbar_wait_bounded(&full[s], (kt / kStages) & 1, kWaitLimitNs)) ||
            *static_cast<volatile int *>(&s_abort)) {
            ok = false;
            break;
        }
        const uint32_t kbase = smem_addr(ring + s * C::kStageBytes);
        const uint32_t vbase = kbase + C::kTileBytes;

        // ---- S = Q K^T: 8 tiles of 8 keys
        float sacc[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int c = 0; c < 4; ++c) sacc[n][c] = 0.f;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(tile_addr<D>(kbase, 16 * np + ((mi >> 1) << 3) + ri,
                                         16 * ks + ((mi & 1) << 3)),
                            b0, b1, b2, b3);
                mma_bf16(sacc[2 * np], qa[ks], b0, b1);
                mma_bf16(sacc[2 * np + 1], qa[ks], b2, b3);
            }

        // ---- causal mask, online softmax (base 2)
        const int kb = kt * kKeys + 2 * tq;
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const int k = kb + 8 * n;
            sacc[n][0] = k <= qpos0 ? sacc[n][0] * p.qscale : -INFINITY;
            sacc[n][1] = k + 1 <= qpos0 ? sacc[n][1] * p.qscale : -INFINITY;
            sacc[n][2] = k <= qpos1 ? sacc[n][2] * p.qscale : -INFINITY;
            sacc[n][3] = k + 1 <= qpos1 ? sacc[n][3] * p.qscale : -INFINITY;
            mx0 = fmaxf(mx0, fmaxf(sacc[n][0], sacc[n][1]));
            mx1 = fmaxf(mx1, fmaxf(sacc[n][2], sacc[n][3]));
        }
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        // A row with nothing unmasked yet keeps reference 0 (no -inf - -inf).
        const float ref0 = mn0 == -INFINITY ? 0.f : mn0, ref1 = mn1 == -INFINITY ? 0.f : mn1;
        const float corr0 = fast_exp2(m0 - ref0), corr1 = fast_exp2(m1 - ref1);
        m0 = mn0;
        m1 = mn1;
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            sacc[n][0] = fast_exp2(sacc[n][0] - ref0);
            sacc[n][1] = fast_exp2(sacc[n][1] - ref0);
            sacc[n][2] = fast_exp2(sacc[n][2] - ref1);
            sacc[n][3] = fast_exp2(sacc[n][3] - ref1);
            ps0 += sacc[n][0] + sacc[n][1];
            ps1 += sacc[n][2] + sacc[n][3];
        }
        l0 = l0 * corr0 + ps0;
        l1 = l1 * corr1 + ps1;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
            oacc[n][0] *= corr0;
            oacc[n][1] *= corr0;
            oacc[n][2] *= corr1;
            oacc[n][3] *= corr1;
        }

        // ---- O += P V: 4 steps of 16 keys, D/8 tiles of 8 dims.  In the
        // last tile, V rows of keys >= kmax (unwritten slots of the last page:
        // any bits at all) are zeroed in the fragments, since 0 * NaN = NaN.
        const bool last = (kt + 1) * kKeys > kmax;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int kq = kt * kKeys + 16 * kk + 2 * tq;
            const uint32_t mlo = last ? ((kq < kmax ? 0xffffu : 0u) | (kq + 1 < kmax ? 0xffff0000u : 0u))
                                      : 0xffffffffu;
            const uint32_t mhi = last ? ((kq + 8 < kmax ? 0xffffu : 0u) |
                                         (kq + 9 < kmax ? 0xffff0000u : 0u))
                                      : 0xffffffffu;
            const uint32_t pa[4] = {pack_bf16(sacc[2 * kk][0], sacc[2 * kk][1]),
                                    pack_bf16(sacc[2 * kk][2], sacc[2 * kk][3]),
                                    pack_bf16(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]),
                                    pack_bf16(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3])};
#pragma unroll
            for (int dn = 0; dn < D / 16; ++dn) {
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4_trans(tile_addr<D>(vbase, 16 * kk + ((mi & 1) << 3) + ri,
                                               16 * dn + ((mi >> 1) << 3)),
                                  b0, b1, b2, b3);
                mma_bf16(oacc[2 * dn], pa, b0 & mlo, b1 & mhi);
                mma_bf16(oacc[2 * dn + 1], pa, b2 & mlo, b3 & mhi);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (!ok) {
        if (lane == 0) {
            raise_flag(p.err_flag, XS_FLAG_TIMEOUT);
            atomicExch(&s_abort, 1);
        }
        return;
    }

    // ---- out = O / l (the row sum over the quad's lanes)
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    __nv_bfloat16 *o0 = p.out + (static_cast<int64_t>(tok0 + i0) * p.Hq + g * G + j0) * D;
    __nv_bfloat16 *o1 = p.out + (static_cast<int64_t>(tok0 + i1) * p.Hq + g * G + j1) * D;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
        const int d = 8 * n + 2 * tq;
        if (v0) *reinterpret_cast<uint32_t *>(o0 + d) = pack_bf16(oacc[n][0] * inv0, oacc[n][1] * inv0);
        if (v1) *reinterpret_cast<uint32_t *>(o1 + d) = pack_bf16(oacc[n][2] * inv1, oacc[n][3] * inv1);
    }
}

// ------------------------------------------------------------------ host side

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                              const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                              const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
EncodeFn encode_fn() {
    static std::once_flag once;
    static EncodeFn fn = nullptr;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(ptr);
        cudaGetLastError();
    });
    return fn;
}

// Tensor map over a pool [num_blocks, Hkv, 16, D] bf16 seen as 3-D
// (64 elements, num_blocks*Hkv*16 rows, D/64 halves) with box
// (64, 16, D/64): one box is one page of one head, landing as [half][row].
int encode_pool(CUtensorMap *tm, const void *pool, int64_t rows, int D) {
    EncodeFn fn = encode_fn();
    if (!fn) return XS_EDEVICE;
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(D / 64)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, 128};
    const cuuint32_t box[3] = {64, kBlock, static_cast<cuuint32_t>(D / 64)};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(pool), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? XS_OK : XS_EUNSUPPORTED;
}

using KernelFn = void (*)(const CUtensorMap, const CUtensorMap, const PParams);

template <int D, int G>
KernelFn kernel_for() {
    return prefill_tc_kernel<D, G>;
}

KernelFn pick(int D, int G) {
    if (D == 128) {
        if (G == 1) return kernel_for<128, 1>();
        if (G == 2) return kernel_for<128, 2>();
        if (G == 4) return kernel_for<128, 4>();
        if (G == 8) return kernel_for<128, 8>();
    } else if (D == 64) {
        if (G == 1) return kernel_for<64, 1>();
        if (G == 2) return kernel_for<64, 2>();
        if (G == 4) return kernel_for<64, 4>();
        if (G == 8) return kernel_for<64, 8>();
    }
    return nullptr;
}

}  // namespace pftc
}  // namespace xs

using namespace xs;

extern "C" int xs_paged_prefill_tc(void *out, const void *q, const void *k_cache,
                                   const void *v_cache, const int32_t *block_ids, int n_ids,
                                   int T, int start_pos, int Hq, int Hkv, int D, int block_size,
                                   int64_t num_blocks, float scale, int dtype, int *err_flag,
                                   cudaStream_t stream) {
    if (!out || !q || !k_cache || !v_cache || !block_ids) return XS_ENULL;
    if (dtype != XS_BF16) return dtype == XS_F32 ? XS_EUNSUPPORTED : XS_EDTYPE;
    if (T < 0 || start_pos < 0 || n_ids < 0 || Hq <= 0 || Hkv <= 0 || num_blocks < 0 ||
        Hq % Hkv != 0)
        return XS_ESHAPE;
    const int G = Hq / Hkv;
    if (block_size != pftc::kBlock || (D != 64 && D != 128) ||
        (G != 1 && G != 2 && G != 4 && G != 8))
        return XS_EUNSUPPORTED;
    if (static_cast<int64_t>(start_pos) + T > static_cast<int64_t>(n_ids) * block_size)
        return XS_ESHAPE;
    const int64_t rows = num_blocks * Hkv * pftc::kBlock;
    if (rows + pftc::kBlock > 0x7fffffff) return XS_EUNSUPPORTED;  // 32-bit TMA row coordinate
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return XS_EALIGN;
    if (T == 0 || num_blocks == 0) return XS_OK;
    pftc::KernelFn fn = pftc::pick(D, G);
    if (!fn) return XS_EUNSUPPORTED;
    CUtensorMap tmk, tmv;
    int st = pftc::encode_pool(&tmk, k_cache, rows, D);
    if (st == XS_OK) st = pftc::encode_pool(&tmv, v_cache, rows, D);
    if (st != XS_OK) return st;
    const int smem = D == 128 ? pftc::TCfg<128>::kSmemBytes : pftc::TCfg<64>::kSmemBytes;
    static std::mutex mu;
    static pftc::KernelFn raised[8] = {};
    {
        std::lock_guard<std::mutex> lock(mu);
        bool done = false;
        for (pftc::KernelFn f : raised) done |= f == fn;
        if (!done) {
            if (cudaFuncSetAttribute(reinterpret_cast<const void *>(fn),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
                cudaSuccess) {
                cudaGetLastError();
                return XS_ELAUNCH;
            }
            for (pftc::KernelFn &f : raised)
                if (!f) {
                    f = fn;
                    break;
                }
        }
    }
    pftc::PParams p;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.block_ids = block_ids;
    p.n_ids = n_ids;
    p.T = T;
    p.start = start_pos;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.num_blocks = num_blocks;
    p.oob_row = static_cast<int>(rows);
    p.qscale = scale * pftc::kLog2e;
    p.err_flag = err_flag;
    const int tq = pftc::kRows / G;
    dim3 grid((T + tq - 1) / tq, Hkv);
    fn<<<grid, pftc::kThreads, smem, stream>>>(tmk, tmv, p);
    return launch_status();
}
