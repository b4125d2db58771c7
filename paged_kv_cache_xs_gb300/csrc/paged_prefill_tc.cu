// Chunked-prefill attention on the 5th-generation tensor cores: a T-token
// chunk at positions start_pos .. start_pos + T - 1 attends causally to every
// cached token of its sequence, gathered through the chunk's block list
// ("xserv compare phase10...cf1e9e4", attention.rs, attention /
// apply_causal_mask / flash_attention: softmax(scale * Q K^T + causal mask) V
// with the mask offset by the cached prefix).
//
// Design (flash-attention style, one pass, no split):
//  * CTA = two Q tiles of 128 query rows, one KV head g, one CTA per SM.  A
//    row is a (query token, query head) pair: 128 / G tokens x the G query
//    heads of the group, so every K/V byte staged serves all G heads of both
//    tiles.  Row r of tile i is TMEM lane r of tile i's 256 columns.
//  * Warps 0 and 3 (TMA): warp 0 copies Q once (one 3-D tensor copy per
//    tile and 64-wide D half, box [64, G heads, 128/G tokens]) and the
//    128-key K tiles (8 pages), warp 3 the V tiles, each into its own 2-slot
//    ring as soon as a slot is free (a K slot frees after both tiles'
//    Q K^T, a V slot after the step's last P V), one 3-D copy per page and
//    D half from a tensor map over the pool.  Every box is 128-byte swizzled, so a D half of a tile is the
//    canonical K-major layout (8-row groups 1024 B apart).  Pages past the
//    last key are requested at a row beyond the pool and arrive as zeros.
//  * Warp 1 (one thread): S = Q K^T with tcgen05.mma (M=128, N=128, K=16 per
//    instruction, A and B from shared-memory descriptors, fp32 accumulators
//    in TMEM); O += P V (M=128, N=D) with P read from TMEM (A operand) and V
//    as an MN-major B descriptor (8-key groups 1024 B apart, D halves one
//    tile-half apart); tcgen05.commit signals each step on an mbarrier.  The
//    softmax writes P (bf16) over the first half of S's columns, so per tile
//    the thread issues P V(t) and then S(t + 1) into the same columns - the
//    tensor pipe runs a thread's MMAs in order - and the two Q tiles
//    alternate: while one tile's softmax works, the tensor cores run the
//    other tile's P V and next scores.  A 128 x 128 x 16 MMA is 64 cycles
//    of tensor pipe and about as long for one thread to issue, and every
//    barrier wait in that thread leaves the pipe idle for ~300 cycles, so
//    it waits for P alone (the softmax checks that V(t) and K(t + 1) have
//    landed before publishing P) and builds its descriptors once.  (With
//    64-key tiles, one Q tile and
//    two CTAs per SM, each Q K^T instruction read 6 KB of shared-memory
//    operands for 128 x 64 x 16 MACs: 681 / 825 TFLOP/s on the 8K / 32K
//    chunked prefills; 128-key tiles read 8 KB for twice the MACs: 809 / 986.)
//  * Warp 2 idle.  Warpgroup 0 gives up registers to the softmax
//    warpgroups with setmaxnreg (kRegsCtl a thread there, kRegsSoftmax in
//    the softmax), so nothing spills at D = 128.
//  * Warps 4-11 (softmax, four per Q tile; warp w reads TMEM lanes
//    32*(w%4)..+31, one row per thread): load the row of S, causal mask
//    (diagonal tiles only), row max (8 chains of three-input maxima),
//    P = 2^(s - m) in base 2 (arguments and sums as packed fp32x2
//    operations), write P back to TMEM for the P V step.  The reference m only
//    moves when a tile's maximum exceeds it by more than 8 (log2 units), and
//    only then is the row of O in TMEM rescaled, so P stays <= 2^8 and most
//    tiles never touch O.  Unwritten slots of the last page (any bits at all)
//    are zeroed in the staged V tile, since 0 * NaN = NaN.  At the end:
//    O / l, bf16, out.
//  * TMEM: all 512 columns (per Q tile S/P 128, O 128).  Every wait is
//    bounded; the MMA thread waits for its last MMA before the CTA frees TMEM.
#include <cuda.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "xs_common.cuh"

namespace xs {
namespace pftc {

constexpr int kBlock = 16;
constexpr int kRows = 128;               // M: rows of one Q tile
constexpr int kQTiles = 2;               // Q tiles per CTA, one softmax warp group each
constexpr int kKeys = 128;               // keys per tile: N of Q K^T, K of P V
constexpr int kPagesPerTile = kKeys / kBlock;
constexpr int kStages = 2;               // depth of the K and V rings
// Warpgroup 0: the TMA warp, the MMA warp and two idle warps; then one
// warpgroup of 4 softmax warps per Q tile.
constexpr int kThreads = 128 + 128 * kQTiles;
// Registers a thread: at launch (65536 / kThreads, rounded down to 8), then
// moved from warpgroup 0 to the softmax warpgroups (setmaxnreg); the shares
// add up to the launch's total.
constexpr int kRegsLaunch = 168, kRegsCtl = 96, kRegsSoftmax = 200;
static_assert(128 * kRegsCtl + 128 * kQTiles * kRegsSoftmax <= kThreads * kRegsLaunch,
              "register split exceeds the launch's registers");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kGroupCols = 256;     // per Q tile: S 128 (P written over its first 64), O 128
constexpr uint32_t kColS = 0, kColP = 0, kColO = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kHeadroom = 8.f;         // log2 units P may exceed 1 before O is rescaled
constexpr uint64_t kWaitLimitNs = 4000000000ull;

template <int D>
struct TCfg {
    static constexpr int kHalves = D / 64;
    static constexpr int kQHalf = kRows * 128;      // one 64-wide D half of a Q tile
    static constexpr int kQTile = kHalves * kQHalf;
    static constexpr int kQBytes = kQTiles * kQTile;
    static constexpr int kKVHalf = kKeys * 128;     // one D half of a K or V tile
    static constexpr int kTile = kHalves * kKVHalf;
    // Separate rings for K and V tiles: a K slot frees when Q K^T of its tile
    // is done (for both Q tiles), long before P V of that tile, so K of the
    // next tiles streams in while the current ones are still in use.
    static constexpr int kKOff = kQBytes;
    static constexpr int kVOff = kQBytes + kStages * kTile;
    static constexpr int kBarOff = kQBytes + 2 * kStages * kTile;
    // q_full, k_full/k_empty/v_full/v_empty per stage, per Q tile s_full,
    // p_full, pv_done, then mma_idle and the TMEM address.
    static constexpr int kNumBars = 1 + 4 * kStages + 3 * kQTiles + 1;
    static constexpr int kBarBytes = (kNumBars + 1) * 8;
    static constexpr int kSmemBytes = kBarOff + kBarBytes + 1024;  // + alignment slack
    // Instruction descriptors (kind::f16): fp32 D, bf16 A and B, M = 128;
    // Q K^T: both K-major, N = 64; P V: B (V) MN-major, N = D.
    static constexpr uint32_t kIdS = (1u << 4) | (1u << 7) | (1u << 10) |
                                     (static_cast<uint32_t>(kKeys >> 3) << 17) |
                                     (static_cast<uint32_t>(kRows >> 4) << 24);
    static constexpr uint32_t kIdPV = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                                      (static_cast<uint32_t>(D >> 3) << 17) |
                                      (static_cast<uint32_t>(kRows >> 4) << 24);
};

struct PParams {
    __nv_bfloat16 *out;            // [T, Hq, D]
    const int32_t *block_ids;      // [n_ids]
    int n_ids;
    int T, start, Hq, Hkv;
    int64_t num_blocks;
    int oob_row;                   // a row coordinate past the pool: zero-filled pages
    float qscale;                  // scale * log2(e)
    int *err_flag;
    // Nonzero (XS_PREFILL_OVERLAP): q, the block ids and the key tiles that
    // end before position start are read before waiting for the previous
    // launch on the stream; the tiles from start on and every write after.
    int early;
};

// Shared-memory matrix descriptor: start, leading and stride byte offsets,
// descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((addr >> 4) & 0x3fff) |
           (static_cast<uint64_t>((lbo >> 4) & 0x3fff) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3fff) << 32) | (1ull << 46) | (2ull << 61);
}
__device__ __forceinline__ void umma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id, int acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
        "l"(a), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id,
                                        int acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d),
        "r"(a_tmem), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 32 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}
// Maximum of three (one instruction).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *tm, int x, int y,
                                            int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmq,
                      const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const PParams p) {
    using C = TCfg<D>;
    constexpr int kTq = kRows / G;  // query tokens per Q tile
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char *qs = sm;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::kBarOff);
    uint64_t *q_full = bars, *k_full = bars + 1, *k_empty = k_full + kStages;
    uint64_t *v_full = k_empty + kStages, *v_empty = v_full + kStages;
    // Per Q tile qi: s_full (S(t) is in TMEM: and, the tensor pipe being in
    // order, P V(t - 1) is done), p_full (P(t) is in TMEM), pv_done.
    uint64_t *grp0 = v_empty + kStages;
    auto s_full = [&](int qi) { return grp0 + 3 * qi; };
    auto p_full = [&](int qi) { return grp0 + 3 * qi + 1; };
    auto pv_done = [&](int qi) { return grp0 + 3 * qi + 2; };
    uint64_t *mma_idle = grp0 + 3 * kQTiles;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_idle + 1);
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Longest first: CTA i takes token tile (tiles - 1 - i / Hkv) of KV head
    // i % Hkv, so the CTAs with the most keys start in the first wave and the
    // launch ends on the short ones.
    const int n_tok_tiles = static_cast<int>(gridDim.x) / p.Hkv;
    const int g = static_cast<int>(blockIdx.x) % p.Hkv;
    const int tok0 = (n_tok_tiles - 1 - static_cast<int>(blockIdx.x) / p.Hkv) * kQTiles * kTq;
    const int ntok = min(kQTiles * kTq, p.T - tok0);  // tokens of this CTA
    const int kmax = p.start + tok0 + ntok;            // keys [0, kmax) are read
    const int ntiles = (kmax + kKeys - 1) / kKeys;
    const int npages = (kmax + kBlock - 1) / kBlock;
    // Q tile qi holds tokens [qi * kTq, qi * kTq + tile_tokens(qi)) of the CTA
    // and attends to key tiles [0, tile_ntiles(qi)).
    auto tile_tokens = [&](int qi) { return max(0, min(kTq, ntok - qi * kTq)); };
    auto tile_ntiles = [&](int qi) {
        const int n = tile_tokens(qi);
        return n > 0 ? (p.start + tok0 + qi * kTq + n + kKeys - 1) / kKeys : 0;
    };

    if (tid == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int qi = 0; qi < kQTiles; ++qi) {
            mbar_init(s_full(qi), 1);
            mbar_init(p_full(qi), 4);
            mbar_init(pv_done(qi), 1);
        }
        mbar_init(mma_idle, 1);
        mbar_fence_init();
        s_abort = 0;
    }
    if (warp == 1) {
        asm volatile(
            "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                smem_addr(tmem_slot)),
            "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto abort_now = [&]() {
        raise_flag(p.err_flag, XS_FLAG_TIMEOUT);
        atomicExch(&s_abort, 1);
    };
    auto aborted = [&]() { return *static_cast<volatile int *>(&s_abort) != 0; };

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtl));
        if (warp == 0 || warp == 3) {
            // ============================================================== TMA
            // Warp 0 loads Q and the K tiles, warp 3 the V tiles: each streams
            // its ring on its own, a tile as soon as its slot is free.
            const int which = warp == 3;  // 0: K, 1: V
            if (which == 0 && lane == 0) {
                mbar_arrive_expect_tx(q_full, C::kQBytes);
                for (int qi = 0; qi < kQTiles; ++qi)
                    for (int h = 0; h < C::kHalves; ++h)
                        tma_load_3d(smem_addr(qs + qi * C::kQTile + h * C::kQHalf), &tmq, 64 * h,
                                    g * G, tok0 + qi * kTq, q_full);
            }
            auto page_row = [&](int kt) {
                int row = p.oob_row;
                const int pg = kt * kPagesPerTile + lane;
                if (lane < kPagesPerTile && pg < npages && XS_BOUNDS(pg < p.n_ids, p.err_flag)) {
                    const int32_t blk = p.block_ids[pg];
                    if (blk < 0 || blk >= p.num_blocks)
                        raise_flag(p.err_flag, XS_FLAG_BAD_BLOCK);  // read as zeros
                    else
                        row = (blk * p.Hkv + g) * kBlock;
                }
                return row;
            };
            // With p.early, the first tile that holds a position from start on
            // (this chunk's rows, which the previous launch appends) waits for
            // that launch, and (warp 0) the next launch may start once it has.
            bool waited = !p.early;
            auto gate = [&](int kt) {
                if (!waited && (kt + 1) * kKeys > p.start) {
                    griddep_wait();
                    if (which == 0) griddep_launch_dependents();
                    waited = true;
                }
            };
            uint64_t *full = which ? v_full : k_full;
            uint64_t *empty = which ? v_empty : k_empty;
            auto issue = [&](int kt, int row) {
                gate(kt);
                const int s = kt % kStages;
                bool ok = true;
                if (lane == 0) {
                    ok = mbar_wait_bounded(&empty[s], ((kt / kStages) & 1) ^ 1, kWaitLimitNs) &&
                         !aborted();
                    if (ok) mbar_arrive_expect_tx(&full[s], C::kTile);
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (ok && lane < kPagesPerTile) {
                    unsigned char *base = sm + (which ? C::kVOff : C::kKOff) + s * C::kTile;
                    for (int h = 0; h < C::kHalves; ++h)
                        tma_load_3d(smem_addr(base + h * C::kKVHalf + lane * kBlock * 128),
                                    which ? &tmv : &tmk, 0, row, h, &full[s]);
                }
                return ok;
            };
            int issued = 0;
            bool ok = true;
            for (int kt = 0; ok && kt < ntiles; ++kt) {
                ok = issue(kt, page_row(kt));
                if (ok) ++issued;
            }
            if (!ok && lane == 0) abort_now();
            gate(ntiles);  // (every launch waits once, whatever it issued)
            // Let the copies this warp issued land before the CTA can exit.
            if (lane == 0) {
                if (which == 0) mbar_wait_bounded(q_full, 0, kWaitLimitNs);
                for (int kt = max(0, issued - kStages); kt < issued; ++kt)
                    mbar_wait_bounded(&full[kt % kStages], (kt / kStages) & 1, kWaitLimitNs);
            }
        } else if (warp == 1) {
            // ============================================================== MMA
            // Per Q tile the softmax writes P(t) over the first half of S(t) in
            // TMEM, so the MMA thread issues, per Q tile, P V(t) and then S(t + 1)
            // into the same columns: the tensor pipe executes a thread's MMAs in
            // order, so P V(t) has read P before S(t + 1) overwrites it, and when
            // S(t + 1) is complete so is P V(t).  The two Q tiles alternate: the
            // tensor cores run one tile's P V and next scores while the other
            // tile's softmax works.  One staged K or V tile serves both Q tiles.
            if (lane == 0) {
                const uint32_t qaddr = smem_addr(qs);
                int nt_q[kQTiles];
#pragma unroll
                for (int qi = 0; qi < kQTiles; ++qi) nt_q[qi] = tile_ntiles(qi);
                // Descriptors of the Q tiles and the K and V slots, built once:
                // an operand's start address is (address >> 4) in the low 14
                // bits, so a step within a tile adds (offset >> 4) (no carry:
                // shared addresses stay below 256 KB).
                uint64_t dq[kQTiles], dk[kStages], dv[kStages];
#pragma unroll
                for (int qi = 0; qi < kQTiles; ++qi)
                    dq[qi] = smem_desc(qaddr + qi * C::kQTile, 16, 1024);
#pragma unroll
                for (int st = 0; st < kStages; ++st) {
                    dk[st] = smem_desc(smem_addr(sm + C::kKOff + st * C::kTile), 16, 1024);
                    dv[st] = smem_desc(smem_addr(sm + C::kVOff + st * C::kTile), C::kKVHalf, 1024);
                }
                static_assert(C::kQHalf == C::kKVHalf, "Q and K D-halves step alike");
                auto issue_s = [&](int qi, int kt) {
                    const uint64_t kd = (kt % kStages) ? dk[1] : dk[0];
                    const uint64_t qd = qi ? dq[1] : dq[0];
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint64_t off = static_cast<uint64_t>(
                            ((ks >> 2) * C::kQHalf + 32 * (ks & 3)) >> 4);
                        umma_ss(tmem + qi * kGroupCols + kColS, qd + off, kd + off, C::kIdS,
                                ks > 0);
                    }
                    umma_commit(s_full(qi));
                };
                auto issue_pv = [&](int qi, int kt) {
                    const uint64_t vd = (kt % kStages) ? dv[1] : dv[0];
                    const uint32_t cols = tmem + qi * kGroupCols;
#pragma unroll
                    for (int kk = 0; kk < kKeys / 16; ++kk)
                        umma_ts(cols + kColO, cols + kColP + 8 * kk,
                                vd + static_cast<uint64_t>((2048 * kk) >> 4), C::kIdPV,
                                kt > 0 || kk > 0);
                    umma_commit(pv_done(qi));
                };
                bool ok = ntiles == 0 || (mbar_wait_bounded(q_full, 0, kWaitLimitNs) &&
                                          mbar_wait_bounded(&k_full[0], 0, kWaitLimitNs));
                if (ok && ntiles > 0) {
                    tc_fence_after();
                    for (int qi = 0; qi < kQTiles; ++qi)
                        if (nt_q[qi] > 0) issue_s(qi, 0);
                    umma_commit(&k_empty[0]);
                }
                // V(kt) and K(kt + 1) have landed once P(kt) is published.  A
                // V slot is released after the step's last P V, before that
                // tile's next scores; a K slot after both tiles' S(kt + 1).
                for (int kt = 0; ok && kt < ntiles; ++kt) {
                    const int s = kt % kStages, s1 = (kt + 1) % kStages;
                    const int last_v = kt < nt_q[kQTiles - 1] ? kQTiles - 1 : 0;
                    bool k_used = false;
                    for (int qi = 0; ok && qi < kQTiles; ++qi) {
                        if (kt >= nt_q[qi]) continue;
                        ok = mbar_wait_bounded(p_full(qi), kt & 1, kWaitLimitNs) && !aborted();
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv(qi, kt);
                        if (qi == last_v) umma_commit(&v_empty[s]);
                        if (kt + 1 < nt_q[qi]) {
                            issue_s(qi, kt + 1);
                            k_used = true;
                        }
                    }
                    if (!ok) break;
                    if (k_used) umma_commit(&k_empty[s1]);
                }
                if (!ok) abort_now();
                // Every MMA issued has completed before the CTA leaves (and TMEM is freed).
                umma_commit(mma_idle);
                mbar_wait_bounded(mma_idle, 0, kWaitLimitNs);
            }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        // ========================================================== softmax
        const int qi = (warp - 4) >> 2;    // Q tile of this warp group
        const int quad = warp & 3;         // TMEM lanes 32 * quad .. + 31 (warp rank in its warpgroup)
        const int r = 32 * quad + lane;    // this thread's row = TMEM lane
        const int tl = qi * kTq + r / G;   // query token within the CTA
        const bool valid = r / G < tile_tokens(qi);
        const int qpos = p.start + tok0 + tl;
        const int my_ntiles = tile_ntiles(qi);
        const uint32_t lane_off = static_cast<uint32_t>(32 * quad) << 16;
        const uint32_t cols = tmem + lane_off + qi * kGroupCols;
        float m_ref = 0.f, l = 0.f;
        bool ok = true;
        for (int kt = 0; kt < my_ntiles; ++kt) {
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(s_full(qi), kt & 1, kWaitLimitNs)) &&
                 !aborted();
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(cols + kColS + 32 * c, sr[c]);
            tmem_wait_ld();

            // Causal mask (by selection: a masked slot may hold any bits) - only
            // tiles that reach past the Q tile's first query position need one.
            // The maximum is taken on raw scores (qscale > 0), the exponent
            // is one fma: 2^(s * qscale - m).  Maximum and sums run as 8
            // independent chains.
            const int k0 = kt * kKeys;
            const bool need_mask = k0 + kKeys - 1 > p.start + tok0 + qi * kTq;
            float v[kKeys];
#pragma unroll
            for (int j = 0; j < kKeys; ++j) v[j] = __uint_as_float(sr[j >> 5][j & 31]);
            if (need_mask) {
#pragma unroll
                for (int j = 0; j < kKeys; ++j) v[j] = k0 + j <= qpos ? v[j] : -INFINITY;
            }
            // Row maximum: 8 independent chains of three-input maxima.
            float mx8[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) mx8[c] = fmaxf(v[c], v[c + 8]);
#pragma unroll
            for (int base = 16; base < kKeys; base += 16)
#pragma unroll
                for (int c = 0; c < 8; ++c) mx8[c] = fmax3(mx8[c], v[base + c], v[base + 8 + c]);
            const float tmax = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                                     fmaxf(mx8[6], mx8[7])) *
                               p.qscale;
            bool rescale = false;
            float m_new = m_ref;
            if (kt == 0) {
                m_ref = tmax == -INFINITY ? 0.f : tmax;
                m_new = m_ref;
            } else if (tmax > m_ref + kHeadroom) {
                rescale = true;
                m_new = tmax;
            }
            // 2^(s * qscale - m) for key pairs: the arguments as packed fp32x2
            // fmas, the sums as 4 packed chains.
            const float2 qs2 = make_float2(p.qscale, p.qscale), nm2 = make_float2(-m_new, -m_new);
            float2 ps4[4];
            uint32_t pr[kKeys / 2];
#pragma unroll
            for (int j = 0; j < kKeys / 2; ++j) {
                const float2 t = __ffma2_rn(make_float2(v[2 * j], v[2 * j + 1]), qs2, nm2);
                const float2 e = make_float2(fast_exp2(t.x), fast_exp2(t.y));
                ps4[j & 3] = j < 4 ? e : __fadd2_rn(ps4[j & 3], e);
                pr[j] = pack_bf16(e.x, e.y);
            }
            const float2 s01 = __fadd2_rn(__fadd2_rn(ps4[0], ps4[1]), __fadd2_rn(ps4[2], ps4[3]));
            const float ps = s01.x + s01.y;
            // A rescale reads and writes O: P V(t - 1) is done (S(t) was issued after it).
            if (__any_sync(0xffffffffu, rescale)) {
                const float corr = rescale ? fast_exp2(m_ref - m_new) : 1.f;
                l *= corr;
#pragma unroll 1
                for (int c = 0; c < D; c += 32) {
                    uint32_t o[32];
                    tmem_ld32(cols + kColO + c, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        o[j] = __float_as_uint(__uint_as_float(o[j]) * corr);
                    tmem_st32(cols + kColO + c, o);
                }
                if (rescale) m_ref = m_new;
            }
            l += ps;
            // P over the first half of S's columns.
            tmem_st32(cols + kColP, *reinterpret_cast<uint32_t(*)[32]>(&pr[0]));
            tmem_st32(cols + kColP + 32, *reinterpret_cast<uint32_t(*)[32]>(&pr[32]));
            tmem_wait_st();
            if (kt == ntiles - 1 && npages * kBlock > kmax) {
                // Unwritten slots of the CTA's last page: zero their V rows
                // (128-byte lines, whole, so the swizzle inside a line does not
                // matter), once the V tile has landed.  (Both Q tiles may end
                // on this tile; each writes the same zeros before its P V.)
                ok = __all_sync(0xffffffffu,
                                mbar_wait_bounded(&v_full[kt % kStages], (kt / kStages) & 1,
                                                  kWaitLimitNs));
                if (!ok) break;
                unsigned char *vt = sm + C::kVOff + (kt % kStages) * C::kTile;
                const int first = kmax - k0, nrow = npages * kBlock - kmax;
                for (int i = r; i < nrow * C::kHalves * 8; i += kRows) {
                    const int line = i >> 3, chunk = i & 7;
                    const int key = first + line % nrow, h = line / nrow;
                    *reinterpret_cast<uint4 *>(vt + h * C::kKVHalf + key * 128 + chunk * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_shared();
            }
            // The tiles this Q tile's next MMAs read, V(kt) and K(kt + 1), have
            // landed before P(kt) is published, so the MMA thread waits for P
            // alone: a barrier wait in the thread that issues the MMAs costs
            // ~300 cycles of an idle tensor pipe, even on a completed phase.
            // (Their copies were issued once every MMA that used the slots
            // before was complete, which S(kt) being here implies.)
            if (quad == 2) {
                bool landed = true;
                if (lane == 0)
                    landed = mbar_wait_bounded(&v_full[kt % kStages], (kt / kStages) & 1,
                                               kWaitLimitNs) &&
                             (kt + 1 >= my_ntiles ||
                              mbar_wait_bounded(&k_full[(kt + 1) % kStages],
                                                ((kt + 1) / kStages) & 1, kWaitLimitNs));
                ok = __all_sync(0xffffffffu, landed);
                if (!ok) break;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full(qi));
        }
        if (ok && my_ntiles > 0) {
            const int kt = my_ntiles - 1;
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(pv_done(qi), kt & 1, kWaitLimitNs));
            tc_fence_after();
        }
        if (p.early) griddep_wait();  // writes come after the previous launch (no-op otherwise)
        if (!ok) {
            if (lane == 0) abort_now();
        } else if (my_ntiles > 0) {
            // out = O / l for this row
            const float inv = l > 0.f ? 1.f / l : 0.f;
            __nv_bfloat16 *orow =
                p.out + (static_cast<int64_t>(tok0 + (valid ? tl : 0)) * p.Hq + g * G + r % G) * D;
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
                uint32_t o[32];
                tmem_ld32(cols + kColO + c, o);
                tmem_wait_ld();
                if (valid && XS_BOUNDS(tok0 + tl < p.T && (g + 1) * G <= p.Hq, p.err_flag)) {
#pragma unroll
                    for (int j = 0; j < 32; j += 8) {
                        uint4 w;
                        w.x = pack_bf16(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv);
                        w.y = pack_bf16(__uint_as_float(o[j + 2]) * inv,
                                        __uint_as_float(o[j + 3]) * inv);
                        w.z = pack_bf16(__uint_as_float(o[j + 4]) * inv,
                                        __uint_as_float(o[j + 5]) * inv);
                        w.w = pack_bf16(__uint_as_float(o[j + 6]) * inv,
                                        __uint_as_float(o[j + 7]) * inv);
                        *reinterpret_cast<uint4 *>(orow + c + j) = w;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols));
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

// A 3-D bf16 tensor map with 128-byte swizzle (zero fill outside the tensor).
int encode(CUtensorMap *tm, const void *base, const cuuint64_t (&dims)[3],
           const cuuint64_t (&strides)[2], const cuuint32_t (&box)[3]) {
    EncodeFn fn = encode_fn();
    if (!fn) return XS_EDEVICE;
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? XS_OK : XS_EUNSUPPORTED;
}

using KernelFn = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const PParams);

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
XS_DEFINE_BOUNDS_COUNTER(bounds_failures_prefill_tc)

}  // namespace xs

using namespace xs;

extern "C" int xs_paged_prefill_tc(void *out, const void *q, const void *k_cache,
                                   const void *v_cache, const int32_t *block_ids, int n_ids,
                                   int T, int start_pos, int Hq, int Hkv, int D, int block_size,
                                   int64_t num_blocks, float scale, int dtype, int *err_flag,
                                   cudaStream_t stream) {
    return xs_paged_prefill_tc_ex(out, q, k_cache, v_cache, block_ids, n_ids, T, start_pos, Hq,
                                  Hkv, D, block_size, num_blocks, scale, 0, dtype, err_flag,
                                  stream);
}

extern "C" int xs_paged_prefill_tc_ex(void *out, const void *q, const void *k_cache,
                                      const void *v_cache, const int32_t *block_ids, int n_ids,
                                      int T, int start_pos, int Hq, int Hkv, int D,
                                      int block_size, int64_t num_blocks, float scale, int flags,
                                      int dtype, int *err_flag, cudaStream_t stream) {
    if (flags & ~XS_PREFILL_OVERLAP) return XS_EUNSUPPORTED;
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
    // q [T, Hq, D] as (D, Hq, T), box (64, G, 128 / G): one D half of a CTA's rows.
    // Pools [num_blocks, Hkv, 16, D] as (64, rows, D / 64) with strides (2 D, 128)
    // bytes, box (64, 16, 1): one D half of one page.
    CUtensorMap tmq, tmk, tmv;
    const cuuint64_t qdims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hq),
                                 static_cast<cuuint64_t>(T)};
    const cuuint64_t qstr[2] = {static_cast<cuuint64_t>(D) * 2,
                                static_cast<cuuint64_t>(Hq) * D * 2};
    const cuuint32_t qbox[3] = {64, static_cast<cuuint32_t>(G),
                                static_cast<cuuint32_t>(pftc::kRows / G)};
    const cuuint64_t pdims[3] = {64, static_cast<cuuint64_t>(rows),
                                 static_cast<cuuint64_t>(D / 64)};
    const cuuint64_t pstr[2] = {static_cast<cuuint64_t>(D) * 2, 128};
    const cuuint32_t pbox[3] = {64, pftc::kBlock, 1};
    int st = pftc::encode(&tmq, q, qdims, qstr, qbox);
    if (st == XS_OK) st = pftc::encode(&tmk, k_cache, pdims, pstr, pbox);
    if (st == XS_OK) st = pftc::encode(&tmv, v_cache, pdims, pstr, pbox);
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
    p.early = (flags & XS_PREFILL_OVERLAP) ? 1 : 0;
    const int tq = pftc::kQTiles * pftc::kRows / G;  // query tokens per CTA
    const int64_t ctas = static_cast<int64_t>((T + tq - 1) / tq) * Hkv;
    if (ctas > 0x7fffffff) return XS_EUNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(pftc::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    if (p.early) {
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    if (cudaLaunchKernelEx(&cfg, fn, tmq, tmk, tmv, p) != cudaSuccess) {
        cudaGetLastError();
        return XS_ELAUNCH;
    }
    return launch_status();
}
