// Paged decode attention for GB300 (sm_103a): one query token per sequence
// attends over all of that sequence's K/V pages, gathered through its block
// table; query heads of a GQA group share every page read.
//
// Definition ("xserv compare phase10...cf1e9e4", crates/xserv-kernels/src/
// attention.rs, paged_decode_attention; "xserv compare phase5...phase9",
// docs/09-kv-cache.md, "After (with cache)"):
//     out[b,h,:] = sum_t softmax_t(scale * q[b,h,:] . K[b,t]) V[b,t]
// with K[b,t] = k_cache[block_tables[b][t/16], h/(Hq/Hkv), t%16, :].
//
// Design (flash-decoding, persistent, warp-specialised):
//  * Work item = (sequence b, KV head g, partition p of P tokens).  Items are
//    numbered by a per-CTA prefix sum over context_lens (item_counts,
//    decode_item) and taken by a persistent grid: the first two per CTA
//    statically, the rest from a device counter that the last CTA resets.
//  * Warp 0 is the producer: it reads block ids (32 at a time, coalesced) and
//    streams each page pair (K page + V page of head g, 16 tokens x D) into an
//    8-stage shared-memory ring completing on mbarriers - bf16 pages as 4-D
//    TMA tensor copies with the 128-byte swizzle, fp32 pages as 1-D bulk
//    copies - and stages the G query rows of each item in a double-buffered
//    q slot.  It claims the next item when a ring of the current one is left.
//  * Warps 1..4 are consumers.  Consumer c takes ring pages c, c+4, ... and
//    keeps its own online-softmax state (running max m, sum l, output o) for
//    all G heads.  bf16: Q K^T and P V with mma.sync m16n8k16 (the G heads as
//    the rows of A, the page's 16 keys as N), fragments by ldmatrix from the
//    swizzled page.  fp32: QK with 8 lanes per token and a reduce-scatter; PV
//    with each lane owning D/32 output dims.
//  * Warp 5 is the merger: it merges the four consumer states of each item
//    and writes the final output (single-partition sequence) or fp32
//    partials (o, m, l) for the split-K combine.
//  * One-launch step (xs_paged_decode_step): the item covering a sequence's
//    last page first writes this step's K/V row into its slot, and the
//    merger counts split items into their group; the item that completes a
//    group combines its partials (staged in shared memory by bulk copies)
//    into out.  With early reads, lengths, item tables, block ids and the
//    first pages are read before waiting on the previous launch (in a launch
//    of at most 16 rounds of items, the first item's next pages are also
//    prefetched into L2).
//  * Small one-launch steps (every (sequence, KV head) group in one wave of
//    thread-block clusters: a single stream, small batches) run a second
//    kernel instead, paged_decode_cluster_kernel: one cluster per group, CTA
//    r taking partition r, the split-K combine over distributed shared
//    memory after a cluster barrier (see its own comment).
//  * Logits are kept in base-2 units (q is pre-scaled by scale*log2(e)) so
//    exponentials are single ex2 instructions.
#include <cuda.h>

#include <algorithm>
#include <cstring>
#include <cmath>
#include <mutex>
#include <type_traits>

#include "tensor_map.h"
#include "xs_common.cuh"

namespace xs {
namespace attn {

constexpr int kBlock = 16;          // tokens per page
constexpr int kConsumerWarps = 4;
constexpr int kThreads = 32 * (kConsumerWarps + 2);  // producer, consumers, merger
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s per bounded wait
constexpr int kMaxBatch = 8192;                   // per-sequence tables live in shared memory
constexpr int kClaimAhead = 8;  // pages of the current item left to issue when the next is claimed
constexpr int kL2Ahead = 16;    // pages of the first item prefetched into L2 before the launch wait

// Limit of every bounded wait.  The debug library (XS_DEBUG_BOUNDS) makes it
// settable, and can make CTA 0's producer skip issuing the copies of one of
// its pages (xs_debug_wait_injection), so a test can make a consumer's wait
// for that page run out: nothing is in flight for the skipped page, so the
// abort path (flag, drain, return) runs with every copy accounted for.
#ifdef XS_DEBUG_BOUNDS
__device__ unsigned long long g_wait_limit_ns = kWaitLimitNs;
__device__ int g_skip_page = -1;  // CTA 0's page counter value whose copies are not issued
__device__ __forceinline__ uint64_t wait_limit() { return g_wait_limit_ns; }
__device__ __forceinline__ bool skip_page(uint32_t c) {
    return blockIdx.x == 0 && static_cast<int>(c) == g_skip_page;
}
#else
__device__ __forceinline__ constexpr uint64_t wait_limit() { return kWaitLimitNs; }
__device__ __forceinline__ constexpr bool skip_page(uint32_t) { return false; }
#endif

// Per-sequence tables a CTA keeps in shared memory: pfull[B + 1], ptail[B + 1]
// (item numbering) and nlen[B] (clamped context lengths).
__host__ __device__ constexpr int table_bytes(int B) { return 4 * (3 * B + 2); }

// S: stages of the page ring.  The default (8) leaves room for two or three
// resident CTAs per SM; the deep ring (16, one CTA per SM) serves launches
// with at most one work item per SM, whose whole first item then fits the
// ring before the launch wait.
constexpr int kRing = 2 * kConsumerWarps, kDeepRing = 4 * kConsumerWarps;
template <typename T, int D, int G, int S = kRing>
struct Cfg {
    static constexpr int kRowBytes = D * static_cast<int>(sizeof(T));
    static constexpr int kPageBytes = kBlock * kRowBytes;
    // Ring of page pairs.  Page c goes to stage c % kStages and to consumer
    // warp c % kConsumerWarps; kStages must be a multiple of kConsumerWarps so
    // every stage is only ever used by one warp.  Otherwise a warp could wait
    // for phase k of a stage whose phase k-1 (another warp's page) has not
    // completed yet, and a parity wait cannot tell phase k from phase k-2.
    static constexpr int kStages = S;
    static constexpr int kChunksPerRow = kRowBytes / 16;
    static constexpr int kChunksPerLane = kChunksPerRow / 8;   // QK: 8 lanes per token
    static constexpr int kElemsPerChunk = 16 / static_cast<int>(sizeof(T));
    static constexpr int kQkDims = kChunksPerLane * kElemsPerChunk;  // = D / 8
    static constexpr int kPvDims = D / 32;                           // PV dims per lane
    static constexpr int kPvBytes = kPvDims * static_cast<int>(sizeof(T));
    static constexpr int kQBytes = G * kRowBytes;
    static constexpr int kLogG = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3;
    static constexpr int kHeadShift = 3 - kLogG;  // lane j of a token group owns head j >> shift
    // Resident CTAs per SM the register budget is sized for.
    static constexpr int kMinBlocks =
        (G == 8 || S > kRing) ? 1 : ((2 * kPageBytes <= 4096) ? 3 : 2);
    // Shared memory carve-up (bytes).
    static constexpr int kRingBytes = kStages * 2 * kPageBytes;
    static constexpr int kQSlotOff = kRingBytes;
    static constexpr int kWOff = kQSlotOff + 2 * kQBytes;
    static constexpr int kWBytes = kConsumerWarps * kBlock * G * 8;   // (w, w) pairs
    static constexpr int kCombOff = kWOff + kWBytes;
    // A merge buffer: the item (32 B), then m[G][4], l[G][4] (each head's
    // four consumer values together), o[4][G][D] (fp32).
    static constexpr int kCombBytes = 32 + kConsumerWarps * G * (D + 2) * 4;  // one buffer
    static constexpr int kMergeBufs = 2;   // consumers run up to kMergeBufs - 1 items ahead
    static constexpr int kBarOff = (kCombOff + kMergeBufs * kCombBytes + 7) / 8 * 8;
    static constexpr int kBarBytes = (2 * kStages + 4 + 3 * kMergeBufs) * 8;
    static constexpr int kItemOff = kBarOff + kBarBytes;             // 2 published items
    static constexpr int kPrefixOff = kItemOff + 2 * 32;
    // The host sizes every launch with this same function.
    // bf16 pages arrive by TMA tensor copies in the 128-byte swizzled
    // [half][row] layout and feed bf16 mma; fp32 pages by 1-D bulk copies
    // and CUDA-core FMA.  The ring must then be 1024-byte aligned: 1024 bytes
    // of slack let the kernel align the dynamic shared memory base.
    static constexpr bool kMma = sizeof(T) == 2;
    static constexpr int kAlignSlack = 1024;
    static __host__ __device__ constexpr int smem_bytes(int B) {
        return kPrefixOff + table_bytes(B) + kAlignSlack;
    }
    static_assert(kStages % kConsumerWarps == 0, "each ring stage must belong to one consumer");
    static_assert((kMergeBufs & (kMergeBufs - 1)) == 0, "item counters wrap: a power of two");
    static_assert(kChunksPerLane >= 1 && kChunksPerRow % 8 == 0, "row must split over 8 lanes");
    static_assert(D % 64 == 0, "PV works on dim pairs: D must split over 32 lanes x 2");
    static_assert(kCombOff % 16 == 0 && kCombBytes % 16 == 0 && (kConsumerWarps * G * 4) % 16 == 0,
                  "merge buffers are read as float4");
};

struct Params {
    void *out;
    float *part_o, *part_m, *part_l;
    const void *q, *k_cache, *v_cache;
    const int32_t *block_tables, *context_lens;
    int max_blocks, B, Hq, Hkv, P, max_parts;
    int64_t num_blocks;
    float qscale;  // scale * log2(e)
    const void *sinks;  // [Hq] sink logits (q's dtype), or null
    int window;         // > 0: attend to the last `window` tokens only
    // Prefill mode (prefill_start >= 0): "sequence" b is query token b of one
    // chunk at position prefill_start + b, attending to prefill_start + b + 1
    // tokens through the one block list (table_stride 0); context_lens unused.
    int prefill_start;
    int table_stride;   // elements between block-table rows (max_blocks, or 0)
    int *err_flag;
    int *work;     // [2] item counter + finished-CTA counter (zero between launches), or null
    // Fused decode step (decode mode only).  k_new/v_new [B, Hkv, D]: this
    // step's rows, written into their slot by the item that covers the
    // sequence's last page before it loads that page; null = no append.
    const void *k_new, *v_new;
    // [B * Hkv] arrival counts (zero between launches): the last item of a
    // split sequence-head combines its partials into out; null = leave the
    // partials for the separate combine kernel.
    int *combine;
    // Shared memory after the per-sequence tables where the merger stages
    // partial rows for a combine: stage_parts partials (x G heads x D fp32)
    // per round trip; stage_bytes is what the launch added for it.
    int stage_bytes, stage_parts;
    // Nonzero: read lengths, tables and the first pages before waiting for
    // the previous launch on the stream (see the kernel's start).
    int early;
};

// Byte offset of the combine staging area (16-byte aligned, after the tables).
__host__ __device__ constexpr int stage_offset(int prefix_off, int B) {
    return (prefix_off + table_bytes(B) + 15) / 16 * 16;
}

// Number of tokens sequence b attends to, clamped to the table's reach.
__device__ __forceinline__ int seq_len(const Params &p, int b, bool report) {
    int n = p.prefill_start >= 0 ? p.prefill_start + b + 1 : p.context_lens[b];
    const int cap = p.max_blocks * kBlock;
    if (n > cap) {
        if (report) raise_flag(p.err_flag, XS_FLAG_BAD_LEN);
        n = cap;
    }
    return n;
}

struct Item {
    int b, g, part, nparts, tok0, tok1, pg0, pg1;
};
static_assert(sizeof(Item) == 32, "item slots and merge-buffer headers are 32 bytes");

// First token a sequence of n tokens attends to: the sliding window keeps
// the last p.window tokens (all of them when p.window is 0).
__device__ __forceinline__ int first_token(const Params &p, int n) {
    return (p.window > 0 && n > p.window) ? n - p.window : 0;
}

// Largest b in [0, B) with table[b] <= x (table is non-decreasing).
// Largest b in [0, B) with table[b] <= x, for a nondecreasing table with
// table[0] <= x, searched by the whole warp: each round the 32 lanes test
// the starts of 32 equal segments of the range and a ballot picks the last
// segment that starts at or below x (one round for B <= 32, two up to 1024).
__device__ __forceinline__ int upper_index(const int *table, int B, int x, int lane) {
    int lo = 0, n = B;  // search [lo, lo + n); table[lo] <= x throughout
    while (n > 32) {
        const int step = (n + 31) >> 5;
        const bool le = lane * step < n && table[lo + lane * step] <= x;
        const int seg = 31 - __clz(__ballot_sync(0xffffffffu, le));
        lo += seg * step;
        n = min(step, n - seg * step);
    }
    const bool le = lane < n && table[lo + lane] <= x;
    return lo + 31 - __clz(__ballot_sync(0xffffffffu, le));
}

// Item numbering: two classes of items, class A numbered before class B,
// each in sequence order; pfull/ptail hold the exclusive prefix sums of the
// per-sequence counts of class A and class B items (item_counts).
//
// Without the fused combine, A = every full partition (P tokens) of every
// sequence and KV head, B = the ragged last partitions (and short
// sequences): the end of a launch is made of small items that balance the
// grid.  With it, A = all items of the sequences split into more than one
// partition, group by group ((b, g) then the partition), and B = the
// sequences that fit one partition (one item per KV head, no combine).  The
// partitions of a group are taken back to back, finish together, and the
// group is combined while the rest of the grid still streams pages; the
// launch ends on single-partition items, which write their output directly.
__device__ __forceinline__ void item_counts(const Params &p, int nw, int &ca, int &cb) {
    if (p.combine) {
        const int np = (nw + p.P - 1) / p.P;
        ca = np > 1 ? np * p.Hkv : 0;
        cb = np == 1 ? p.Hkv : 0;
    } else {
        ca = (nw / p.P) * p.Hkv;
        cb = (nw % p.P != 0) * p.Hkv;
    }
}

__device__ __forceinline__ Item decode_item(const Params &p, const int *pfull, const int *ptail,
                                            const int *nlen, int item, int lane) {
    Item it;
    const int n_a = pfull[p.B];
    int b;
    if (item < n_a) {
        b = upper_index(pfull, p.B, item, lane);
        const int r = item - pfull[b];
        const int na = (pfull[b + 1] - pfull[b]) / p.Hkv;  // class-A items per KV head
        it.g = r / na;
        it.part = r - it.g * na;
    } else {
        const int j = item - n_a;
        b = upper_index(ptail, p.B, j, lane);
        it.g = j - ptail[b];
        it.part = p.combine ? 0 : (nlen[b] - first_token(p, nlen[b])) / p.P;
    }
    it.b = b;
    const int n = nlen[b], t0 = first_token(p, n);
    it.nparts = (n - t0 + p.P - 1) / p.P;
    it.tok0 = t0 + it.part * p.P;
    it.tok1 = min(n, it.tok0 + p.P);
    it.pg0 = it.tok0 / kBlock;
    it.pg1 = (it.tok1 + kBlock - 1) / kBlock;
    return it;
}

// Load kPvDims consecutive elements of a V row (one lane's share) as fp32.
template <typename T, int kPvDims>
__device__ __forceinline__ void load_v(const unsigned char *src, float *vf) {
    if constexpr (sizeof(T) == 2 && kPvDims == 2) {
        const uint32_t raw = *reinterpret_cast<const uint32_t *>(src);
        vf[0] = __uint_as_float(raw << 16);
        vf[1] = __uint_as_float(raw & 0xffff0000u);
    } else if constexpr (sizeof(T) == 2 && kPvDims == 4) {
        const uint2 raw = *reinterpret_cast<const uint2 *>(src);
        vf[0] = __uint_as_float(raw.x << 16);
        vf[1] = __uint_as_float(raw.x & 0xffff0000u);
        vf[2] = __uint_as_float(raw.y << 16);
        vf[3] = __uint_as_float(raw.y & 0xffff0000u);
    } else if constexpr (sizeof(T) == 4 && kPvDims == 2) {
        const float2 raw = *reinterpret_cast<const float2 *>(src);
        vf[0] = raw.x;
        vf[1] = raw.y;
    } else {
        static_assert(sizeof(T) == 4 && kPvDims == 4, "unsupported V row split");
        const float4 raw = *reinterpret_cast<const float4 *>(src);
        vf[0] = raw.x;
        vf[1] = raw.y;
        vf[2] = raw.z;
        vf[3] = raw.w;
    }
}

// One consumer warp folds one page (16 tokens of one KV head) into its
// online-softmax state; only tokens [t_lo, t_hi) of the page count.  kFull:
// all 16 are valid (every page but the first and last of a windowed or
// ragged range), which lets the PV loop unroll completely.
template <typename T, int D, int G, bool kFull>
__device__ __forceinline__ void consume_page(const unsigned char *Ks, const unsigned char *Vs,
                                             int t_lo, int t_hi, const float (&qf)[G][D / 8],
                                             float &m_own, float &l_own,
                                             float2 (&o)[G][D / 64], float2 *W2, int lane) {
    using C = Cfg<T, D, G>;
    const int tg = lane >> 3, j = lane & 7;
    const int own_head = j >> C::kHeadShift;

    // ---- QK: 4 passes x 4 tokens; lane (tg, j) covers dims of chunks j, j+8, ...
    float sc[4];
#pragma unroll
    for (int pass = 0; pass < 4; ++pass) {
        const int t = pass * 4 + tg;
        float2 acc[G];
#pragma unroll
        for (int h = 0; h < G; ++h) acc[h] = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < C::kChunksPerLane; ++c) {
            const uint4 raw =
                *reinterpret_cast<const uint4 *>(Ks + t * C::kRowBytes + (j + 8 * c) * 16);
            float f[C::kElemsPerChunk];
            unpack16(raw, f, static_cast<T *>(nullptr));
#pragma unroll
            for (int e = 0; e < C::kElemsPerChunk; e += 2) {
                const float2 kv = make_float2(f[e], f[e + 1]);
#pragma unroll
                for (int h = 0; h < G; ++h)
                    acc[h] = __ffma2_rn(make_float2(qf[h][c * C::kElemsPerChunk + e],
                                                    qf[h][c * C::kElemsPerChunk + e + 1]),
                                        kv, acc[h]);
            }
        }
        float v[G];
#pragma unroll
        for (int h = 0; h < G; ++h) v[h] = acc[h].x + acc[h].y;
        // Reduce-scatter over the 8 lanes of the token group: lane j keeps head j >> shift.
        int cnt = G;
#pragma unroll
        for (int mask = 4; mask >= 1; mask >>= 1) {
            if (cnt > 1) {
                const int half = cnt >> 1;
                const bool upper = (lane & mask) != 0;
#pragma unroll
                for (int i = 0; i < (G > 1 ? G / 2 : 1); ++i) {
                    if (i < half) {
                        const float send = upper ? v[i] : v[i + half];
                        const float keep = upper ? v[i + half] : v[i];
                        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
                    }
                }
                cnt = half;
            } else {
                v[0] += __shfl_xor_sync(0xffffffffu, v[0], mask);
            }
        }
        sc[pass] = (kFull || (t >= t_lo && t < t_hi)) ? v[0] : -INFINITY;
    }

    // ---- online softmax for head own_head (lanes sharing j agree)
    float pm = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 8));
    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
    const float m_new = fmaxf(m_own, pm);
    const float corr_own = fast_exp2(m_own - m_new);
    m_own = m_new;
    float w[4], ps = 0.f;
#pragma unroll
    for (int pass = 0; pass < 4; ++pass) {
        w[pass] = fast_exp2(sc[pass] - m_new);
        ps += w[pass];
    }
    ps += __shfl_xor_sync(0xffffffffu, ps, 8);
    ps += __shfl_xor_sync(0xffffffffu, ps, 16);
    l_own = l_own * corr_own + ps;
    if ((j & ((1 << C::kHeadShift) - 1)) == 0) {
#pragma unroll
        for (int pass = 0; pass < 4; ++pass)
            W2[(pass * 4 + tg) * G + own_head] = make_float2(w[pass], w[pass]);
    }
    float2 corr[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const float c = __shfl_sync(0xffffffffu, corr_own, h << C::kHeadShift);
        corr[h] = make_float2(c, c);
    }
    __syncwarp();

    // ---- PV: lane owns dims [lane*kPvDims, +kPvDims) of every head
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int d = 0; d < C::kPvDims / 2; ++d) o[h][d] = __fmul2_rn(o[h][d], corr[h]);
    const unsigned char *vrow = Vs + lane * C::kPvBytes;
    auto pv_token = [&](int t) {
        float vf[C::kPvDims];
        load_v<T, C::kPvDims>(vrow + t * C::kRowBytes, vf);
        const float2 *wt = W2 + t * G;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float2 wh = wt[h];
#pragma unroll
            for (int d = 0; d < C::kPvDims / 2; ++d)
                o[h][d] = __ffma2_rn(wh, make_float2(vf[2 * d], vf[2 * d + 1]), o[h][d]);
        }
    };
    if constexpr (kFull) {
#pragma unroll
        for (int t = 0; t < kBlock; ++t) pv_token(t);
    } else {
        for (int t = t_lo; t < t_hi; ++t) pv_token(t);
    }
    __syncwarp();
}

// Split-K combine of one split sequence-head group, run by one warp (the
// merger of the item that finished last): for each of the G heads,
//     out = sum_j 2^(m_j - M) l_j o_j / (sum_j 2^(m_j - M) l_j [+ sink term])
// with M = max_j m_j, over the nparts partials (o_j already divided by l_j).
// The partials were written by other CTAs of this launch: read through L2.
// Lane j holds m and l of partials j, j + 32, ... (one load round for up to
// 32 partials), the weights reach the other lanes by shuffles, and the
// partial rows are loaded 16 at a time, all G heads together.
// Store n consecutive output values (fp32 in, T out, round to nearest)
// with one vector store.
template <typename T, int n>
__device__ __forceinline__ void store_row(T *dst, const float *v) {
    if constexpr (sizeof(T) == 2) {
        static_assert(n == 2 || n == 4, "bf16 rows of 2 or 4 values");
        uint32_t w[n / 2];
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t *>(&b);
        }
        if constexpr (n == 4)
            *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[1]);
        else
            *reinterpret_cast<uint32_t *>(dst) = w[0];
    } else {
        static_assert(n == 2 || n == 4, "fp32 rows of 2 or 4 values");
        if constexpr (n == 4)
            *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
        else
            *reinterpret_cast<float2 *>(dst) = make_float2(v[0], v[1]);
    }
}

// The merger's staging area: an mbarrier, its phase, then the rows.
struct Stage {
    uint64_t bar;
    uint32_t phase;
    uint32_t pad;
    __device__ float *rows() { return reinterpret_cast<float *>(this + 1); }
};
static_assert(sizeof(Stage) == 16, "staged rows start 16 bytes in");

// The launch's dynamic shared memory.  Helpers that are not inlined take
// byte offsets into it (not pointers, which would be generic there), so their
// shared-memory accesses stay shared-memory accesses.
__device__ __forceinline__ unsigned char *dyn_smem() {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    return smem_raw;
}

// Split-K combine of one (sequence, KV head) group by one warp: for each of
// the G heads, out = sum_j e^(m_j - M) o_j / sum_j e^(m_j - M) l_j over the
// group's np partials (o_j already divided by l_j's partition sum, so the
// weight of o_j is e^(m_j - M) l_j).  Partials are taken in chunks, each
// one memory round trip: for each head, the first stage_parts partials of a
// chunk are contiguous in part_o and arrive in the staging area by one bulk
// copy (the copy engine, not the load unit); the first chunk also takes up
// to kRegParts more straight into registers, and lane k loads m and l of
// partial k, all in flight together.  The running maximum M is raised per
// chunk and what was accumulated is rescaled.  The caller has acquired the
// partials (generic proxy); the proxy fence below orders the bulk copies
// after that.  Returns false if a copy did not complete in time (nothing is
// written then).
template <typename T, int D, int G>
__device__ __noinline__ bool combine_partials(const Params &p, const Item &it, int64_t head0,
                                              int lane, int stage_off) {
    Stage *stage = reinterpret_cast<Stage *>(dyn_smem() + stage_off);
    constexpr int kDims = D / 32;   // output dims per lane
    using Vec = typename std::conditional<kDims == 4, float4, float2>::type;
    // 16 rows held in registers, where the register budget allows (not at
    // three resident CTAs per SM).
    constexpr int kRegParts = Cfg<T, D, G>::kMinBlocks >= 3 ? 0 : 16 / G;
    constexpr int kRegSlots = kRegParts > 0 ? kRegParts : 1;
    const int np = it.nparts;
    const int K = p.stage_parts;
    const float *pm = p.part_m + head0 * p.max_parts;
    const float *pl = p.part_l + head0 * p.max_parts;
    float *rows = stage->rows();
    if (!XS_BOUNDS(np >= 1 && np <= p.max_parts && head0 >= 0 &&
                       head0 + G <= static_cast<int64_t>(p.B) * p.Hq &&
                       static_cast<int>(sizeof(Stage)) + G * K * D * 4 <= p.stage_bytes,
                   p.err_flag))
        return true;  // (debug build) nothing read or written
    float acc[G][kDims], den[G], run_m[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        den[h] = 0.f;
        run_m[h] = -INFINITY;
#pragma unroll
        for (int d = 0; d < kDims; ++d) acc[h][d] = 0.f;
    }
    for (int j0 = 0; j0 < np;) {
        const int cnt = min(K, np - j0);  // staged partials
        // The first chunk's next partials (up to kRegParts, 32 in all) go to registers.
        const int nreg = j0 == 0 ? min(np - cnt, min(kRegParts, 32 - cnt)) : 0;
        Vec vr[kRegSlots][G];
#pragma unroll
        for (int u = 0; u < kRegParts; ++u)
#pragma unroll
            for (int h = 0; h < G; ++h)
                if (u < nreg)
                    vr[u][h] = __ldcg(reinterpret_cast<const Vec *>(
                        p.part_o + ((head0 + h) * p.max_parts + cnt + u) * D + lane * kDims));
        const int tot = cnt + nreg;  // partials of this chunk (<= 32: lane k holds k's m, l)
        // Row h * cnt + k of the staging area receives partial j0 + k of head h.
        const uint32_t phase = stage->phase;
        if (lane == 0) {
            fence_proxy_async_global();  // partials acquired above -> async-proxy reads
            fence_proxy_async_shared();  // last chunk's reads of the rows -> overwrite
            mbar_arrive_expect_tx(&stage->bar, static_cast<uint32_t>(G * cnt * D * 4));
#pragma unroll
            for (int h = 0; h < G; ++h)
                bulk_g2s(rows + h * cnt * D, p.part_o + ((head0 + h) * p.max_parts + j0) * D,
                         static_cast<uint32_t>(cnt * D * 4), &stage->bar);
        }
        // m and l of partial j0 + lane, all G heads in flight together; the
        // G maxima reduce side by side (independent shuffle chains).
        float mj[G], lj[G], cm[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            mj[h] = -INFINITY;
            lj[h] = 0.f;
            if (lane < tot) {
                mj[h] = __ldcg(pm + h * p.max_parts + j0 + lane);
                lj[h] = __ldcg(pl + h * p.max_parts + j0 + lane);
            }
            cm[h] = mj[h];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int h = 0; h < G; ++h) cm[h] = fmaxf(cm[h], __shfl_xor_sync(0xffffffffu, cm[h], o));
        float wgt[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float m_new = fmaxf(run_m[h], cm[h]);
            const float ref = m_new == -INFINITY ? 0.f : m_new;
            const float corr = fast_exp2(run_m[h] - ref);  // 0 while nothing is accumulated
            run_m[h] = m_new;
            wgt[h] = lane < tot ? fast_exp2(mj[h] - ref) * lj[h] : 0.f;
            den[h] = den[h] * corr + wgt[h];
#pragma unroll
            for (int d = 0; d < kDims; ++d) acc[h][d] *= corr;
        }
        // The register partials were requested first: fold them in while the
        // staged rows land.
#pragma unroll
        for (int u = 0; u < kRegParts; ++u)
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float w = __shfl_sync(0xffffffffu, wgt[h], (cnt + u) & 31);
                if (u < nreg) {
                    const float *f = reinterpret_cast<const float *>(&vr[u][h]);
#pragma unroll
                    for (int d = 0; d < kDims; ++d) acc[h][d] += w * f[d];
                }
            }
        const bool landed =
            __all_sync(0xffffffffu, mbar_wait_bounded(&stage->bar, phase, wait_limit()));
        __syncwarp();
        if (lane == 0) stage->phase = phase ^ 1u;
        if (!landed) {
            // The caller flags it; first give the copies in flight (bounded)
            // time to land, so none writes into this CTA's memory after it exits.
            if (lane == 0) mbar_wait_bounded(&stage->bar, phase, wait_limit());
            __syncwarp();
            return false;
        }
        // Staged rows, kRound partials per round (8 rows of the G heads): the
        // weights' shuffles and the rows' shared-memory loads of a round are
        // all issued before its FMAs.
        auto fold = [&](int k, auto kU) {
            constexpr int kU_ = decltype(kU)::value;
            float w[kU_][G];
            Vec v[kU_][G];
#pragma unroll
            for (int u = 0; u < kU_; ++u)
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    w[u][h] = __shfl_sync(0xffffffffu, wgt[h], k + u);
                    v[u][h] = *reinterpret_cast<const Vec *>(rows + (h * cnt + k + u) * D +
                                                             lane * kDims);
                }
#pragma unroll
            for (int u = 0; u < kU_; ++u)
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float *f = reinterpret_cast<const float *>(&v[u][h]);
#pragma unroll
                    for (int d = 0; d < kDims; ++d) acc[h][d] += w[u][h] * f[d];
                }
        };
        constexpr int kRound = G >= 4 ? 1 : 8 / G;  // (more rows per round spill at G = 4)
        int k = 0;
        for (; k + kRound <= cnt; k += kRound) fold(k, std::integral_constant<int, kRound>());
        for (; k < cnt; ++k) fold(k, std::integral_constant<int, 1>());
        __syncwarp();  // the next chunk overwrites the staging area
        j0 += tot;
    }
    // The G denominators reduce side by side, then each head's output row.
    float lt[G];
#pragma unroll
    for (int h = 0; h < G; ++h) lt[h] = den[h];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int h = 0; h < G; ++h) lt[h] += __shfl_xor_sync(0xffffffffu, lt[h], o);
#pragma unroll
    for (int h = 0; h < G; ++h) {
        if (p.sinks)
            lt[h] += fast_exp2(Elem<T>::to_f32(static_cast<const T *>(p.sinks)[it.g * G + h]) *
                                   kLog2e -
                               run_m[h]);
        const float inv = 1.f / lt[h];
        float o[kDims];
#pragma unroll
        for (int d = 0; d < kDims; ++d) o[d] = acc[h][d] * inv;
        store_row<T, kDims>(static_cast<T *>(p.out) + (head0 + h) * D + lane * kDims, o);
    }
    return true;
}

// ---- bf16 tensor-core pieces (the page layout they read is the one the
// producer's tensor copies write: per page, [D/64 halves][16 rows] of 128-byte
// lines, the 16-byte chunk c of line L stored at chunk c ^ (L % 8)).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// d += a (16x16 bf16, row-major) * b (16x8 bf16, column-major), fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Transpose of an 8x8 b16 matrix spread over the warp as in an mma
// accumulator (thread t: row t/4, columns 2 (t%4) and 2 (t%4) + 1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}
template <int D>
__device__ __forceinline__ uint32_t page_addr(uint32_t base, int key, int d) {
    const int line = (d >> 6) * kBlock + key;
    return base + line * 128 + ((((d & 63) >> 3) ^ (line & 7)) << 4);
}

// One page of the bf16 path for one consumer warp, on the tensor cores
// (mma.sync m16n8k16), both products transposed so that the page's 16 keys
// (and, for P V, 16 output dims) fill the 16 rows of A and the G query heads
// are the 8 columns of B (rows G..7 of B zero):
//   S^T = K q^T:      A = K (16 keys x 16 dims, ldmatrix), B = q^T (qa);
//   O^T += V^T P^T:   A = V^T (16 dims x 16 keys, ldmatrix.trans), B = P^T;
// one MMA per 16 dims for each product.  Thread t holds S^T for keys t/4 and
// t/4 + 8 of heads 2 (t%4) and 2 (t%4) + 1, so a head's maximum is reduced
// over the 8 threads with the same t % 4, and P^T moves from that layout to
// the B layout with one movmatrix.trans per 8 keys.  O^T: oacc[dn] holds dims
// 16 dn + t/4 and 16 dn + t/4 + 8 of heads 2 (t%4) (elements 0, 2) and
// 2 (t%4) + 1 (elements 1, 3); m2, l2: the running maximum (base 2) and this
// thread's share of the sum for those two heads.  Keys outside [t_lo, t_hi)
// are masked out of S and their V entries zeroed in the fragments (a slot past
// the sequence's end may hold any bits).  qa: per 16-dim step, row t/4 of q
// (head t/4) as two bf16 pairs.  kSplit: Q K^T as two independent
// accumulator chains (even and odd 16-dim steps) added at the end (for the
// deep-ring kernel, whose one CTA per SM leaves the registers).
template <int D, bool kFull, bool kSplit = false>
__device__ __forceinline__ void consume_page_mma(uint32_t kaddr, uint32_t vaddr, int t_lo, int t_hi,
                                                 const uint32_t (&qa)[D / 16][2], float qscale,
                                                 float (&m2)[2], float (&l2)[2],
                                                 float (&oacc)[D / 16][4], int lane) {
    const int tq = lane & 3, mi = lane >> 3, ri = lane & 7, kr = lane >> 2;
    constexpr int kChains = kSplit ? 2 : 1;
    float sch[kChains][4];
#pragma unroll
    for (int k = 0; k < kChains; ++k)
#pragma unroll
        for (int c = 0; c < 4; ++c) sch[k][c] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        // Tiles: keys 0-7 / dims 0-7, keys 0-7 / dims 8-15, keys 8-15 / dims
        // 0-7, keys 8-15 / dims 8-15; A wants rows 0-7 k 0-7, rows 8-15 k 0-7,
        // rows 0-7 k 8-15, rows 8-15 k 8-15.
        uint32_t r0, r1, r2, r3;
        ldsm_x4(page_addr<D>(kaddr, ((mi >> 1) << 3) + ri, 16 * ks + ((mi & 1) << 3)), r0, r1, r2,
                r3);
        mma_16816(sch[ks % kChains], r0, r2, r1, r3, qa[ks][0], qa[ks][1]);
    }
    // s: (key kr, head 2tq), (kr, 2tq + 1), (kr + 8, 2tq), (kr + 8, 2tq + 1).
    float s[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const float x = (kSplit ? sch[0][c] + sch[kChains - 1][c] : sch[0][c]) * qscale;
        const int t = kr + ((c >> 1) << 3);
        s[c] = (kFull || (t >= t_lo && t < t_hi)) ? x : -INFINITY;
    }
    float mx[2] = {fmaxf(s[0], s[2]), fmaxf(s[1], s[3])};
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1)
#pragma unroll
        for (int e = 0; e < 2; ++e) mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], o));
    float ref[2], corr[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const float m_new = fmaxf(m2[e], mx[e]);
        ref[e] = m_new == -INFINITY ? 0.f : m_new;
        corr[e] = fast_exp2(m2[e] - ref[e]);
        m2[e] = m_new;
    }
    float pv[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) pv[c] = fast_exp2(s[c] - ref[c & 1]);
#pragma unroll
    for (int e = 0; e < 2; ++e) l2[e] = l2[e] * corr[e] + (pv[e] + pv[e + 2]);
#pragma unroll
    for (int dn = 0; dn < D / 16; ++dn) {
        oacc[dn][0] *= corr[0];
        oacc[dn][1] *= corr[1];
        oacc[dn][2] *= corr[0];
        oacc[dn][3] *= corr[1];
    }
    // P^T in the B layout: keys 0-7, then keys 8-15.
    const uint32_t pb0 = movmatrix_trans(pack_bf16x2(pv[0], pv[1]));
    const uint32_t pb1 = movmatrix_trans(pack_bf16x2(pv[2], pv[3]));
    // V fragment masks: keys 2tq + {0,1} (low, high half), and +8.
    uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
    if (!kFull) {
        const int k = 2 * tq;
        mlo = ((k >= t_lo && k < t_hi) ? 0xffffu : 0u) | ((k + 1 >= t_lo && k + 1 < t_hi) ? 0xffff0000u : 0u);
        mhi = ((k + 8 >= t_lo && k + 8 < t_hi) ? 0xffffu : 0u) |
              ((k + 9 >= t_lo && k + 9 < t_hi) ? 0xffff0000u : 0u);
    }
#pragma unroll
    for (int dn = 0; dn < D / 16; ++dn) {
        // Transposed tiles (same addresses as for K): V^T dims 0-7 / keys 0-7,
        // dims 8-15 / keys 0-7, dims 0-7 / keys 8-15, dims 8-15 / keys 8-15 -
        // already the A order.
        uint32_t v0, v1, v2, v3;
        ldsm_x4_t(page_addr<D>(vaddr, ((mi >> 1) << 3) + ri, 16 * dn + ((mi & 1) << 3)), v0, v1, v2,
                  v3);
        mma_16816(oacc[dn], v0 & mlo, v1 & mlo, v2 & mhi, v3 & mhi, pb0, pb1);
    }
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *tm, int w,
                                            uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %2, %2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(0), "r"(w), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// One consumer warp's share of an item's merge, once all four consumer
// states are in the merge buffer: for dims [cw * D/4, (cw + 1) * D/4) of
// every head, the four (m, l, O) are combined by their log-sum-exp weights
// into the final output (a sequence in one partition: with the sink in the
// denominator) or that quarter of the item's fp32 partial (consumer 0 also
// writes the partial's m and l).  The four warps merge side by side.
template <typename T, int D, int G>
__device__ __forceinline__ void merge_quarter(const Params &p, const Item &it,
                                              const unsigned char *mb, int cw, int lane) {
    static_assert(kConsumerWarps == 4, "m and l of a head's four consumers are one float4");
    constexpr int kQ = D / kConsumerWarps;     // dims per consumer
    constexpr int kPerHead = kQ / 4;           // float4 chunks per head and consumer
    constexpr int kChunks = G * kPerHead, kIters = (kChunks + 31) / 32;
    const float *cM = reinterpret_cast<const float *>(mb + 32);
    const float *cL = cM + kConsumerWarps * G;
    const float *cO = cL + kConsumerWarps * G;
    const bool single = it.nparts == 1;
    const int64_t head0 = static_cast<int64_t>(it.b) * p.Hq + static_cast<int64_t>(it.g) * G;
#pragma unroll
    for (int i = 0; i < kIters; ++i) {
        const int ch = lane + 32 * i;
        if (kChunks % 32 != 0 && ch >= kChunks) continue;
        const int h = ch / kPerHead, d = cw * kQ + (ch - h * kPerHead) * 4;
        const float4 m4 = *reinterpret_cast<const float4 *>(cM + h * kConsumerWarps);
        const float4 l4 = *reinterpret_cast<const float4 *>(cL + h * kConsumerWarps);
        const float mx = fmaxf(fmaxf(m4.x, m4.y), fmaxf(m4.z, m4.w));
        const float f[kConsumerWarps] = {fast_exp2(m4.x - mx), fast_exp2(m4.y - mx),
                                         fast_exp2(m4.z - mx), fast_exp2(m4.w - mx)};
        const float lt = f[0] * l4.x + f[1] * l4.y + f[2] * l4.z + f[3] * l4.w;
        float4 ot = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w2 = 0; w2 < kConsumerWarps; ++w2) {
            const float4 v = *reinterpret_cast<const float4 *>(&cO[(w2 * G + h) * D + d]);
            ot.x += f[w2] * v.x;
            ot.y += f[w2] * v.y;
            ot.z += f[w2] * v.z;
            ot.w += f[w2] * v.w;
        }
        // A sink is one more logit with no value row: it only adds to the
        // final denominator (partials leave it to the combine).
        float den = lt;
        if (single && p.sinks)
            den += fast_exp2(Elem<T>::to_f32(static_cast<const T *>(p.sinks)[it.g * G + h]) *
                                 kLog2e -
                             mx);
        const float inv = 1.f / den;
        const float o4[4] = {ot.x * inv, ot.y * inv, ot.z * inv, ot.w * inv};
        if (single) {
            store_row<T, 4>(static_cast<T *>(p.out) + (head0 + h) * D + d, o4);
        } else {
            const int64_t pi = (head0 + h) * p.max_parts + it.part;
            store_row<float, 4>(&p.part_o[pi * D + d], o4);
            if (d == 0) {
                p.part_m[pi] = mx;
                p.part_l[pi] = lt;
            }
        }
    }
}

// One consumer warp's share of a split group's combine (a job the merger
// hands over once the producer has no more items, so the four consumer
// warps are free): for dims [cw * D/4, (cw + 1) * D/4) of the G heads,
//     out = sum_j 2^(m_j - M) l_j o_j / sum_j 2^(m_j - M) l_j  (+ sink term)
// over the group's np partials.  Partials are read straight from L2 into
// registers, kRound of them per round trip together with their m and l
// (lane j holds partial j0 + j's); the round's weights go through this
// warp's scratch in shared memory (its own ring stage, idle by then).  The
// partials were acquired by the merger's count and handed over through a
// CTA barrier.
template <typename T, int D, int G>
__device__ __noinline__ void combine_quarter(const Params &p, int b, int g, int np, int cw, int lane,
                                             int scratch_off) {
    using Vec = float4;
    constexpr int kQ = D / kConsumerWarps;       // dims per warp
    constexpr int kPerHead = kQ / 4;             // float4 chunks per head
    constexpr int kChunks = G * kPerHead;        // chunks per warp
    constexpr int kPer = (kChunks + 31) / 32;    // chunks per lane
    // Partials per round trip, as many as the register budget holds.
    constexpr int kRound = Cfg<T, D, G>::kMinBlocks >= 3 ? 6 : (kPer == 1 ? 20 : 10);
    float *W = reinterpret_cast<float *>(dyn_smem() + scratch_off);  // [G][kRound]
    if (!XS_BOUNDS(np >= 1 && np <= p.max_parts && b >= 0 && b < p.B && g >= 0 && g < p.Hkv,
                   p.err_flag))
        return;  // (debug build) nothing read or written
    const int64_t head0 = static_cast<int64_t>(b) * p.Hq + static_cast<int64_t>(g) * G;
    int hh[kPer], dd[kPer];
    bool on[kPer];
    float acc[kPer][4];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int c = lane + 32 * i;
        on[i] = kChunks % 32 == 0 || c < kChunks;
        hh[i] = on[i] ? c / kPerHead : 0;
        dd[i] = cw * kQ + (c - hh[i] * kPerHead) * 4;
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[i][e] = 0.f;
    }
    float run_m[G], den[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        run_m[h] = -INFINITY;
        den[h] = 0.f;
    }
    const float *pm = p.part_m + head0 * p.max_parts;
    const float *pl = p.part_l + head0 * p.max_parts;
    for (int j0 = 0; j0 < np; j0 += kRound) {
        const int n = min(kRound, np - j0);
        // The round's rows first (no dependence on the weights), then m, l.
        Vec rows[kRound][kPer];
#pragma unroll
        for (int u = 0; u < kRound; ++u)
#pragma unroll
            for (int i = 0; i < kPer; ++i)
                if (u < n && on[i])
                    rows[u][i] = __ldcg(reinterpret_cast<const Vec *>(
                        p.part_o + ((head0 + hh[i]) * p.max_parts + j0 + u) * D + dd[i]));
        float mj[G], lj[G], cm[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            mj[h] = -INFINITY;
            lj[h] = 0.f;
            if (lane < n) {
                mj[h] = __ldcg(pm + h * p.max_parts + j0 + lane);
                lj[h] = __ldcg(pl + h * p.max_parts + j0 + lane);
            }
            cm[h] = mj[h];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int h = 0; h < G; ++h) cm[h] = fmaxf(cm[h], __shfl_xor_sync(0xffffffffu, cm[h], o));
        float corr[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float m_new = fmaxf(run_m[h], cm[h]);
            const float ref = m_new == -INFINITY ? 0.f : m_new;
            corr[h] = fast_exp2(run_m[h] - ref);  // 0 while nothing is accumulated
            run_m[h] = m_new;
            const float w = lane < n ? fast_exp2(mj[h] - ref) * lj[h] : 0.f;
            den[h] = den[h] * corr[h] + w;
            if (lane < kRound) W[h * kRound + lane] = w;
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            float c = corr[0];
#pragma unroll
            for (int h = 1; h < G; ++h) c = hh[i] == h ? corr[h] : c;
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][e] *= c;
        }
#pragma unroll
        for (int u = 0; u < kRound; ++u)
#pragma unroll
            for (int i = 0; i < kPer; ++i)
                if (u < n && on[i]) {
                    const float w = W[hh[i] * kRound + u];
                    acc[i][0] += w * rows[u][i].x;
                    acc[i][1] += w * rows[u][i].y;
                    acc[i][2] += w * rows[u][i].z;
                    acc[i][3] += w * rows[u][i].w;
                }
        __syncwarp();  // the next round overwrites the weights
    }
    // Denominators: the lanes' sums, reduced side by side for the G heads.
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int h = 0; h < G; ++h) den[h] += __shfl_xor_sync(0xffffffffu, den[h], o);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        if (!on[i]) continue;
        float lt = den[0], mh = run_m[0];
#pragma unroll
        for (int h = 1; h < G; ++h) {
            lt = hh[i] == h ? den[h] : lt;
            mh = hh[i] == h ? run_m[h] : mh;
        }
        if (p.sinks)
            lt += fast_exp2(Elem<T>::to_f32(static_cast<const T *>(p.sinks)[g * G + hh[i]]) * kLog2e -
                            mh);
        const float inv = 1.f / lt;
        const float o4[4] = {acc[i][0] * inv, acc[i][1] * inv, acc[i][2] * inv, acc[i][3] * inv};
        store_row<T, 4>(static_cast<T *>(p.out) + (head0 + hh[i]) * D + dd[i], o4);
    }
}

// The merger's batched count: queue entry k (held by lane k < npend) is a
// split item of group (b, g) with np partitions whose partials this warp has
// written.  One fence publishes them all; each entry's group count is then
// raised (all in flight together) and every entry that completes its group
// combines it and clears the count for the next launch.
template <typename T, int D, int G, typename Post>
__device__ __forceinline__ bool count_and_combine(const Params &p, int lane, int pend_b, int pend_g,
                                                  int pend_np, int npend, int stage_off,
                                                  bool to_consumers, Post &&post) {
    // Every lane's partial stores are gathered by the warp barrier; each
    // counting lane's acquire-release add releases them (cumulatively) and
    // acquires the group's earlier partials; a second barrier hands that to
    // every lane.
    __syncwarp();
    int *cnt = p.combine + static_cast<int64_t>(pend_b) * p.Hkv + pend_g;
    int prior = 0;
    if (lane < npend &&
        XS_BOUNDS(pend_b >= 0 && pend_b < p.B && pend_g >= 0 && pend_g < p.Hkv, p.err_flag))
        prior = atomic_add_acq_rel_gpu(cnt, 1);
    const bool last = lane < npend && prior == pend_np - 1;
    unsigned todo = __ballot_sync(0xffffffffu, last);
    if (todo) __syncwarp();
    bool ok = true;
    const unsigned combined = todo;
    while (todo && ok) {
        const int k = __ffs(todo) - 1;
        todo &= todo - 1;
        Item ci;
        ci.b = __shfl_sync(0xffffffffu, pend_b, k);
        ci.g = __shfl_sync(0xffffffffu, pend_g, k);
        ci.nparts = __shfl_sync(0xffffffffu, pend_np, k);
        const int64_t h0 = static_cast<int64_t>(ci.b) * p.Hq + static_cast<int64_t>(ci.g) * G;
        ok = to_consumers ? post(ci.b, ci.g, ci.nparts)
                          : combine_partials<T, D, G>(p, ci, h0, lane, stage_off);
    }
    // Leave the completed groups' counts zero for the next launch - after
    // the combines (or their hand-over), so no fence above waits for these
    // writes.
    if (combined & (1u << lane)) atomicExch(cnt, 0);
    return ok;
}

template <typename T, int D, int G, int S>
__global__ void __launch_bounds__(kThreads, Cfg<T, D, G, S>::kMinBlocks)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv, const Params p) {
    using C = Cfg<T, D, G, S>;
    constexpr int kStages = C::kStages;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    // The base rounded up to 1024 bytes by pointer arithmetic on the shared
    // array (not through an integer), so accesses through it stay
    // shared-memory accesses.
    unsigned char *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
    uint64_t *empty = full + kStages;
    uint64_t *qfull = empty + kStages;
    uint64_t *qempty = qfull + 2;
    uint64_t *merged = qempty + 2;  // per merge buffer: the four consumer states are in
    uint64_t *freed = merged + C::kMergeBufs;  // per merge buffer: the merger has read it
    uint64_t *quartered = freed + C::kMergeBufs;  // per merge buffer: the four quarters are merged
    Item *item_slot = reinterpret_cast<Item *>(smem + C::kItemOff);
    int *pfull = reinterpret_cast<int *>(smem + C::kPrefixOff);
    int *ptail = pfull + p.B + 1;
    int *nlen = ptail + p.B + 1;
    __shared__ int s_abort;
    // Role warps still running, and the producer's page and item counts:
    // the last warp to finish drains the copies after an abort (exit_role).
    __shared__ int s_roles_left;
    __shared__ uint32_t s_issued[2];
    // Set by the producer once it has no more items for this CTA.  From then
    // on the merger hands the combines of completed groups to the consumer
    // warps (s_job: b, g, nparts; b < 0 ends the consumers' service).
    __shared__ int s_no_more;
    __shared__ int s_job[3];
    __shared__ uint64_t s_job_full, s_job_done;
    // Only where a quarter of a group's dims fills a warp (G * D / 16 float4
    // chunks per warp >= 32 lanes); narrower groups stay with the merger.
    constexpr bool kJobs = G * D >= 512;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    // The launch must provide the shared memory this B needs; refuse (flag,
    // return before touching shared memory) if it does not.
    if (dynamic_smem_bytes() < static_cast<uint32_t>(C::smem_bytes(p.B) + p.stage_bytes) ||
        (p.combine && p.stage_parts < 1)) {
        if (tid == 0) raise_flag(p.err_flag, XS_FLAG_CONFIG);
        return;
    }

    // ---- prologue: barriers, item prefix sums, zero outputs of empty sequences
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&qfull[s], 1);
            mbar_init(&qempty[s], kConsumerWarps);
        }
        for (int s = 0; s < C::kMergeBufs; ++s) {
            mbar_init(&merged[s], kConsumerWarps);
            mbar_init(&freed[s], 1);
            mbar_init(&quartered[s], kConsumerWarps);
        }
        mbar_init(&s_job_full, 1);
        mbar_init(&s_job_done, kConsumerWarps);
        if (p.combine) {
            Stage *st = reinterpret_cast<Stage *>(smem + stage_offset(C::kPrefixOff, p.B));
            mbar_init(&st->bar, 1);
            st->phase = 0;
        }
        mbar_fence_init();
        s_abort = 0;
        s_roles_left = kConsumerWarps + 2;
        s_issued[0] = s_issued[1] = 0;
        s_no_more = 0;
    }
    // Programmatic dependent launch.  griddep_wait returns once the previous
    // launch on the stream has completed and its writes are visible; only
    // then may the next launch start placing CTAs (so a launch never runs
    // beside any but its immediate predecessor).  By default nothing in
    // global memory is touched before the wait.  With p.early the lengths,
    // the item tables, the first item's block ids and its first pages (all
    // but a page that receives this launch's appended row) are read before
    // it: the caller promises that the previous launch writes none of them.
    // q, k_new/v_new and every write come after the wait.  (No-ops in a
    // launch made without the attribute.)
    if (!p.early) {
        griddep_wait();
        griddep_launch_dependents();
    }
    {
        // Per sequence: its class A and class B item counts (item_counts).
        // Chunked scan of both counts over the block.
        const int per = (p.B + kThreads - 1) / kThreads;
        const int b0 = min(p.B, tid * per), b1 = min(p.B, b0 + per);
        int lf = 0, lt = 0;
        for (int b = b0; b < b1; ++b) {
            const int n = max(seq_len(p, b, blockIdx.x == 0), 0);
            int ca, cb;
            item_counts(p, n - first_token(p, n), ca, cb);  // tokens inside the window
            lf += ca;
            lt += cb;
        }
        int xf = lf, xt = lt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int yf = __shfl_up_sync(0xffffffffu, xf, o);
            const int yt = __shfl_up_sync(0xffffffffu, xt, o);
            if (lane >= o) {
                xf += yf;
                xt += yt;
            }
        }
        __shared__ int warp_tot[2][kThreads / 32];
        if (lane == 31) {
            warp_tot[0][warp] = xf;
            warp_tot[1][warp] = xt;
        }
        __syncthreads();
        int basef = 0, baset = 0;
        for (int w = 0; w < warp; ++w) {
            basef += warp_tot[0][w];
            baset += warp_tot[1][w];
        }
        int runf = basef + xf - lf, runt = baset + xt - lt;  // exclusive prefixes
        for (int b = b0; b < b1; ++b) {
            const int n = max(seq_len(p, b, false), 0);
            int ca, cb;
            item_counts(p, n - first_token(p, n), ca, cb);
            pfull[b] = runf;
            ptail[b] = runt;
            nlen[b] = n;
            runf += ca;
            runt += cb;
        }
        if (tid == kThreads - 1) {
            pfull[p.B] = basef + xf;
            ptail[p.B] = baset + xt;
        }
    }
    __syncthreads();
    const int total_items = pfull[p.B] + ptail[p.B];
    // Every role warp calls this once, as its last action.  After an abort
    // (a bounded wait that ran out, in any warp) consumers may have left
    // without waiting for pages already requested, so the last warp to
    // finish lets every copy the producer issued land before the CTA exits:
    // only the last kStages pages can be in flight (an older page's stage
    // was reissued, which took its consumer's release after the page
    // landed), and only the last two q slots.  Nothing waits otherwise.
    auto exit_role = [&]() {
        __syncwarp();
        if (lane != 0) return;
        __threadfence_block();
        if (atomicSub(&s_roles_left, 1) != 1) return;
        __threadfence_block();
        if (!*static_cast<volatile int *>(&s_abort)) return;
        const uint32_t pages = s_issued[0], items = s_issued[1];
        for (uint32_t c = pages > kStages ? pages - kStages : 0; c < pages; ++c)
            mbar_wait_bounded(&full[c % kStages], (c / kStages) & 1, wait_limit());
        for (uint32_t k = items > 2 ? items - 2 : 0; k < items; ++k)
            mbar_wait_bounded(&qfull[k & 1], (k >> 1) & 1, wait_limit());
    };
    if (warp != 0) {
        // Every warp but the producer passes the wait here; the producer
        // passes it after its early reads.
        if (p.early) {
            griddep_wait();
            griddep_launch_dependents();
        }
        // Sequences with no tokens produce zeros.
        for (int b = blockIdx.x; b < p.B && p.prefill_start < 0; b += gridDim.x) {
            if (nlen[b] > 0) continue;
            T *o = static_cast<T *>(p.out) + static_cast<int64_t>(b) * p.Hq * D;
            for (int i = tid - 32; i < p.Hq * D; i += kThreads - 32) o[i] = Elem<T>::from_f32(0.f);
        }
    }

    if (warp == 0) {
        // ================================================================ producer
        // Takes items (from the shared work counter, or blockIdx.x + k*gridDim.x
        // without one), publishes each item's ranges and q rows in a
        // double-buffered slot, then streams its pages into the ring.  An item
        // with b < 0 tells the consumers to stop.  The producer runs one item
        // ahead: while it issues item A's pages, item B is decoded with its
        // first block ids loading, and the counter fetch for the item after
        // B is in flight.
        const uint64_t pol = policy_evict_first();
        const unsigned char *kbase = static_cast<const unsigned char *>(p.k_cache);
        const unsigned char *vbase = static_cast<const unsigned char *>(p.v_cache);
        const unsigned char *qbase = static_cast<const unsigned char *>(p.q);
        uint32_t page_ctr = 0, item_ctr = 0;
        int static_next = blockIdx.x;
        int grabs = 0;
        // The first two items of CTA c are c and c + gridDim.x (no atomic on
        // the start-up path); later ones come from the shared counter (items
        // 2*gridDim.x + its value) or, without one, from c + k * gridDim.x.
        // grab() only starts the fetch; item_of() turns it into an item id
        // when it is needed, so the counter's round trip is not waited for
        // early (the warp issues in order).  Lane 0's value is the one used.
        struct Ticket {
            int raw;
            bool counted;
        };
        auto grab = [&]() {
            Ticket t{static_next, false};
            if (p.work && grabs >= 2) {
                t.counted = true;
                t.raw = atomic_add_if(&p.work[0], 1, lane == 0);  // no branch: not waited on here
            }
            ++grabs;
            static_next += gridDim.x;
            return t;
        };
        auto item_of = [&](const Ticket &t) {
            const int raw = __shfl_sync(0xffffffffu, t.raw, 0);
            return t.counted ? 2 * static_cast<int>(gridDim.x) + raw : raw;
        };
        auto decode = [&](int item) {
            Item it;
            if (item < total_items) {
                it = decode_item(p, pfull, ptail, nlen, item, lane);
            } else {
                if (lane == 0) *static_cast<volatile int *>(&s_no_more) = 1;
                it.b = -1;
                it.g = it.part = it.nparts = it.tok0 = it.tok1 = it.pg0 = it.pg1 = 0;
            }
            return it;
        };
        // Block ids of pages [base, base + 32) of an item, one per lane (0 past the end).
        // Only starts the loads; the ids are checked where they are used.
        auto load_ids = [&](const Item &it, int base) {
            int32_t blk = 0;
            const int pg = base + lane;
            if (it.b >= 0 && pg < it.pg1 &&
                XS_BOUNDS(it.b < p.B && pg >= 0 && pg < p.max_blocks, p.err_flag))
                blk = p.block_tables[static_cast<int64_t>(it.b) * p.table_stride + pg];
            return blk;
        };
        // Fused append: the item whose range ends at the sequence's last
        // token writes this step's K and V rows of head g into their slot
        // before it loads that page.  Rows are fetched one item ahead, with
        // the sequence's unclamped length (a length beyond the table appends
        // nothing, as in the separate append).
        constexpr int kRowChunks = 2 * C::kChunksPerRow;  // K row, then V row
        constexpr int kRowPerLane = (kRowChunks + 31) / 32;
        struct Row {
            uint4 v[kRowPerLane];
            int raw_len;  // context_lens[b]; 0 = this item appends nothing
        };
        auto load_row = [&](const Item &it) {
            Row r;
            r.raw_len = 0;
            if (p.k_new && it.b >= 0 && it.tok1 == nlen[it.b] && it.tok1 > 0 &&
                XS_BOUNDS(it.b < p.B && it.g >= 0 && it.g < p.Hkv, p.err_flag)) {
                r.raw_len = p.context_lens[it.b];
                const int64_t row = static_cast<int64_t>(it.b) * p.Hkv + it.g;
                const uint4 *kn = static_cast<const uint4 *>(p.k_new) + row * C::kChunksPerRow;
                const uint4 *vn = static_cast<const uint4 *>(p.v_new) + row * C::kChunksPerRow;
#pragma unroll
                for (int u = 0; u < kRowPerLane; ++u) {
                    const int c = lane + 32 * u;
                    if (c < C::kChunksPerRow)
                        r.v[u] = kn[c];
                    else if (c < kRowChunks)
                        r.v[u] = vn[c - C::kChunksPerRow];
                }
            }
            return r;
        };
        // Write the row of item `it` into block `blk`, then order those
        // generic-proxy writes before the bulk copies that read the page.
        auto store_row = [&](const Item &it, const Row &r, int32_t blk) {
            const int n = r.raw_len;
            if (n <= 0 || n > p.max_blocks * kBlock) return;  // nothing to append
            if (blk < 0 || blk >= p.num_blocks) {
                if (lane == 0) raise_flag(p.err_flag, XS_FLAG_BAD_BLOCK);
                return;
            }
            const int64_t dst_row =
                ((static_cast<int64_t>(blk) * p.Hkv + it.g) * kBlock + (n - 1) % kBlock) *
                C::kChunksPerRow;
            uint4 *kc = static_cast<uint4 *>(const_cast<void *>(p.k_cache)) + dst_row;
            uint4 *vc = static_cast<uint4 *>(const_cast<void *>(p.v_cache)) + dst_row;
#pragma unroll
            for (int u = 0; u < kRowPerLane; ++u) {
                const int c = lane + 32 * u;
                if (c < C::kChunksPerRow)
                    kc[c] = r.v[u];
                else if (c < kRowChunks)
                    vc[c - C::kChunksPerRow] = r.v[u];
            }
            fence_proxy_async_global();
        };
        // Publish an item (or the end marker) in the next q slot.
        auto publish = [&](const Item &it) {
            bool ok = true;
            if (lane == 0) {
                const uint32_t slot = item_ctr & 1, k = item_ctr >> 1;
                ok = mbar_wait_bounded(&qempty[slot], (k & 1) ^ 1, wait_limit());
                if (ok) {
                    item_slot[slot] = it;
                    if (it.b < 0 || !XS_BOUNDS(it.b < p.B && it.g >= 0 && (it.g + 1) * G <= p.Hq,
                                               p.err_flag)) {
                        mbar_arrive(&qfull[slot]);  // end marker (or, debug build: skipped rows)
                    } else {
                        unsigned char *dst = smem + C::kQSlotOff + slot * C::kQBytes;
                        const int64_t qoff = (static_cast<int64_t>(it.b) * p.Hq +
                                              static_cast<int64_t>(it.g) * G) *
                                             C::kRowBytes;
                        mbar_arrive_expect_tx(&qfull[slot], C::kQBytes);
                        bulk_g2s(dst, qbase + qoff, C::kQBytes, &qfull[slot]);
                    }
                }
            }
            ++item_ctr;
            return __shfl_sync(0xffffffffu, ok, 0);
        };
        // Issue the copies of pages base + [from, to) of item `it`: lane i
        // holds the block id of page base + i (cnt of them valid).  Each
        // round, the lanes test the stages of the next (up to kStages) pages
        // and every lane of the leading run of free stages issues its page's
        // two copies - one warp instruction for all of them - so a producer
        // that has fallen behind catches up several pages at a time.  False
        // if a bounded wait for a free stage ran out.
        auto issue = [&](const Item &it, int32_t ids, int cnt, int from, int to) {
            const int64_t head_off = static_cast<int64_t>(it.g) * C::kPageBytes;
            const int64_t blk_stride = static_cast<int64_t>(p.Hkv) * C::kPageBytes;
            // An id outside the pool reads block 0 instead (flagged).
            const bool bad_id = lane < cnt && (ids < 0 || ids >= p.num_blocks);
            if (__any_sync(0xffffffffu, bad_id) && lane == 0) raise_flag(p.err_flag, XS_FLAG_BAD_BLOCK);
            const int64_t my_off = static_cast<int64_t>(bad_id ? 0 : ids) * blk_stride + head_off;
            const int my_page = (bad_id ? 0 : ids) * p.Hkv + it.g;  // tensor-map page index
            int done = from;
            while (done < to) {
                const int want = min(to - done, kStages);
                const uint32_t c = page_ctr + lane;
                const uint32_t st = c % kStages;
                const bool is_free =
                    lane < want && mbar_test_wait(&empty[st], ((c / kStages) & 1) ^ 1);
                const int n = __ffs(~__ballot_sync(0xffffffffu, is_free)) - 1;
                const int64_t off = __shfl_sync(0xffffffffu, my_off, (done + lane) & 31);
                const int pidx = __shfl_sync(0xffffffffu, my_page, (done + lane) & 31);
                if (n == 0) {
                    // No stage free yet: wait (bounded) for the next one.
                    bool w = true;
                    if (lane == 0)
                        w = mbar_wait_bounded(&empty[page_ctr % kStages],
                                              ((page_ctr / kStages) & 1) ^ 1, wait_limit());
                    if (!__shfl_sync(0xffffffffu, w, 0)) return false;
                    continue;
                }
                if (lane < n && !skip_page(c)) {  // (a skipped page: debug library only)
                    unsigned char *dk = smem + st * 2 * C::kPageBytes;
                    mbar_arrive_expect_tx(&full[st], 2 * C::kPageBytes);
                    if constexpr (C::kMma) {
                        tma_load_4d(smem_addr(dk), &tmk, pidx, &full[st], pol);
                        tma_load_4d(smem_addr(dk + C::kPageBytes), &tmv, pidx, &full[st], pol);
                    } else {
                        bulk_g2s(dk, kbase + off, C::kPageBytes, &full[st], pol);
                        bulk_g2s(dk + C::kPageBytes, vbase + off, C::kPageBytes, &full[st], pol);
                    }
                }
                done += n;
                page_ctr += n;  // pages issued so far
            }
            return true;
        };
        // Item B is published (q rows copied in) before item A's pages are
        // issued, so consumers finishing A find B's q already in place.
        Item A = decode(item_of(grab()));
        int32_t idsA = load_ids(A, A.pg0);
        bool ok = true;
        int pre = 0;  // pages of the first item issued before the wait
        if (p.early) {
            // Up to a ring of the first item's pages, stopping before a page
            // that receives this launch's appended row.
            if (A.b >= 0) {
                const int end = A.tok1 == nlen[A.b] ? A.pg1 - 1 : A.pg1;
                pre = min(kStages, max(0, end - A.pg0));
                if (pre > 0) ok = issue(A, idsA, min(32, A.pg1 - A.pg0), 0, pre);
                // In a launch of at most 16 rounds of items, the item's next
                // kL2Ahead pages also go to L2 (a cache hint: no shared memory,
                // nothing waits for it), so after the wait they stream from L2
                // while the previous launch's tail has left HBM underused.  L2
                // is the device's point of coherence, so a page the previous
                // launch writes later still reads right.  (Measured: 64-sequence
                // mixes 1.3-3.3 % faster; a 30-round launch, where the start
                // is a small share, 0.3 % slower, hence the bound.)
                const bool l2_ahead = total_items <= 16 * static_cast<int>(gridDim.x);
                const int lim = l2_ahead ? min(min(32, A.pg1 - A.pg0), pre + kL2Ahead) : 0;
                if (lane >= pre && lane < lim && idsA >= 0 && idsA < p.num_blocks) {
                    const int64_t off =
                        (static_cast<int64_t>(idsA) * p.Hkv + A.g) * C::kPageBytes;
                    prefetch_l2(kbase + off, C::kPageBytes);
                    prefetch_l2(vbase + off, C::kPageBytes);
                }
            }
            griddep_wait();
            griddep_launch_dependents();
        }
        Row rowA = load_row(A);
        if (ok) ok = publish(A);
        while (ok && A.b >= 0) {
            // Stream A's pages, 32 block ids at a time (the next 32 load
            // meanwhile); lane i owns page base + i of a chunk.  The next item
            // is claimed only when kClaimAhead of A's pages are left to issue
            // (its counter fetch then returns while they stream): a CTA holds
            // no item it will not start soon, so the grid's ends even out.
            const int claim_at = max(A.pg0, A.pg1 - kClaimAhead);
            Ticket next{0, false};
            int32_t ids = idsA;
            for (int base = A.pg0; ok && base < A.pg1; base += 32) {
                const int32_t ids_next = (base + 32 < A.pg1) ? load_ids(A, base + 32) : 0;
                const int cnt = min(32, A.pg1 - base);
                if (rowA.raw_len > 0 && base + 32 >= A.pg1)  // the chunk with the last page
                    store_row(A, rowA, __shfl_sync(0xffffffffu, ids, A.pg1 - 1 - base));
                __syncwarp();
                const int from = base == A.pg0 ? pre : 0;
                if (claim_at >= base && claim_at < base + cnt) {
                    const int split = max(from, claim_at - base);
                    ok = issue(A, ids, cnt, from, split);
                    next = grab();  // unconditionally: a branch here would wait for the fetch
                    ok = ok && issue(A, ids, cnt, split, cnt);
                } else {
                    ok = issue(A, ids, cnt, from, cnt);
                }
                ids = ids_next;
            }
            if (!ok) break;
            pre = 0;
            A = decode(item_of(next));
            idsA = load_ids(A, A.pg0);
            rowA = load_row(A);
            ok = publish(A);
        }
        if (lane == 0) {
            if (!ok) {
                raise_flag(p.err_flag, XS_FLAG_TIMEOUT);
                atomicExch(&s_abort, 1);
            }
            if (p.work) {
                // The last CTA to stop taking items resets the counters for the
                // next launch on this workspace.
                __threadfence();
                if (atomicAdd(&p.work[1], 1) == static_cast<int>(gridDim.x) - 1) {
                    atomicExch(&p.work[0], 0);
                    atomicExch(&p.work[1], 0);
                }
            }
            s_issued[0] = page_ctr;
            s_issued[1] = item_ctr;
        }
        exit_role();
        return;
    }

    if (warp == kConsumerWarps + 1) {
        // ================================================================ merger
        // Waits for the four consumer states of each item, merges them (each
        // lane 4 consecutive dims of one head at a time) and writes the final
        // output or the split-K partials, then frees the buffer.
        //
        // Fused combine: a split item's partials must be visible (a fence)
        // before it is counted in its sequence-head group, and the count's
        // result decides whether this item combines the group.  Both are
        // memory round trips, so split items are queued (lane k holds entry
        // k) and counted in batches - one fence, up to 32 counts in flight -
        // whenever the next item's states are not ready yet, the queue is
        // full, or the consumers are done.
        constexpr int kMaxPend = 8;
        int pend_b = 0, pend_g = 0, pend_np = 0, npend = 0;
        const int stage_off =
            static_cast<int>(smem - smem_raw) + stage_offset(C::kPrefixOff, p.B);
        // Hand a completed group's combine to the consumer warps (their job
        // slot is reused once all four have finished the previous job).
        uint32_t njobs = 0;
        auto post = [&](int b, int g, int np) {
            bool ok = true;
            if (lane == 0) {
                if (njobs > 0) ok = mbar_wait_bounded(&s_job_done, (njobs - 1) & 1, wait_limit());
                if (ok) {
                    s_job[0] = b;
                    s_job[1] = g;
                    s_job[2] = np;
                    mbar_arrive(&s_job_full);
                }
            }
            ++njobs;
            return __shfl_sync(0xffffffffu, ok, 0);
        };
        auto flush = [&](bool to_consumers) {
            if (npend == 0) return;
            if (!count_and_combine<T, D, G>(p, lane, pend_b, pend_g, pend_np, npend, stage_off,
                                            to_consumers, post) &&
                lane == 0) {
                raise_flag(p.err_flag, XS_FLAG_TIMEOUT);
                atomicExch(&s_abort, 1);
            }
            npend = 0;
        };
        for (uint32_t item_ctr = 0;; ++item_ctr) {
            const int buf = item_ctr % C::kMergeBufs;
            unsigned char *mb = smem + C::kCombOff + buf * C::kCombBytes;
            const uint32_t mpar = (item_ctr / C::kMergeBufs) & 1;
            // Idle until the next item: count the queued ones now - unless the
            // producer is out of items, when the consumers will soon be free
            // to share the combines (counted after their last item).
            if (npend > 0 && !(kJobs && *static_cast<volatile int *>(&s_no_more)) &&
                !__shfl_sync(0xffffffffu, mbar_test_wait(&quartered[buf], mpar), 0))
                flush(false);
            if (!mbar_wait_bounded(&quartered[buf], mpar, wait_limit())) {
                if (lane == 0) {
                    raise_flag(p.err_flag, XS_FLAG_TIMEOUT);
                    atomicExch(&s_abort, 1);
                }
                break;
            }
            const Item it = *reinterpret_cast<const Item *>(mb);
            if (it.b < 0) break;  // the consumers have no more items
            const bool valid = it.b < p.B && it.g >= 0 && it.g < p.Hkv && it.part >= 0 &&
                               it.part < p.max_parts && !*static_cast<volatile int *>(&s_abort);
            const bool single = it.nparts == 1;
            // The consumers have merged and stored this item (its output, or
            // its partial): the buffer is free again.
            __syncwarp();
            if (lane == 0) mbar_arrive(&freed[buf]);
            if (valid && !single && p.combine) {
                if (lane == npend) {
                    pend_b = it.b;
                    pend_g = it.g;
                    pend_np = it.nparts;
                }
                if (++npend == kMaxPend) flush(false);
            }
        }
        // The consumers are past their last item: the remaining combines are
        // theirs, then the end of their service.
        if (!*static_cast<volatile int *>(&s_abort)) flush(kJobs);
        if (kJobs && p.combine) post(-1, 0, 0);
        exit_role();
        return;
    }

    // ==================================================================== consumers
    const int cw = warp - 1;
    // A consumer's state for item `it` is in merge buffer `buf`: announce it,
    // wait (bounded) for the other three, merge this warp's quarter of the
    // dims, and report the quarter done to the merger.  False if the wait
    // for the other states ran out.
    auto hand_over = [&](const Item &it, const unsigned char *mb, int buf, uint32_t item_ctr,
                         bool done) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&merged[buf]);
        const bool in = __all_sync(0xffffffffu, mbar_wait_bounded(&merged[buf],
                                                                  (item_ctr / C::kMergeBufs) & 1,
                                                                  wait_limit()));
        if (!in) {
            if (lane == 0) {
                raise_flag(p.err_flag, XS_FLAG_TIMEOUT);
                atomicExch(&s_abort, 1);
            }
            return false;
        }
        const bool valid = it.b >= 0 && it.b < p.B && it.g >= 0 && it.g < p.Hkv && it.part >= 0 &&
                           it.part < p.max_parts && !*static_cast<volatile int *>(&s_abort);
        if (!done && valid) merge_quarter<T, D, G>(p, it, mb, cw, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(&quartered[buf]);
        return true;
    };
    if constexpr (C::kMma) {
        // bf16: tensor-core pages (consume_page_mma); per item the G query rows
        // become A fragments (lane quad g holds head g, unscaled: scores are
        // scaled after the product), and the state handed to the merger is
        // this lane quad's head row: m, l (summed over the quad) and O.
        const int grp = lane >> 2, tq = lane & 3;
        uint32_t page_ctr = 0;
        for (uint32_t item_ctr = 0;; ++item_ctr) {
            const uint32_t slot = item_ctr & 1;
            bool bad = !__all_sync(0xffffffffu, mbar_wait_bounded(&qfull[slot], (item_ctr >> 1) & 1,
                                                                  wait_limit()));
            Item it = item_slot[slot];
            const bool done = !bad && it.b < 0;
            uint32_t qa[D / 16][2];
            if (!done) {
                const unsigned char *qs = smem + C::kQSlotOff + slot * C::kQBytes;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const unsigned char *row = qs + (grp < G ? grp : 0) * C::kRowBytes + (16 * ks + 2 * tq) * 2;
                    qa[ks][0] = grp < G ? *reinterpret_cast<const uint32_t *>(row) : 0u;
                    qa[ks][1] = grp < G ? *reinterpret_cast<const uint32_t *>(row + 16) : 0u;
                }
                __syncwarp();
                if (lane == 0 && !bad) mbar_arrive(&qempty[slot]);
            }
            if (bad || done) {
                it.b = -1;
                it.pg0 = it.pg1 = 0;
            }
            float m2[2] = {-INFINITY, -INFINITY}, l2[2] = {0.f, 0.f};
            float oacc[D / 16][4];
#pragma unroll
            for (int n = 0; n < D / 16; ++n)
#pragma unroll
                for (int c = 0; c < 4; ++c) oacc[n][c] = 0.f;
            const int first = (cw - static_cast<int>(page_ctr % kConsumerWarps) + kConsumerWarps) %
                              kConsumerWarps;
            for (int pg = it.pg0 + first; pg < it.pg1; pg += kConsumerWarps) {
                const uint32_t c = page_ctr + (pg - it.pg0);
                const uint32_t s = c % kStages, k = c / kStages;
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[s], k & 1, wait_limit())) ||
                    *static_cast<volatile int *>(&s_abort)) {
                    bad = true;
                    break;
                }
                const uint32_t kaddr = smem_addr(smem + s * 2 * C::kPageBytes);
                const int t_lo = max(0, it.tok0 - pg * kBlock);
                const int t_hi = min(kBlock, it.tok1 - pg * kBlock);
                if (t_lo == 0 && t_hi == kBlock)
                    consume_page_mma<D, true, (S > kRing)>(kaddr, kaddr + C::kPageBytes, 0, kBlock, qa,
                                                           p.qscale, m2, l2, oacc, lane);
                else
                    consume_page_mma<D, false, (S > kRing)>(kaddr, kaddr + C::kPageBytes, t_lo, t_hi,
                                                            qa, p.qscale, m2, l2, oacc, lane);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            page_ctr += static_cast<uint32_t>(it.pg1 - it.pg0);
            if (bad && lane == 0) {
                raise_flag(p.err_flag, XS_FLAG_TIMEOUT);
                atomicExch(&s_abort, 1);
            }
            const int buf = item_ctr % C::kMergeBufs;
            unsigned char *mb = smem + C::kCombOff + buf * C::kCombBytes;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&freed[buf],
                                                           ((item_ctr / C::kMergeBufs) & 1) ^ 1,
                                                           wait_limit()))) {
                if (lane == 0) {
                    raise_flag(p.err_flag, XS_FLAG_TIMEOUT);
                    atomicExch(&s_abort, 1);
                }
                break;
            }
            float *cM = reinterpret_cast<float *>(mb + 32);
            float *cL = cM + kConsumerWarps * G;
            float *cO = cL + kConsumerWarps * G;
            if (cw == 0 && lane == 0) *reinterpret_cast<Item *>(mb) = it;
            // Each head's sum: the shares of the 8 threads that hold it.
            float lsum[2] = {l2[0], l2[1]};
#pragma unroll
            for (int o = 4; o <= 16; o <<= 1)
#pragma unroll
                for (int e = 0; e < 2; ++e) lsum[e] += __shfl_xor_sync(0xffffffffu, lsum[e], o);
            if (!done) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int h = 2 * tq + e;
                    if (h >= G) continue;
                    float *dst = &cO[(cw * G + h) * D + grp];
#pragma unroll
                    for (int dn = 0; dn < D / 16; ++dn) {
                        dst[16 * dn] = oacc[dn][e];
                        dst[16 * dn + 8] = oacc[dn][e + 2];
                    }
                    if (grp == 0) {
                        cM[h * kConsumerWarps + cw] = m2[e];
                        cL[h * kConsumerWarps + cw] = lsum[e];
                    }
                }
            }
            if (!hand_over(it, mb, buf, item_ctr, done)) break;
            if (done || *static_cast<volatile int *>(&s_abort)) break;
        }
    } else {
        const int j = lane & 7;
        float2 *W2 = reinterpret_cast<float2 *>(smem + C::kWOff) + cw * kBlock * G;
        uint32_t page_ctr = 0;

        for (uint32_t item_ctr = 0;; ++item_ctr) {
            // Every consumer sees the producer's end marker (b < 0) in the same
            // slot and leaves; warp 0 passes the marker on to the merger.  A
            // failed (timed-out) wait marks the item bad: the warp skips its pages.
            // All waits in the CTA are bounded, so no warp can wait forever.
            const uint32_t slot = item_ctr & 1;
            bool bad = !__all_sync(0xffffffffu,
                                   mbar_wait_bounded(&qfull[slot], (item_ctr >> 1) & 1, wait_limit()));
            Item it = item_slot[slot];
            const bool done = !bad && it.b < 0;
            float qf[G][C::kQkDims];
            if (!done) {
                const unsigned char *qs = smem + C::kQSlotOff + slot * C::kQBytes;
    #pragma unroll
                for (int h = 0; h < G; ++h)
    #pragma unroll
                    for (int c = 0; c < C::kChunksPerLane; ++c) {
                        const uint4 raw = *reinterpret_cast<const uint4 *>(
                            qs + h * C::kRowBytes + (j + 8 * c) * 16);
                        float f[C::kElemsPerChunk];
                        unpack16(raw, f, static_cast<T *>(nullptr));
    #pragma unroll
                        for (int e = 0; e < C::kElemsPerChunk; ++e)
                            qf[h][c * C::kElemsPerChunk + e] = f[e] * p.qscale;
                    }
                __syncwarp();
                if (lane == 0 && !bad) mbar_arrive(&qempty[slot]);
            }
            if (bad || done) {
                it.b = -1;
                it.pg0 = it.pg1 = 0;
            }

            float m_own = -INFINITY, l_own = 0.f;
            float2 o[G][C::kPvDims / 2];
    #pragma unroll
            for (int h = 0; h < G; ++h)
    #pragma unroll
                for (int d = 0; d < C::kPvDims / 2; ++d) o[h][d] = make_float2(0.f, 0.f);

            // Pages of this item for this warp: page_ctr advances over every page of
            // the item; this warp takes those with page_ctr % kConsumerWarps == cw.
            const int first = (cw - static_cast<int>(page_ctr % kConsumerWarps) + kConsumerWarps) %
                              kConsumerWarps;
            for (int pg = it.pg0 + first; pg < it.pg1; pg += kConsumerWarps) {
                const uint32_t c = page_ctr + (pg - it.pg0);
                const uint32_t s = c % kStages, k = c / kStages;
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[s], k & 1, wait_limit())) ||
                    *static_cast<volatile int *>(&s_abort)) {
                    bad = true;
                    break;
                }
                const unsigned char *Ks = smem + s * 2 * C::kPageBytes;
                const unsigned char *Vs = Ks + C::kPageBytes;
                const int t_lo = max(0, it.tok0 - pg * kBlock);
                const int t_hi = min(kBlock, it.tok1 - pg * kBlock);
                if (t_lo == 0 && t_hi == kBlock)
                    consume_page<T, D, G, true>(Ks, Vs, 0, kBlock, qf, m_own, l_own, o, W2, lane);
                else
                    consume_page<T, D, G, false>(Ks, Vs, t_lo, t_hi, qf, m_own, l_own, o, W2, lane);
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            page_ctr += static_cast<uint32_t>(it.pg1 - it.pg0);
            if (bad && lane == 0) {
                raise_flag(p.err_flag, XS_FLAG_TIMEOUT);
                atomicExch(&s_abort, 1);
            }

            // ---- hand this warp's state to the merger (buffer item_ctr % kMergeBufs;
            // a buffer is reused once the merger has freed it).
            const int buf = item_ctr % C::kMergeBufs;
            unsigned char *mb = smem + C::kCombOff + buf * C::kCombBytes;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&freed[buf],
                                                           ((item_ctr / C::kMergeBufs) & 1) ^ 1,
                                                           wait_limit()))) {
                if (lane == 0) {
                    raise_flag(p.err_flag, XS_FLAG_TIMEOUT);
                    atomicExch(&s_abort, 1);
                }
                break;
            }
            float *cM = reinterpret_cast<float *>(mb + 32);
            float *cL = cM + kConsumerWarps * G;
            float *cO = cL + kConsumerWarps * G;
            if (cw == 0 && lane == 0) *reinterpret_cast<Item *>(mb) = it;
            if (!done) {
    #pragma unroll
                for (int h = 0; h < G; ++h) {
                    float *dst = &cO[(cw * G + h) * D + lane * C::kPvDims];
                    if constexpr (C::kPvDims == 4)
                        *reinterpret_cast<float4 *>(dst) =
                            make_float4(o[h][0].x, o[h][0].y, o[h][1].x, o[h][1].y);
                    else
                        *reinterpret_cast<float2 *>(dst) = o[h][0];
                }
                if (lane < 8 && (j & ((1 << C::kHeadShift) - 1)) == 0) {
                    const int own_head = j >> C::kHeadShift;
                    cM[own_head * kConsumerWarps + cw] = m_own;
                    cL[own_head * kConsumerWarps + cw] = l_own;
                }
            }
            if (!hand_over(it, mb, buf, item_ctr, done)) break;
            if (done || *static_cast<volatile int *>(&s_abort)) break;
        }
    }
    // Combine jobs from the merger (one per split group completed after the
    // producer ran out of items), each shared by the four consumer warps.
    // This warp's scratch is its own first ring stage: every page copied
    // into it has been consumed by now.
    if (kJobs && p.combine && !*static_cast<volatile int *>(&s_abort)) {
        const int scratch_off = static_cast<int>(smem - smem_raw) + cw * 2 * C::kPageBytes;
        for (uint32_t k = 0;; ++k) {
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&s_job_full, k & 1, wait_limit()))) {
                if (lane == 0) {
                    raise_flag(p.err_flag, XS_FLAG_TIMEOUT);
                    atomicExch(&s_abort, 1);
                }
                break;
            }
            const int jb = s_job[0], jg = s_job[1], jnp = s_job[2];
            if (jb < 0) break;
            combine_quarter<T, D, G>(p, jb, jg, jnp, cw, lane, scratch_off);
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_job_done);
        }
    }
    exit_role();
}

// ---------------------------------------------------------------- cluster step
//
// A one-launch step whose (sequence, KV head) groups all fit one wave of
// thread-block clusters runs as one cluster per group instead of the
// persistent grid: CTA r of the cluster takes partition r of the group's
// tokens, copies all of its pages into shared memory at once (one warp
// issues them, one lane per page) and eight consumer warps attend over them
// (consume_page_mma).  The consumers' eight states are merged into the CTA's
// partial (m, l, unnormalised o per head) in its own shared memory; after a
// cluster barrier every CTA combines a slice of the group's output from all
// partials, read over distributed shared memory:
//     out = sum_r 2^(m_r - M) o_r / (sum_r 2^(m_r - M) l_r  [+ 2^(sink - M)])
// (flash-decoding's split-K combine).  No partial leaves the GPC and no
// count goes through global memory, which is what a small launch's latency
// is made of.  A second cluster barrier keeps every CTA's shared memory
// alive until the others have read it.  Every wait is bounded; a wait that
// runs out raises XS_FLAG_TIMEOUT, and every thread still reaches both
// cluster barriers, so no CTA waits for one that left.
constexpr int kCluConsumers = 8;
constexpr int kCluThreads = 32 * (1 + kCluConsumers);  // producer + consumers
constexpr int kCluStages = 24;    // ring stages (page pairs) of a CTA
constexpr int kCluMaxSize = 16;   // CTAs per cluster (the non-portable maximum)
// Pages of a partition up to which clusters were measured faster than the
// persistent grid over every SM (a 32768-token sequence split 12 ways is
// 171 pages a CTA: 27.5 against 30.8 us); beyond, the persistent grid.
constexpr int kCluMaxPartPages = 192;
// Pages of a partition up to which a launch trades larger partitions for a
// spare cluster slot (cluster_plan).
constexpr int kCluSpareMaxPages = 32;

template <int D, int G>
struct CluCfg {
    static constexpr int kRowBytes = D * 2;
    static constexpr int kPageBytes = kBlock * kRowBytes;
    static constexpr int kStageBytes = 2 * kPageBytes;  // K page, then V page (swizzled)
    // The CTA's partial: m[8], l[8], o[G][D] (fp32, o not divided by l).
    // A consumer's state has the same layout and goes in the consumer's
    // first stage, which only it ever reads.
    static constexpr int kPartOff = kCluStages * kStageBytes;
    static constexpr int kPartBytes = 64 + G * D * 4;
    static constexpr int kBarOff = kPartOff + kPartBytes;
    static constexpr int kBarBytes = 2 * kCluStages * 8;  // full, then empty
    static constexpr int kAlignSlack = 1024;  // the stages are 1024-byte aligned
    static constexpr int kBytes = kBarOff + kBarBytes + kAlignSlack;
    // D = 64: a 98 KB ring and fewer registers, so two CTAs share an SM and
    // twice as many clusters fit at once.
    static constexpr int kMinBlocks = D == 64 ? 2 : 1;
    static_assert(kPartBytes <= kStageBytes, "a consumer state fits its stage");
    static_assert(kCluStages >= kCluConsumers && kCluStages <= 32, "one lane per page");
    static_assert(kPartOff % 16 == 0 && kBarOff % 8 == 0, "float4 partial rows, 8-byte barriers");
};

__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// The same barrier without ordering this thread's earlier memory accesses:
// for a barrier that only has to know the other CTAs are past their reads of
// this CTA's shared memory (values they have already used), so the arrive
// need not wait for this thread's global stores to complete.
__device__ __forceinline__ void cluster_barrier_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed;\n\tbarrier.cluster.wait;" ::: "memory");
}
// The address of a shared-memory location in cluster CTA `rank`.
__device__ __forceinline__ uint32_t dsmem_map(uint32_t local, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(local), "r"(rank));
    return a;
}
__device__ __forceinline__ float dsmem_ld_f32(uint32_t a) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ float4 dsmem_ld_v4(uint32_t a) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(a)
                 : "memory");
    return v;
}

// Grid (cluster size, B * Hkv), clusters along x: blockIdx.y = b * Hkv + g,
// blockIdx.x = the partition.  p.P is the partition length (a multiple of
// 16; with a window a partition's start need not fall on a page); the host
// picked it so that gridDim.x partitions cover every sequence.  A CTA's
// pages go round a ring of kCluStages stages; page i uses stage
// i % kCluStages and consumer i % kCluConsumers, so every stage belongs to
// one consumer.
template <int D, int G>
__global__ void __launch_bounds__(kCluThreads, CluCfg<D, G>::kMinBlocks)
    paged_decode_cluster_kernel(const __grid_constant__ CUtensorMap tmk,
                                const __grid_constant__ CUtensorMap tmv, const Params p) {
    using C = CluCfg<D, G>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
    uint64_t *empty = full + kCluStages;
    float *part = reinterpret_cast<float *>(smem + C::kPartOff);
    __shared__ int s_abort;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = blockIdx.x, cs = gridDim.x;
    const int b = blockIdx.y / p.Hkv, g = blockIdx.y - b * p.Hkv;
    // Uniform over the launch, so every CTA of every cluster returns here
    // together (before any cluster barrier).
    if (dynamic_smem_bytes() < static_cast<uint32_t>(C::kBytes) || b >= p.B) {
        if (tid == 0) raise_flag(p.err_flag, XS_FLAG_CONFIG);
        return;
    }
    if (tid == 0) {
        for (int i = 0; i < 2 * kCluStages; ++i) mbar_init(&full[i], 1);  // full, then empty
        mbar_fence_init();
        s_abort = 0;
    }
    __syncthreads();
    // This CTA's tokens [tok0, tok1) of the window [first_token, n), its
    // pages [pg0, pg0 + np).  Lengths are read after the launch wait, or
    // before it with p.early (the caller promises the previous launch does
    // not write them).
    auto range = [&](int n, int &tok0, int &tok1, int &pg0, int &np) {
        tok0 = first_token(p, n) + r * p.P;
        tok1 = min(n, tok0 + p.P);
        pg0 = tok0 / kBlock;
        np = tok1 > tok0 ? (tok1 + kBlock - 1) / kBlock - pg0 : 0;
    };
    int n_seq;  // the sequence's length (clamped to the table), read once per thread
    if (warp == 0) {
        // ======================================================== producer
        if (!p.early) {
            griddep_wait();
            griddep_launch_dependents();
        }
        // Without a window the partition's first page does not depend on the
        // length: its first ring of block ids is requested together with the
        // length (entries past the sequence are read but not used).
        const bool no_window = p.window == 0;
        const int pg_first = (r * p.P) / kBlock;
        int32_t id_early = 0;
        if (no_window && lane < kCluStages && pg_first + lane < p.max_blocks &&
            XS_BOUNDS(b < p.B && pg_first + lane >= 0, p.err_flag))
            id_early = p.block_tables[static_cast<int64_t>(b) * p.table_stride + pg_first + lane];
        const int n = seq_len(p, b, r == 0 && g == 0 && lane == 0);
        n_seq = n;
        int tok0, tok1, pg0, np;
        range(n, tok0, tok1, pg0, np);
        // The page holding the sequence's last token receives this step's
        // row: it is copied after the row is written (and only when the
        // length is within the table, as in the separate append).
        const int raw_len = p.k_new && tok1 == n && np > 0 ? p.context_lens[b] : 0;
        const bool appends = raw_len == n && n > 0;
        const int last = appends ? np - 1 : -1;
        const uint64_t pol = policy_evict_first();
        // Pages go round the ring kCluStages at a time, lane j issuing page
        // base + j into stage j.  An id outside the pool reads block 0
        // instead (flagged) and takes no appended row.
        auto check_id = [&](int32_t id) {
            if (id < 0 || id >= p.num_blocks) {
                raise_flag(p.err_flag, XS_FLAG_BAD_BLOCK);
                id = -1;
            }
            return id;
        };
        auto load_id = [&](int i) {
            if (i >= np || !XS_BOUNDS(pg0 + i >= 0 && pg0 + i < p.max_blocks, p.err_flag)) return 0;
            return check_id(p.block_tables[static_cast<int64_t>(b) * p.table_stride + pg0 + i]);
        };
        int my_last = -1;  // the last page this lane issued (its stage's last phase)
        auto issue = [&](int i, int32_t id) {
            // (The debug library can skip one page of CTA (0, 0) to make a
            // consumer's wait run out.)
            if (blockIdx.y == 0 && skip_page(static_cast<uint32_t>(i))) return;
            const int st = i % kCluStages;
            const uint32_t dk = smem_addr(smem + st * C::kStageBytes);
            const int page = max(id, 0) * p.Hkv + g;
            mbar_arrive_expect_tx(&full[st], 2 * C::kPageBytes);
            tma_load_4d(dk, &tmk, page, &full[st], pol);
            tma_load_4d(dk + C::kPageBytes, &tmv, page, &full[st], pol);
            my_last = i;
        };
        const bool first = lane < kCluStages && lane < np;
        const int32_t id0 = !first ? 0 : no_window ? check_id(id_early) : load_id(lane);
        if (first && lane != last) issue(lane, id0);
        if (p.early) {
            griddep_wait();
            griddep_launch_dependents();
        }
        if (appends) {
            // K row then V row, one 16-byte chunk per lane, into slot (n - 1)
            // of the last page; then the generic-proxy writes are ordered
            // before the tensor copy that reads the page.
            constexpr int kChunks = C::kRowBytes / 16;
            const bool in_table = XS_BOUNDS(pg0 + last < p.max_blocks && b < p.B, p.err_flag);
            const int32_t lid = !in_table ? -1
                                : last < kCluStages ? __shfl_sync(0xffffffffu, id0, last)
                                                    : p.block_tables[static_cast<int64_t>(b) *
                                                                         p.table_stride + pg0 + last];
            const bool ok_id = lid >= 0 && lid < p.num_blocks;
            const int64_t row = static_cast<int64_t>(b) * p.Hkv + g;
            const int64_t dst =
                ((static_cast<int64_t>(lid) * p.Hkv + g) * kBlock + (n - 1) % kBlock) * kChunks;
            for (int c = lane; ok_id && c < 2 * kChunks; c += 32) {
                const bool is_k = c < kChunks;
                const int cc = is_k ? c : c - kChunks;
                const uint4 v = static_cast<const uint4 *>(is_k ? p.k_new : p.v_new)[row * kChunks + cc];
                static_cast<uint4 *>(const_cast<void *>(is_k ? p.k_cache : p.v_cache))[dst + cc] = v;
            }
            fence_proxy_async_global();
            __syncwarp();
            if (last < kCluStages && lane == last) issue(lane, id0);  // (later: in the ring loop)
        }
        // The rest of the pages, each into its stage once the consumer has
        // released the stage's previous page (bounded wait).
        bool ok = true;
        for (int base = kCluStages; ok && base < np; base += kCluStages) {
            const int i = base + lane;
            const bool mine = lane < kCluStages && i < np;
            const int32_t id = mine ? load_id(i) : 0;
            bool w = true;
            if (mine) {
                w = mbar_wait_bounded(&empty[lane], (base / kCluStages - 1) & 1, wait_limit());
                if (w) issue(i, id);
            }
            ok = __all_sync(0xffffffffu, w);
        }
        if (!ok && lane == 0) {
            raise_flag(p.err_flag, XS_FLAG_TIMEOUT);
            atomicExch(&s_abort, 1);
        }
        // Every copy issued lands before the CTA can exit: in the normal
        // path the consumers have waited for all of them; after an abort
        // this wait (bounded) covers the ones they gave up on - per stage
        // the last page issued, whose phase is the only one that can still
        // be open.  Done after the first cluster barrier, when the consumers
        // are finished.
        cluster_barrier();
        if (my_last >= 0)
            mbar_wait_bounded(&full[my_last % kCluStages], (my_last / kCluStages) & 1, wait_limit());
    } else {
        // ======================================================== consumers
        griddep_wait();
        griddep_launch_dependents();
        const int cw = warp - 1;
        const int grp = lane >> 2, tq = lane & 3;
        // The G query rows straight from global memory into the B fragments
        // (lane quad grp holds head grp; rows G..7 zero), requested together
        // with the length: one round trip after the launch wait, nothing
        // staged.
        uint32_t qa[D / 16][2];
        const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
            static_cast<const unsigned char *>(p.q) +
            ((static_cast<int64_t>(b) * p.Hq + static_cast<int64_t>(g) * G + (grp < G ? grp : 0)) *
             C::kRowBytes));
        const bool q_in = grp < G && XS_BOUNDS((g + 1) * G <= p.Hq && b < p.B, p.err_flag);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            qa[ks][0] = q_in ? qrow[8 * ks + tq] : 0u;
            qa[ks][1] = q_in ? qrow[8 * ks + 4 + tq] : 0u;
        }
        const int n = seq_len(p, b, false);
        n_seq = n;
        int tok0, tok1, pg0, np;
        range(n, tok0, tok1, pg0, np);
        float m2[2] = {-INFINITY, -INFINITY}, l2[2] = {0.f, 0.f};
        float oacc[D / 16][4];
#pragma unroll
        for (int i = 0; i < D / 16; ++i)
#pragma unroll
            for (int c = 0; c < 4; ++c) oacc[i][c] = 0.f;
        if (cw < np) {
            bool ok = true;
            for (int i = cw; ok && i < np; i += kCluConsumers) {
                const int st = i % kCluStages;
                if (!__all_sync(0xffffffffu,
                                mbar_wait_bounded(&full[st], (i / kCluStages) & 1, wait_limit())) ||
                    *static_cast<volatile int *>(&s_abort)) {
                    ok = false;
                    break;
                }
                const uint32_t kaddr = smem_addr(smem + st * C::kStageBytes);
                const int pg = pg0 + i;
                const int t_lo = max(0, tok0 - pg * kBlock);
                const int t_hi = min(kBlock, tok1 - pg * kBlock);
                if (t_lo == 0 && t_hi == kBlock)
                    consume_page_mma<D, true, true>(kaddr, kaddr + C::kPageBytes, 0, kBlock, qa,
                                                    p.qscale, m2, l2, oacc, lane);
                else
                    consume_page_mma<D, false, true>(kaddr, kaddr + C::kPageBytes, t_lo, t_hi, qa,
                                                     p.qscale, m2, l2, oacc, lane);
                // The stage's next page may come in once every lane has its
                // fragments of this one.
                __syncwarp();
                if (i + kCluStages < np && lane == 0) mbar_arrive(&empty[st]);
            }
            if (!ok && lane == 0) {
                raise_flag(p.err_flag, XS_FLAG_TIMEOUT);
                atomicExch(&s_abort, 1);
            }
        }
        // This consumer's state into its own stage (its first page, consumed).
        float lsum[2] = {l2[0], l2[1]};
#pragma unroll
        for (int o = 4; o <= 16; o <<= 1)
#pragma unroll
            for (int e = 0; e < 2; ++e) lsum[e] += __shfl_xor_sync(0xffffffffu, lsum[e], o);
        float *st = reinterpret_cast<float *>(smem + cw * C::kStageBytes);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int h = 2 * tq + e;
            if (h >= G) continue;
            float *dst = st + 16 + h * D + grp;
#pragma unroll
            for (int dn = 0; dn < D / 16; ++dn) {
                dst[16 * dn] = oacc[dn][e];
                dst[16 * dn + 8] = oacc[dn][e + 2];
            }
            if (grp == 0) {
                st[h] = m2[e];
                st[8 + h] = lsum[e];
            }
        }
        named_barrier_sync(1, 32 * kCluConsumers);
        // The eight states merged into the CTA's partial, a float4 of one
        // head per thread.
        for (int c = tid - 32; c < G * D / 4; c += 32 * kCluConsumers) {
            const int h = c / (D / 4), d = (c - h * (D / 4)) * 4;
            float mx = -INFINITY;
#pragma unroll
            for (int w = 0; w < kCluConsumers; ++w)
                mx = fmaxf(mx, reinterpret_cast<const float *>(smem + w * C::kStageBytes)[h]);
            const float ref = mx == -INFINITY ? 0.f : mx;
            float lt = 0.f;
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < kCluConsumers; ++w) {
                const float *sw = reinterpret_cast<const float *>(smem + w * C::kStageBytes);
                const float f = fast_exp2(sw[h] - ref);  // 0 for a consumer with no pages
                lt += f * sw[8 + h];
                const float4 v = *reinterpret_cast<const float4 *>(sw + 16 + h * D + d);
                o.x += f * v.x;
                o.y += f * v.y;
                o.z += f * v.z;
                o.w += f * v.w;
            }
            *reinterpret_cast<float4 *>(part + 16 + h * D + d) = o;
            if (d == 0) {
                part[h] = mx;
                part[8 + h] = lt;
            }
        }
        cluster_barrier();
    }
    // ============================================================ combine
    // Every partial of the group is in place.  This CTA writes float4
    // chunks r, r + cs, ... of the group's G x D outputs; a half-warp per
    // chunk, lane j of it reading partial j.
    {
        constexpr int kChunks = G * D / 4;
        constexpr int kHalves = 2 * (kCluThreads / 32);
        const int j = lane & 15;
        const int n = n_seq;
        const uint32_t remote = dsmem_map(smem_addr(part), static_cast<uint32_t>(j < cs ? j : 0));
        for (int k0 = 2 * warp; r + k0 * cs < kChunks; k0 += kHalves) {
            const int c = r + (k0 + (lane >> 4)) * cs;
            const bool valid = c < kChunks;
            const int h = valid ? c / (D / 4) : 0, d = valid ? (c - h * (D / 4)) * 4 : 0;
            float mj = -INFINITY, lj = 0.f;
            float4 oj = make_float4(0.f, 0.f, 0.f, 0.f);
            if (valid && j < cs) {
                mj = dsmem_ld_f32(remote + 4 * h);
                lj = dsmem_ld_f32(remote + 4 * (8 + h));
                oj = dsmem_ld_v4(remote + 4 * (16 + h * D + d));
            }
            float mx = mj;
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float ref = mx == -INFINITY ? 0.f : mx;
            const float f = fast_exp2(mj - ref);
            float s[5] = {f * lj, f * oj.x, f * oj.y, f * oj.z, f * oj.w};
#pragma unroll
            for (int o = 1; o < 16; o <<= 1)
#pragma unroll
                for (int e = 0; e < 5; ++e) s[e] += __shfl_xor_sync(0xffffffffu, s[e], o);
            if (valid && j == 0 && XS_BOUNDS(g * G + h < p.Hq && b < p.B, p.err_flag)) {
                float den = s[0];
                if (p.sinks)
                    den += fast_exp2(Elem<__nv_bfloat16>::to_f32(
                                         static_cast<const __nv_bfloat16 *>(p.sinks)[g * G + h]) *
                                         kLog2e -
                                     ref);
                // A sequence with no tokens produces zeros.
                const float inv = n > 0 ? 1.f / den : 0.f;
                const float o4[4] = {s[1] * inv, s[2] * inv, s[3] * inv, s[4] * inv};
                store_row<__nv_bfloat16, 4>(
                    static_cast<__nv_bfloat16 *>(p.out) +
                        (static_cast<int64_t>(b) * p.Hq + static_cast<int64_t>(g) * G + h) * D + d,
                    o4);
            }
        }
    }
    // No CTA leaves while another may still read its partial.  (Every read of
    // a partial has delivered its value, which the reader used before it
    // arrives; the output stores need not complete before the exit.)
    cluster_barrier_relaxed();
}

// Split-K combine: one CTA of D threads per (sequence, query head).
// With sinks, a sink is one more logit (no value row) in the denominator;
// with a window, only the last `window` tokens were split into partitions.
template <typename T>
__global__ void paged_decode_reduce_kernel(T *__restrict__ out, const float *__restrict__ part_o,
                                           const float *__restrict__ part_m,
                                           const float *__restrict__ part_l,
                                           const int32_t *__restrict__ lens, int Hq, int D, int P,
                                           int max_parts, const T *__restrict__ sinks,
                                           int window, int prefill_start) {
    const int bh = blockIdx.x;
    const int b = bh / Hq;
    int n = prefill_start >= 0 ? prefill_start + b + 1 : lens[b];
    if (window > 0 && n > window) n = window;
    int np = n > 0 ? (n + P - 1) / P : 0;
    np = min(np, max_parts);
    if (np <= 1) return;
    const int64_t base = static_cast<int64_t>(bh) * max_parts;
    float mx = -INFINITY;
#pragma unroll 8
    for (int i = 0; i < np; ++i) mx = fmaxf(mx, part_m[base + i]);
    const int d = threadIdx.x;
    float lt = 0.f, acc = 0.f;
#pragma unroll 8
    for (int i = 0; i < np; ++i) {
        const float f = fast_exp2(part_m[base + i] - mx) * part_l[base + i];
        lt += f;
        if (d < D) acc += f * part_o[(base + i) * D + d];
    }
    if (sinks) lt += fast_exp2(Elem<T>::to_f32(sinks[bh % Hq]) * kLog2e - mx);
    if (d < D) out[static_cast<int64_t>(bh) * D + d] = Elem<T>::from_f32(acc / lt);
}

// ------------------------------------------------------------------ host side

using KernelFn = void (*)(const CUtensorMap, const CUtensorMap, const Params);

template <typename T, int D, int G, int S>
KernelFn kernel_for() {
    return paged_decode_kernel<T, D, G, S>;
}

// The kernel for a shape, with the deep ring when asked and instantiated
// (bf16, D = 128).
KernelFn pick_kernel(int dtype, int D, int G, bool deep, int *smem_base_fn_B0) {
#define XS_PICK(TT, DD, GG)                                                          \
    if (D == DD && G == GG) {                                                        \
        *smem_base_fn_B0 = Cfg<TT, DD, GG>::kPrefixOff;                              \
        return kernel_for<TT, DD, GG, kRing>();                                      \
    }
#define XS_PICK_DEEP(TT, DD, GG)                                                     \
    if (D == DD && G == GG) {                                                        \
        *smem_base_fn_B0 = Cfg<TT, DD, GG, kDeepRing>::kPrefixOff;                   \
        return kernel_for<TT, DD, GG, kDeepRing>();                                  \
    }
    if (dtype == XS_BF16 && deep) {
        XS_PICK_DEEP(__nv_bfloat16, 128, 1) XS_PICK_DEEP(__nv_bfloat16, 128, 2)
        XS_PICK_DEEP(__nv_bfloat16, 128, 4) XS_PICK_DEEP(__nv_bfloat16, 128, 8)
    }
    if (dtype == XS_BF16) {
        XS_PICK(__nv_bfloat16, 64, 1) XS_PICK(__nv_bfloat16, 64, 2)
        XS_PICK(__nv_bfloat16, 64, 4) XS_PICK(__nv_bfloat16, 64, 8)
        XS_PICK(__nv_bfloat16, 128, 1) XS_PICK(__nv_bfloat16, 128, 2)
        XS_PICK(__nv_bfloat16, 128, 4) XS_PICK(__nv_bfloat16, 128, 8)
    } else if (dtype == XS_F32) {
        XS_PICK(float, 64, 1) XS_PICK(float, 64, 2) XS_PICK(float, 64, 4) XS_PICK(float, 64, 8)
        XS_PICK(float, 128, 1) XS_PICK(float, 128, 2) XS_PICK(float, 128, 4)
        XS_PICK(float, 128, 8)
    }
#undef XS_PICK
#undef XS_PICK_DEEP
    return nullptr;
}

template <int D, int G>
KernelFn cluster_kernel_for() {
    return paged_decode_cluster_kernel<D, G>;
}

// The cluster-step kernel for a shape (bf16, D = 64 or 128) and its dynamic
// shared memory, or null.
KernelFn pick_cluster_kernel(int D, int G, int *smem) {
#define XS_PICK_CLU(DD, GG)                                                          \
    if (D == DD && G == GG) {                                                        \
        *smem = CluCfg<DD, GG>::kBytes;                                              \
        return cluster_kernel_for<DD, GG>();                                         \
    }
    XS_PICK_CLU(128, 1) XS_PICK_CLU(128, 2) XS_PICK_CLU(128, 4) XS_PICK_CLU(128, 8)
    XS_PICK_CLU(64, 1) XS_PICK_CLU(64, 2) XS_PICK_CLU(64, 4) XS_PICK_CLU(64, 8)
#undef XS_PICK_CLU
    return nullptr;
}

// Clusters of `cs` CTAs of a cluster-step kernel that an idle device holds at
// once (0 if none, or if a query failed), cached per (kernel, device, cs).
int cluster_capacity(KernelFn fn, int smem, int cs) {
    struct Entry {
        KernelFn fn;
        int dev, cs, n;
    };
    static std::mutex mu;
    static Entry cache[64];
    static int n_cached = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    bool configured = false;
    for (int i = 0; i < n_cached; ++i) {
        if (cache[i].fn == fn && cache[i].dev == dev && cache[i].cs == cs) return cache[i].n;
        configured |= cache[i].fn == fn && cache[i].dev == dev;
    }
    int n = 0;
    const void *f = reinterpret_cast<const void *>(fn);
    if (configured ||
        (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess &&
         cudaFuncSetAttribute(f, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess)) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cs, 1);
        cfg.blockDim = dim3(kCluThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute a[1];
        a[0].id = cudaLaunchAttributeClusterDimension;
        a[0].val.clusterDim.x = cs;
        a[0].val.clusterDim.y = 1;
        a[0].val.clusterDim.z = 1;
        cfg.attrs = a;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();  // do not leave a failed query for an unrelated later check
    if (n_cached < 64) cache[n_cached++] = Entry{fn, dev, cs, n};
    return n;
}

// Whether a one-launch step runs as clusters (paged_decode_cluster_kernel):
// bf16, and every (sequence, KV head) group's tokens - at most the
// table's reach, or the window - split into cs partitions of at most
// kCluMaxPartPages pages (one fewer with a window) with all B * Hkv clusters
// resident at once.  The largest such cs up to 16 (and no more than one
// partition per 64 tokens) is taken - the fewer pages a CTA holds, the
// shorter the launch - unless it fills every cluster slot with partitions of
// at most kCluSpareMaxPages pages: then the largest smaller cs that leaves a
// slot free, if its partitions are at most half as long again.  Returns cs
// (0: the persistent grid) and sets the partition length, kernel and shared
// memory.
int cluster_plan(int B, int Hkv, int D, int G, int max_blocks, int window, int dtype, int *P,
                 KernelFn *fn, int *smem) {
    if (dtype != XS_BF16 || static_cast<int64_t>(B) * Hkv > 65535) return 0;
    *fn = pick_cluster_kernel(D, G, smem);
    if (!*fn) return 0;
    int64_t L = static_cast<int64_t>(max_blocks) * kBlock;
    if (window > 0) L = std::min<int64_t>(L, window);
    const int extra = window > 0 ? 1 : 0;  // a window's first token need not start a page
    const int64_t groups = static_cast<int64_t>(B) * Hkv;
    // More groups than even the smallest clusters can hold at once: no
    // cluster size fits (the common case for large batches, settled here
    // with one cached lookup).
    if (groups > cluster_capacity(*fn, *smem, 2)) return 0;
    auto part_of = [&](int cs) { return ((L + cs - 1) / cs + kBlock - 1) / kBlock * kBlock; };
    int fit = 0;
    for (int cs = static_cast<int>(std::min<int64_t>(kCluMaxSize, (L + 63) / 64)); cs >= 2; --cs) {
        if (part_of(cs) / kBlock + extra > kCluMaxPartPages) return 0;  // fewer CTAs only add pages
        if (groups <= cluster_capacity(*fn, *smem, cs)) {
            fit = cs;
            break;
        }
    }
    if (fit == 0) return 0;
    // A launch that fills the device's cluster slots exactly leaves the next
    // launch nowhere to start until it ends; with a slot to spare, the next
    // layer's first clusters begin (and read their pages early) while this
    // one finishes.  For short partitions that overlap is worth more than a
    // few extra pages a CTA: measured per layer, one 4,097-token sequence
    // with 8 KV heads ran 6.26 us at cs = 12 (8 slots, 22 pages a CTA) and
    // 5.64 us at cs = 10 (13 slots, 26 pages); at 8,192 tokens (43 pages at
    // cs = 12) the extra pages cost more (9.78 against 10.24 us).
    int cs = fit;
    const int64_t fit_pages = part_of(fit) / kBlock;
    if (groups == cluster_capacity(*fn, *smem, fit) && fit_pages <= kCluSpareMaxPages) {
        for (int c = fit - 1; c >= 2 && 2 * (part_of(c) / kBlock) <= 3 * fit_pages; --c)
            if (groups < cluster_capacity(*fn, *smem, c)) {
                cs = c;
                break;
            }
    }
    *P = static_cast<int>(part_of(cs));
    return cs;
}

struct DeviceInfo {
    int sms = 0;
    int max_smem_optin = 0;
    int smem_per_sm = 0;         // shared memory of one SM
    int reserved_per_block = 0;  // what the system keeps of it per resident CTA
};

int device_info(DeviceInfo *info) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return XS_EDEVICE;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev].sms == 0) {
        DeviceInfo d;
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                   dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                                   dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.reserved_per_block, cudaDevAttrReservedSharedMemoryPerBlock,
                                   dev) != cudaSuccess)
            return XS_EDEVICE;
        cache[dev] = d;
    }
    *info = cache[dev];
    return XS_OK;
}

// Static shared memory of a kernel, cached.
int static_smem(KernelFn fn, int *bytes) {
    struct Entry {
        KernelFn fn;
        int bytes;
    };
    static std::mutex mu;
    static Entry cache[32];
    static int n_cached = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_cached; ++i)
        if (cache[i].fn == fn) {
            *bytes = cache[i].bytes;
            return XS_OK;
        }
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, reinterpret_cast<const void *>(fn)) != cudaSuccess) {
        cudaGetLastError();
        return XS_ELAUNCH;
    }
    *bytes = static_cast<int>(fa.sharedSizeBytes);
    if (n_cached < 32) cache[n_cached++] = Entry{fn, *bytes};
    return XS_OK;
}

// Resident CTAs per SM for a kernel at a given dynamic smem size (raises the
// kernel's smem limit first).  Cached per (kernel, device, smem size).
int occupancy(KernelFn fn, int smem, int *per_sm) {
    struct Entry {
        KernelFn fn;
        int dev, smem, per_sm;
    };
    static std::mutex mu;
    static Entry cache[64];
    static int n_cached = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return XS_EDEVICE;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_cached; ++i)
        if (cache[i].fn == fn && cache[i].dev == dev && cache[i].smem == smem) {
            *per_sm = cache[i].per_sm;
            return XS_OK;
        }
    // Allow the kernel the device's whole opt-in shared memory once; the
    // attribute is never lowered, so any cached size stays launchable.
    bool raised = false;
    for (int i = 0; i < n_cached; ++i) raised |= cache[i].fn == fn && cache[i].dev == dev;
    if (!raised) {
        // Opt-in maximum minus the kernel's own static shared memory.
        int max_optin = 0;
        cudaFuncAttributes fa;
        if (cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess ||
            cudaFuncGetAttributes(&fa, reinterpret_cast<const void *>(fn)) != cudaSuccess ||
            cudaFuncSetAttribute(reinterpret_cast<const void *>(fn),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 max_optin - static_cast<int>(fa.sharedSizeBytes)) !=
                cudaSuccess) {
            cudaGetLastError();  // do not leave the failure for an unrelated later check
            return XS_ELAUNCH;
        }
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, reinterpret_cast<const void *>(fn),
                                                      kThreads, smem) != cudaSuccess) {
        cudaGetLastError();
        return XS_ELAUNCH;
    }
    *per_sm = n > 0 ? n : 1;
    Entry e{fn, dev, smem, *per_sm};
    if (n_cached < 64) cache[n_cached++] = e;  // a full cache just stops caching
    return XS_OK;
}

// Tensor maps of a K and a V pool (bf16), cached per pool and shape: a
// decode loop launches over the same pools every step.
int pool_maps(const void *k, const void *v, int64_t num_blocks, int Hkv, int D, CUtensorMap *tmk,
              CUtensorMap *tmv) {
    struct Entry {
        const void *k, *v;
        int64_t nb;
        int hkv, d;
        CUtensorMap mk, mv;
    };
    static std::mutex mu;
    static Entry cache[16];
    static int n_cached = 0, next = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_cached; ++i)
        if (cache[i].k == k && cache[i].v == v && cache[i].nb == num_blocks &&
            cache[i].hkv == Hkv && cache[i].d == D) {
            *tmk = cache[i].mk;
            *tmv = cache[i].mv;
            return XS_OK;
        }
    const cuuint64_t dims[4] = {64, kBlock, static_cast<cuuint64_t>(D / 64),
                                static_cast<cuuint64_t>(num_blocks) * Hkv};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, 128,
                                   static_cast<cuuint64_t>(kBlock) * D * 2};
    const cuuint32_t box[4] = {64, kBlock, static_cast<cuuint32_t>(D / 64), 1};
    int st = encode_bf16_map<4>(tmk, k, dims, strides, box);
    if (st == XS_OK) st = encode_bf16_map<4>(tmv, v, dims, strides, box);
    if (st != XS_OK) return st;
    Entry &e = cache[n_cached < 16 ? n_cached++ : (next++ % 16)];
    e = Entry{k, v, num_blocks, Hkv, D, *tmk, *tmv};
    return XS_OK;
}

}  // namespace attn
XS_DEFINE_BOUNDS_COUNTER(bounds_failures_decode)

}  // namespace xs

using namespace xs;

extern "C" int xs_version(void) { return 100; }

extern "C" int xs_debug_bounds_failures(int reset) {
#ifdef XS_DEBUG_BOUNDS
    int total = 0;
    for (const int v : {bounds_failures_append(reset), bounds_failures_decode(reset),
                        bounds_failures_prefill_tc(reset)}) {
        if (v < 0) return v;
        total += v;
    }
    return total;
#else
    (void)reset;
    return XS_EUNSUPPORTED;
#endif
}

extern "C" int xs_debug_wait_injection(int64_t wait_limit_ns, int skip_page) {
#ifdef XS_DEBUG_BOUNDS
    if (wait_limit_ns <= 0 || skip_page < -1) return XS_ESHAPE;
    const unsigned long long limit = static_cast<unsigned long long>(wait_limit_ns);
    if (cudaMemcpyToSymbol(attn::g_wait_limit_ns, &limit, sizeof(limit)) != cudaSuccess ||
        cudaMemcpyToSymbol(attn::g_skip_page, &skip_page, sizeof(skip_page)) != cudaSuccess) {
        cudaGetLastError();
        return XS_EDEVICE;
    }
    return XS_OK;
#else
    (void)wait_limit_ns;
    (void)skip_page;
    return XS_EUNSUPPORTED;
#endif
}

extern "C" int xs_paged_decode_partition_tokens(int B, int Hkv, int64_t total_context_tokens,
                                                int max_context_len, int num_sms) {
    if (B < 0 || Hkv <= 0 || max_context_len < 0 || num_sms <= 0) return XS_ESHAPE;
    if (B == 0) return 64;
    const double tokens = total_context_tokens > 0
                              ? static_cast<double>(total_context_tokens)
                              : static_cast<double>(B) * std::max(max_context_len, 1);
    // Cost model, in units of "one page per consumer warp": an item of P
    // tokens costs P/16/4 + kItemCost (q staging, the four-warp merge and the
    // partials it writes and the reduce reads back); items are taken by
    // 2 resident CTAs per SM, so the step takes about items / CTAs + 1 item
    // times (the last round is ragged).  Each sequence adds about half a
    // partition of ragged tail.  At
    // least 4 pages per item, so every consumer warp has a page.
    constexpr double kItemCost = 1.5;
    const double ctas = 2.0 * num_sms;
    int best = 64;
    double best_cost = 1e300;
    for (int P = 64; P <= 2048; P *= 2) {
        const double items = std::max((tokens / P + 0.5 * B) * Hkv, static_cast<double>(B) * Hkv);
        const double cost = (items / ctas + 1.0) * (P / 64.0 + kItemCost);
        if (cost <= best_cost * (1.0 + 1e-9)) {  // ties go to the larger partition
            best_cost = cost;
            best = P;
        }
    }
    return best;
}

extern "C" int xs_paged_decode_step_partition_tokens(int B, int Hq, int Hkv,
                                                     int64_t total_context_tokens,
                                                     int max_context_len, int num_sms) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_context_len < 0 || num_sms <= 0)
        return XS_ESHAPE;
    if (B == 0) return 64;
    const double tokens = total_context_tokens > 0
                              ? static_cast<double>(total_context_tokens)
                              : static_cast<double>(B) * std::max(max_context_len, 1);
    // The cost model of xs_paged_decode_partition_tokens, refitted to
    // one-launch step times: an item of P tokens costs P/64 + kItemCost
    // page-times (q staging, first-page latency, the four-warp merge); the
    // grid takes items / CTAs rounds plus kTailRounds of ragged end - or,
    // when every sequence has the same length, exactly ceil(items / CTAs)
    // rounds (a batch one item over a round takes a whole second round) -
    // and the split-K combine at the end of the longest sequence adds
    // kCombineCost per partition.  P runs over multiples of 64 so that a
    // batch can land just under a whole number of rounds.  Fitted to a sweep
    // of every candidate P on the 11 shapes of the persistent grid
    // (launches too large for one wave of thread-block clusters: log-uniform
    // mixes of 48-256 sequences, equal-length batches of 32-64 sequences, a
    // uniform-length batch, the long batch), launched back to back: mean
    // 0.6 % and at most 2.1 % slower than the best measured P.
    constexpr double kItemCost = 2.25;
    constexpr double kTailRounds = 0.5;
    constexpr double kCombineCost = 0.2;
    constexpr int kCandidates[] = {64,  128, 192, 256,  320,  384,  448,  512,
                                   576, 640, 768, 896, 1024, 1280, 1536, 2048};
    const double ctas = 2.0 * num_sms;
    const int longest = std::max(max_context_len, 1);
    const bool uniform = tokens >= 0.98 * static_cast<double>(B) * longest;
    int best = 64;
    double best_cost = 1e300;
    for (const int P : kCandidates) {
        const int np = (longest + P - 1) / P;
        double cost;
        if (uniform) {
            const double items = static_cast<double>(B) * Hkv * np;
            cost = std::ceil(items / ctas) * (P / 64.0 + kItemCost);
        } else {
            const double items =
                std::max((tokens / P + 0.5 * B) * Hkv, static_cast<double>(B) * Hkv);
            cost = (items / ctas + kTailRounds) * (P / 64.0 + kItemCost);
        }
        if (np > 1) cost += kCombineCost * np;
        if (cost <= best_cost * (1.0 + 1e-9)) {  // ties go to the larger partition
            best_cost = cost;
            best = P;
        }
    }
    return best;
}

extern "C" int xs_paged_decode_max_partitions(int max_blocks_per_seq, int block_size,
                                              int partition_tokens) {
    if (max_blocks_per_seq < 0 || block_size <= 0 || partition_tokens <= 0) return XS_ESHAPE;
    const int64_t cap = static_cast<int64_t>(max_blocks_per_seq) * block_size;
    return static_cast<int>(std::max<int64_t>(1, (cap + partition_tokens - 1) / partition_tokens));
}

extern "C" int xs_paged_decode_num_splits(int B, int Hkv, int max_context_len, int sm_count) {
    if (B < 0 || Hkv <= 0 || max_context_len < 0 || sm_count <= 0) return XS_ESHAPE;
    const int P = xs_paged_decode_partition_tokens(
        B, Hkv, static_cast<int64_t>(B) * max_context_len, max_context_len, sm_count);
    if (P < 0) return P;
    return std::max(1, (max_context_len + P - 1) / P);
}

extern "C" size_t xs_paged_decode_workspace_bytes(int B, int Hq, int D, int max_partitions) {
    if (B <= 0 || Hq <= 0 || D <= 0 || max_partitions <= 0) return 0;
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t n = static_cast<size_t>(B) * Hq * max_partitions;
    return up(n * D * 4) + 2 * up(n * 4);
}

static int check_attn_args(const void *out, const float *po, const float *pm, const float *pl,
                           const void *q, const void *kc, const void *vc, const int32_t *bt,
                           int max_blocks, const int32_t *lens, int B, int Hq, int Hkv, int D,
                           int bs, int64_t num_blocks, int P, int max_parts, int dtype,
                           bool prefill = false) {
    if (!out || !q || !kc || !vc || !bt || (!lens && !prefill)) return XS_ENULL;
    if (!elem_bytes(dtype)) return XS_EDTYPE;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || max_blocks < 0 || num_blocks < 0) return XS_ESHAPE;
    if (Hq % Hkv != 0) return XS_ESHAPE;
    const int G = Hq / Hkv;
    if (bs != attn::kBlock || (D != 64 && D != 128) || (G != 1 && G != 2 && G != 4 && G != 8))
        return XS_EUNSUPPORTED;
    if (B > attn::kMaxBatch) return XS_EUNSUPPORTED;
    if (P < attn::kBlock || P % attn::kBlock != 0) return XS_ESHAPE;
    if (max_parts < xs_paged_decode_max_partitions(max_blocks, bs, P)) return XS_EWORKSPACE;
    if (max_parts > 1 && (!po || !pm || !pl)) return XS_EWORKSPACE;
    if (!aligned16(out) || !aligned16(q) || !aligned16(kc) || !aligned16(vc)) return XS_EALIGN;
    if (max_parts > 1 && (!aligned16(po) || !aligned16(pm) || !aligned16(pl))) return XS_EALIGN;
    return XS_OK;
}

static int launch_attn(void *out, float *part_o, float *part_m, float *part_l, const void *q,
                       const void *k_cache, const void *v_cache, const int32_t *block_tables,
                       int max_blocks_per_seq, const int32_t *context_lens, int B, int Hq,
                       int Hkv, int D, int block_size, int64_t num_blocks, float scale,
                       const void *sinks, int window, int partition_tokens, int max_partitions,
                       int dtype, int *err_flag, int *work_counters, cudaStream_t stream,
                       int prefill_start = -1, const void *k_new = nullptr,
                       const void *v_new = nullptr, int *combine = nullptr, int early = 0,
                       bool allow_cluster = true) {
    if (window < 0) return XS_ESHAPE;
    const bool prefill = prefill_start >= 0;
    int st = check_attn_args(out, part_o, part_m, part_l, q, k_cache, v_cache, block_tables,
                             max_blocks_per_seq, context_lens, B, Hq, Hkv, D, block_size,
                             num_blocks, partition_tokens, max_partitions, dtype, prefill);
    if (st != XS_OK) return st;
    if (B == 0) return XS_OK;
    attn::DeviceInfo dev;
    if ((st = attn::device_info(&dev)) != XS_OK) return st;
    // A step small enough for one wave of clusters runs as clusters.
    attn::KernelFn fn = nullptr;
    int smem = 0, cluster = 0, cluster_P = 0;
    if (combine && !prefill && allow_cluster)
        cluster = attn::cluster_plan(B, Hkv, D, Hq / Hkv, max_blocks_per_seq, window, dtype,
                                     &cluster_P, &fn, &smem);
    int per_sm = 1;
    if (!cluster) {
        int smem0 = 0;
        // At most one work item per SM: one CTA per SM with the deep ring.
        const bool deep = static_cast<int64_t>(B) * Hkv * max_partitions <= dev.sms;
        fn = attn::pick_kernel(dtype, D, Hq / Hkv, deep, &smem0);
        if (!fn) return XS_EUNSUPPORTED;
        smem = smem0 + attn::table_bytes(B) + 1024;  // = Cfg<...>::smem_bytes(B)
        if (smem + 1024 > dev.max_smem_optin) return XS_EUNSUPPORTED;  // room for static smem
        if ((st = attn::occupancy(fn, smem, &per_sm)) != XS_OK) return st;
    }
    // The in-launch combine stages partial rows in shared memory: as many
    // partials (G rows of D fp32 each) as fit beside the CTAs that are
    // resident anyway, at least one, at most 32 or 32 KB.
    int stage_bytes = 0, stage_parts = 0;
    if (combine && !cluster) {
        int st_smem = 0;
        if ((st = attn::static_smem(fn, &st_smem)) != XS_OK) return st;
        const int part_bytes = Hq / Hkv * D * 4;
        const int avail = dev.smem_per_sm / per_sm - dev.reserved_per_block - st_smem - smem - 32;
        stage_parts = std::max(1, std::min({avail / part_bytes, 32, 32768 / part_bytes,
                                            std::max(max_partitions, 1)}));
        stage_bytes = stage_parts * part_bytes + 32;  // + its header and alignment
        smem += stage_bytes;
        if (smem + 1024 > dev.max_smem_optin) return XS_EUNSUPPORTED;
        if ((st = attn::occupancy(fn, smem, &per_sm)) != XS_OK) return st;
    }
    const int64_t max_items = static_cast<int64_t>(B) * Hkv * max_partitions;
    const int64_t resident = static_cast<int64_t>(dev.sms) * per_sm;
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min(max_items, resident)));
    // bf16 pages travel as TMA tensor copies: the pools as 4-D (64 elements,
    // 16 rows, D/64 halves, num_blocks * Hkv pages) with strides (2 D, 128,
    // 32 D) bytes, one box (64, 16, D/64, 1) per page.  fp32 uses 1-D copies.
    CUtensorMap tmk, tmv;
    memset(&tmk, 0, sizeof(tmk));
    memset(&tmv, 0, sizeof(tmv));
    if (dtype == XS_BF16) {
        if (num_blocks * Hkv > 0x7fffffff) return XS_EUNSUPPORTED;  // 32-bit page coordinate
        if ((st = attn::pool_maps(k_cache, v_cache, num_blocks, Hkv, D, &tmk, &tmv)) != XS_OK)
            return st;
    }
    attn::Params p;
    p.out = out;
    p.part_o = part_o;
    p.part_m = part_m;
    p.part_l = part_l;
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.max_blocks = max_blocks_per_seq;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.P = partition_tokens;
    p.max_parts = max_partitions;
    p.num_blocks = num_blocks;
    p.qscale = scale * attn::kLog2e;
    p.sinks = sinks;
    p.window = window;
    p.prefill_start = prefill_start;
    p.table_stride = prefill ? 0 : max_blocks_per_seq;
    p.err_flag = err_flag;
    p.work = work_counters;
    p.k_new = k_new;
    p.v_new = v_new;
    p.combine = combine;
    p.early = early;
    p.stage_bytes = stage_bytes;
    p.stage_parts = stage_parts;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(attn::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cluster) {
        // One cluster of `cluster` CTAs per (sequence, KV head).
        p.P = cluster_P;
        p.max_parts = cluster;
        cfg.gridDim = dim3(cluster, B * Hkv);
        cfg.blockDim = dim3(attn::kCluThreads);
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = cluster;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    if (cudaLaunchKernelEx(&cfg, fn, tmk, tmv, p) != cudaSuccess) {
        cudaGetLastError();
        return XS_ELAUNCH;
    }
    return launch_status();
}

extern "C" int xs_paged_decode_attn(void *out, float *part_o, float *part_m, float *part_l,
                                    const void *q, const void *k_cache, const void *v_cache,
                                    const int32_t *block_tables, int max_blocks_per_seq,
                                    const int32_t *context_lens, int B, int Hq, int Hkv, int D,
                                    int block_size, int64_t num_blocks, float scale,
                                    int partition_tokens, int max_partitions, int dtype,
                                    int *err_flag, int *work_counters, cudaStream_t stream) {
    return launch_attn(out, part_o, part_m, part_l, q, k_cache, v_cache, block_tables,
                       max_blocks_per_seq, context_lens, B, Hq, Hkv, D, block_size, num_blocks,
                       scale, nullptr, 0, partition_tokens, max_partitions, dtype, err_flag,
                       work_counters, stream);
}

extern "C" int xs_paged_decode_attn_sinks(void *out, float *part_o, float *part_m, float *part_l,
                                          const void *q, const void *k_cache, const void *v_cache,
                                          const int32_t *block_tables, int max_blocks_per_seq,
                                          const int32_t *context_lens, const void *sinks,
                                          int window, int B, int Hq, int Hkv, int D,
                                          int block_size, int64_t num_blocks, float scale,
                                          int partition_tokens, int max_partitions, int dtype,
                                          int *err_flag, int *work_counters,
                                          cudaStream_t stream) {
    return launch_attn(out, part_o, part_m, part_l, q, k_cache, v_cache, block_tables,
                       max_blocks_per_seq, context_lens, B, Hq, Hkv, D, block_size, num_blocks,
                       scale, sinks, window, partition_tokens, max_partitions, dtype, err_flag,
                       work_counters, stream);
}

static int launch_reduce(void *out, const float *part_o, const float *part_m,
                         const float *part_l, const int32_t *context_lens, const void *sinks,
                         int window, int B, int Hq, int D, int partition_tokens,
                         int max_partitions, int dtype, cudaStream_t stream,
                         int prefill_start = -1) {
    if (!out || (!context_lens && prefill_start < 0)) return XS_ENULL;
    if (window < 0) return XS_ESHAPE;
    if (!elem_bytes(dtype)) return XS_EDTYPE;
    if (B < 0 || Hq <= 0 || D <= 0 || D > 1024 || partition_tokens <= 0 || max_partitions <= 0)
        return XS_ESHAPE;
    if (B == 0 || max_partitions == 1) return XS_OK;
    if (!part_o || !part_m || !part_l) return XS_EWORKSPACE;
    const int64_t blocks = static_cast<int64_t>(B) * Hq;
    if (blocks > 0x7fffffff) return XS_ESHAPE;
    const int threads = (D + 31) / 32 * 32;
    if (dtype == XS_BF16)
        attn::paged_decode_reduce_kernel<__nv_bfloat16><<<static_cast<int>(blocks), threads, 0,
                                                          stream>>>(
            static_cast<__nv_bfloat16 *>(out), part_o, part_m, part_l, context_lens, Hq, D,
            partition_tokens, max_partitions, static_cast<const __nv_bfloat16 *>(sinks), window,
            prefill_start);
    else
        attn::paged_decode_reduce_kernel<float><<<static_cast<int>(blocks), threads, 0, stream>>>(
            static_cast<float *>(out), part_o, part_m, part_l, context_lens, Hq, D,
            partition_tokens, max_partitions, static_cast<const float *>(sinks), window,
            prefill_start);
    return launch_status();
}

extern "C" int xs_paged_decode_reduce(void *out, const float *part_o, const float *part_m,
                                      const float *part_l, const int32_t *context_lens, int B,
                                      int Hq, int D, int partition_tokens, int max_partitions,
                                      int dtype, cudaStream_t stream) {
    return launch_reduce(out, part_o, part_m, part_l, context_lens, nullptr, 0, B, Hq, D,
                         partition_tokens, max_partitions, dtype, stream);
}

// The partition length for a split given as a count (num_splits partitions
// cover the table's reach), or XS_ESHAPE.
static int splits_partition(int max_blocks_per_seq, int block_size, int num_splits) {
    if (num_splits <= 0 || max_blocks_per_seq < 0 || block_size <= 0) return XS_ESHAPE;
    const int64_t cap = static_cast<int64_t>(max_blocks_per_seq) * block_size;
    const int64_t per = (cap + num_splits - 1) / num_splits;
    const int64_t P = std::max<int64_t>(attn::kBlock, (per + attn::kBlock - 1) / attn::kBlock *
                                                          attn::kBlock);
    return P > 0x7fffffff ? XS_ESHAPE : static_cast<int>(P);
}

extern "C" int xs_paged_decode_attn_splits(void *out, float *part_o, float *part_m,
                                           float *part_l, const void *q, const void *k_cache,
                                           const void *v_cache, const int32_t *block_tables,
                                           int max_blocks_per_seq, const int32_t *context_lens,
                                           int B, int Hq, int Hkv, int D, int block_size,
                                           int64_t num_blocks, float scale, int num_splits,
                                           int dtype, int *err_flag, cudaStream_t stream) {
    const int P = splits_partition(max_blocks_per_seq, block_size, num_splits);
    if (P < 0) return P;
    return xs_paged_decode_attn(out, part_o, part_m, part_l, q, k_cache, v_cache, block_tables,
                                max_blocks_per_seq, context_lens, B, Hq, Hkv, D, block_size,
                                num_blocks, scale, P, num_splits, dtype, err_flag, nullptr, stream);
}

extern "C" int xs_paged_decode_reduce_splits(void *out, const float *part_o, const float *part_m,
                                             const float *part_l, const int32_t *context_lens,
                                             int max_blocks_per_seq, int B, int Hq, int D,
                                             int block_size, int num_splits, int dtype,
                                             cudaStream_t stream) {
    const int P = splits_partition(max_blocks_per_seq, block_size, num_splits);
    if (P < 0) return P;
    if (num_splits == 1) return XS_OK;  // every sequence was one partition
    return xs_paged_decode_reduce(out, part_o, part_m, part_l, context_lens, B, Hq, D, P,
                                  num_splits, dtype, stream);
}

extern "C" int xs_paged_decode_reduce_sinks(void *out, const float *part_o, const float *part_m,
                                            const float *part_l, const int32_t *context_lens,
                                            const void *sinks, int window, int B, int Hq, int D,
                                            int partition_tokens, int max_partitions, int dtype,
                                            cudaStream_t stream) {
    return launch_reduce(out, part_o, part_m, part_l, context_lens, sinks, window, B, Hq, D,
                         partition_tokens, max_partitions, dtype, stream);
}

extern "C" int xs_paged_decode(void *out, float *part_o, float *part_m, float *part_l,
                               const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *block_tables, int max_blocks_per_seq,
                               const int32_t *context_lens, int B, int Hq, int Hkv, int D,
                               int block_size, int64_t num_blocks, float scale,
                               int partition_tokens, int max_partitions, int dtype, int *err_flag,
                               int *work_counters, cudaStream_t stream) {
    int st = xs_paged_decode_attn(out, part_o, part_m, part_l, q, k_cache, v_cache, block_tables,
                                  max_blocks_per_seq, context_lens, B, Hq, Hkv, D, block_size,
                                  num_blocks, scale, partition_tokens, max_partitions, dtype,
                                  err_flag, work_counters, stream);
    if (st != XS_OK || max_partitions <= 1) return st;
    return xs_paged_decode_reduce(out, part_o, part_m, part_l, context_lens, B, Hq, D,
                                  partition_tokens, max_partitions, dtype, stream);
}

extern "C" int xs_paged_decode_sinks(void *out, float *part_o, float *part_m, float *part_l,
                                     const void *q, const void *k_cache, const void *v_cache,
                                     const int32_t *block_tables, int max_blocks_per_seq,
                                     const int32_t *context_lens, const void *sinks, int window,
                                     int B, int Hq, int Hkv, int D, int block_size,
                                     int64_t num_blocks, float scale, int partition_tokens,
                                     int max_partitions, int dtype, int *err_flag,
                                     int *work_counters, cudaStream_t stream) {
    int st = xs_paged_decode_attn_sinks(out, part_o, part_m, part_l, q, k_cache, v_cache,
                                        block_tables, max_blocks_per_seq, context_lens, sinks,
                                        window, B, Hq, Hkv, D, block_size, num_blocks, scale,
                                        partition_tokens, max_partitions, dtype, err_flag,
                                        work_counters, stream);
    if (st != XS_OK || max_partitions <= 1) return st;
    return xs_paged_decode_reduce_sinks(out, part_o, part_m, part_l, context_lens, sinks, window,
                                        B, Hq, D, partition_tokens, max_partitions, dtype, stream);
}

// ---------------------------------------------------------------- fused decode step
//
// Append + attention + split-K combine in one launch; see the header for the
// contract.  counters = [item counter, finished-CTA counter, B * Hkv combine
// counts], all zero between launches.

extern "C" int xs_paged_decode_step_ex(void *out, const void *q, const void *k_new,
                                       const void *v_new, void *k_cache, void *v_cache,
                                       const int32_t *block_tables, int max_blocks_per_seq,
                                       const int32_t *context_lens, const void *sinks, int window,
                                       int B, int Hq, int Hkv, int D, int block_size,
                                       int64_t num_blocks, float scale, int partition_tokens,
                                       int max_partitions, float *part_o, float *part_m,
                                       float *part_l, int *counters, int flags, int dtype,
                                       int *err_flag, cudaStream_t stream) {
    if (flags & ~(XS_STEP_EARLY_READS | XS_STEP_PERSISTENT)) return XS_EUNSUPPORTED;
    if (!k_new != !v_new) return XS_ENULL;
    if (!counters) return XS_EWORKSPACE;
    if (k_new && (!aligned16(k_new) || !aligned16(v_new))) return XS_EALIGN;
    return launch_attn(out, part_o, part_m, part_l, q, k_cache, v_cache, block_tables,
                       max_blocks_per_seq, context_lens, B, Hq, Hkv, D, block_size, num_blocks,
                       scale, sinks, window, partition_tokens, max_partitions, dtype, err_flag,
                       counters, stream, -1, k_new, v_new, counters + 2,
                       (flags & XS_STEP_EARLY_READS) ? 1 : 0, !(flags & XS_STEP_PERSISTENT));
}

extern "C" int xs_paged_decode_step(void *out, const void *q, const void *k_new,
                                    const void *v_new, void *k_cache, void *v_cache,
                                    const int32_t *block_tables, int max_blocks_per_seq,
                                    const int32_t *context_lens, const void *sinks, int window,
                                    int B, int Hq, int Hkv, int D, int block_size,
                                    int64_t num_blocks, float scale, int partition_tokens,
                                    int max_partitions, float *part_o, float *part_m,
                                    float *part_l, int *counters, int dtype, int *err_flag,
                                    cudaStream_t stream) {
    return xs_paged_decode_step_ex(out, q, k_new, v_new, k_cache, v_cache, block_tables,
                                   max_blocks_per_seq, context_lens, sinks, window, B, Hq, Hkv, D,
                                   block_size, num_blocks, scale, partition_tokens,
                                   max_partitions, part_o, part_m, part_l, counters, 0, dtype,
                                   err_flag, stream);
}

extern "C" int xs_paged_decode_step_cluster_size(int B, int Hq, int Hkv, int D,
                                                 int max_blocks_per_seq, int window, int dtype) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_blocks_per_seq < 0 || window < 0)
        return XS_ESHAPE;
    if (B == 0) return 0;
    int P = 0, smem = 0;
    attn::KernelFn fn = nullptr;
    return attn::cluster_plan(B, Hkv, D, Hq / Hkv, max_blocks_per_seq, window, dtype, &P, &fn,
                              &smem);
}

extern "C" int64_t xs_paged_decode_step_counters(int B, int Hkv) {
    if (B < 0 || Hkv <= 0) return XS_ESHAPE;
    return 2 + static_cast<int64_t>(B) * Hkv;
}

// ---------------------------------------------------------------- chunked prefill
//
// Causal attention of a T-token chunk at positions start_pos .. over one
// sequence's paged cache, on the decode kernel: query token i is treated as
// a sequence of start_pos + i + 1 tokens that shares the chunk's block list.

extern "C" int xs_paged_prefill_attn(void *out, float *part_o, float *part_m, float *part_l,
                                     const void *q, const void *k_cache, const void *v_cache,
                                     const int32_t *block_ids, int n_ids, int T, int start_pos,
                                     int Hq, int Hkv, int D, int block_size, int64_t num_blocks,
                                     float scale, int partition_tokens, int max_partitions,
                                     int dtype, int *err_flag, int *work_counters,
                                     cudaStream_t stream) {
    if (T < 0 || start_pos < 0 || n_ids < 0) return XS_ESHAPE;
    if (static_cast<int64_t>(start_pos) + T > static_cast<int64_t>(n_ids) * block_size)
        return XS_ESHAPE;  // the block list does not cover the chunk
    return launch_attn(out, part_o, part_m, part_l, q, k_cache, v_cache, block_ids, n_ids,
                       nullptr, T, Hq, Hkv, D, block_size, num_blocks, scale, nullptr, 0,
                       partition_tokens, max_partitions, dtype, err_flag, work_counters, stream,
                       start_pos);
}

extern "C" int xs_paged_prefill_reduce(void *out, const float *part_o, const float *part_m,
                                       const float *part_l, int T, int start_pos, int Hq, int D,
                                       int partition_tokens, int max_partitions, int dtype,
                                       cudaStream_t stream) {
    if (start_pos < 0) return XS_ESHAPE;
    return launch_reduce(out, part_o, part_m, part_l, nullptr, nullptr, 0, T, Hq, D,
                         partition_tokens, max_partitions, dtype, stream, start_pos);
}

extern "C" int xs_paged_prefill(void *out, float *part_o, float *part_m, float *part_l,
                                const void *q, const void *k_cache, const void *v_cache,
                                const int32_t *block_ids, int n_ids, int T, int start_pos, int Hq,
                                int Hkv, int D, int block_size, int64_t num_blocks, float scale,
                                int partition_tokens, int max_partitions, int dtype,
                                int *err_flag, int *work_counters, cudaStream_t stream) {
    int st = xs_paged_prefill_attn(out, part_o, part_m, part_l, q, k_cache, v_cache, block_ids,
                                   n_ids, T, start_pos, Hq, Hkv, D, block_size, num_blocks, scale,
                                   partition_tokens, max_partitions, dtype, err_flag,
                                   work_counters, stream);
    if (st != XS_OK || max_partitions <= 1) return st;
    return xs_paged_prefill_reduce(out, part_o, part_m, part_l, T, start_pos, Hq, D,
                                   partition_tokens, max_partitions, dtype, stream);
}

// ---------------------------------------------------------------- no-allocation variant
//
// Split-K partials for callers that cannot allocate device memory: a fixed
// array of XS_NOALLOC_SCRATCH_BYTES at file scope, reserved on every device
// that loads this library.  Host code must not use the symbol itself as a
// pointer (in host code it names a host-side stand-in), so every call looks
// up the array's device address for the current device and context with
// cudaGetSymbolAddress.  Nothing is cached: a cached address could outlive
// its context (cudaDeviceReset, or another context made current).

static __device__ __align__(256) unsigned char g_noalloc_scratch[XS_NOALLOC_SCRATCH_BYTES];

static int noalloc_scratch(unsigned char **out) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
        cudaGetLastError();  // do not leave the failure for an unrelated later check
        return XS_EDEVICE;
    }
    *out = static_cast<unsigned char *>(p);
    return XS_OK;
}

extern "C" int xs_paged_decode_noalloc(void *out, const void *q, const void *k_cache,
                                       const void *v_cache, const int32_t *block_tables,
                                       int max_blocks_per_seq, const int32_t *context_lens,
                                       int B, int Hq, int Hkv, int D, int block_size,
                                       int64_t num_blocks, float scale, int partition_tokens,
                                       int dtype, int *err_flag, cudaStream_t stream) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || max_blocks_per_seq < 0 || block_size <= 0)
        return XS_ESHAPE;
    if (partition_tokens <= 0) {
        attn::DeviceInfo dev;
        const int st = attn::device_info(&dev);
        if (st != XS_OK) return st;
        partition_tokens = xs_paged_decode_partition_tokens(
            B, Hkv, static_cast<int64_t>(B) * max_blocks_per_seq * block_size,
            max_blocks_per_seq * block_size, dev.sms);
        if (partition_tokens < 0) return partition_tokens;
    }
    const int max_parts =
        xs_paged_decode_max_partitions(max_blocks_per_seq, block_size, partition_tokens);
    if (max_parts < 0) return max_parts;
    const bool split = max_parts > 1 && B > 0;
    size_t need = 0;
    if (split) {
        need = xs_paged_decode_workspace_bytes(B, Hq, D, max_parts);
        if (need == 0) return XS_ESHAPE;
        if (need > XS_NOALLOC_SCRATCH_BYTES) return XS_ESCRATCH;
    }
    // Validate everything else before touching the device (the partial
    // pointers stand in for the array's aligned address).
    float *const stand_in = reinterpret_cast<float *>(256);
    int st = check_attn_args(out, stand_in, stand_in, stand_in, q, k_cache, v_cache, block_tables,
                             max_blocks_per_seq, context_lens, B, Hq, Hkv, D, block_size,
                             num_blocks, partition_tokens, max_parts, dtype);
    if (st != XS_OK) return st;
    // The array's address on the current device, looked up on every call
    // (the first call on a device may load the library's device code).
    unsigned char *base = nullptr;
    if ((st = noalloc_scratch(&base)) != XS_OK) return st;
    float *po = nullptr, *pm = nullptr, *pl = nullptr;
    if (split) {
        const size_t n = static_cast<size_t>(B) * Hq * max_parts;
        const size_t o_bytes = (n * D * 4 + 255) / 256 * 256;
        const size_t ml_bytes = (n * 4 + 255) / 256 * 256;
        po = reinterpret_cast<float *>(base);
        pm = reinterpret_cast<float *>(base + o_bytes);
        pl = reinterpret_cast<float *>(base + o_bytes + ml_bytes);
    }
    return xs_paged_decode(out, po, pm, pl, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                           context_lens, B, Hq, Hkv, D, block_size, num_blocks, scale,
                           partition_tokens, max_parts, dtype, err_flag, nullptr, stream);
}
