// Forward exact attention for short key sequences (at most 256 keys) and
// head dims up to 64: the shapes of the flash-attn timing issue ("2.6.3 is
// faster than 2.7.0 for flash-attn v2 CUDA fwd/bwd": embed 256 over 16 heads,
// so head dim 16, sequences of 50 to 300), where each (batch, head) is a
// small problem and there are thousands of them.
//
// What is computed is the forward of "Why FlashAttention is fast" (section
// 2 item 4: S = scale Q K^T, softmax, times V), with S kept on chip (section
// 3.2). With every key of a head in one tile, the softmax needs no running
// rescale: the row max is taken over the whole tile before any exponential,
// which is section 3.3's online softmax with a single block.
//
// A work item is one 128-row query tile of one (batch, head) against all of
// its keys (or, grouped, one 32-row query block of four heads: below).
// Persistent CTAs (one per SM) deal their items to two or three TMEM slots,
// so several items are in flight per SM and the latency chain of each
// (loads, QK^T, softmax, PV, store) overlaps the others':
//   warp 0        TMA producer: Q tile, K and V of the item into a ring of
//                 shared-memory stages (grouped: the query block of the
//                 item, and the group's K and V once per group).
//   warp 1        TMEM owner; issues every QK^T MMA (one thread): S = Q K^T
//                 into the item's slot.
//   warp 2        grouped items: copies each query block onto its
//                 block-diagonal tile; else idle.
//   warp 3        issues every P V MMA (one thread).
//   warps 4..     one softmax warpgroup per slot (the kernel is compiled
//                 for 2 and 3 slots); warpgroup g owns slot g, and thread i
//                 of warp w owns row 32 (w % 4) + i of its tile.
// TMEM slot g spans columns [g W, g W + W): S in [0, N) (N = sk rounded up
// to 32), overwritten by P two 16-bit keys per column in [0, N/2), and the
// O accumulator in [o_off, o_off + d) (64 columns when grouped) once S has
// been read.
// The softmax reads S once, 64 columns at a time, with the lazy reference
// max of the general forward: the first 64 columns set it, and a later pair
// of chunks whose max exceeds it by more than 8 (log2 units) moves it and
// rescales the P already stored (rare). So no thread holds a whole score
// row and each chunk costs one TMEM round trip.
//
// Grouped items (head dim 16, heads a multiple of 4). At head dim 16 a
// query or key row of one head is 32 bytes, with the other heads' rows
// between them, and loading a head by itself moves 32-byte pieces: a TMA box
// (or cp.async) of such rows ran at about 7 bytes per cycle per SM, which
// is what set the pace of whole calls. So four consecutive heads are loaded
// as one: their rows are 128 contiguous bytes (the [b, s, h / 4, 64] view
// of the same memory), one TMA box per tile. A work item is one 32-row
// query block of such a group of four heads, 128 rows in all, and the
// group's K and V tiles (N keys by 4 x 16) are loaded once and serve every
// query block of the group. The four heads must not see each other's keys,
// and one MMA multiplies one A tile by one B tile, so warp 2 copies the
// query block onto the block diagonal of a zeroed 128 x 64 tile: rows
// [32p, 32p + 32) hold head p's 16 query columns at columns [16p, 16p + 16)
// and zeros elsewhere. Four MMAs accumulate S, the p-th over the 16 columns
// of head p in both the diagonal tile and the group's K tile; every other
// head's columns are zero in row block p, so each row gets the scores
// against its own head's keys. P V runs once with N = 64 over the group's V
// tile (the four heads side by side), and row block p keeps O columns
// [16p, 16p + 16). A K that holds an infinity or a NaN therefore also turns
// the other heads of its group to NaN (zero times infinity); the inputs are
// taken to be finite.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace exattn {
namespace {

// Bit 13 of a kind::f16 instruction descriptor: negate the A operand.
constexpr uint32_t kIdescNegateA = 1u << 13;

constexpr int SH_WG = SHORT_MAX_SLOTS;          // most softmax warpgroups
constexpr int SH_BAR_BYTES = 1024;             // barriers and flags, before the tiles

// barriers: full[stages] | empty[stages] | s_full[slots] | p_full[slots] |
//           o_full[slots] | free[slots] | done[2] | (grouped items:) diagonal
//           tile full[stages] | group K/V full[kv stages] | empty[kv stages]
constexpr int SH_MAX_KV_STAGES = 3;
constexpr int BAR_FULL = 0;
constexpr int BAR_EMPTY = BAR_FULL + SHORT_MAX_STAGES;
constexpr int BAR_SF = BAR_EMPTY + SHORT_MAX_STAGES;
constexpr int BAR_PF = BAR_SF + SH_WG;
constexpr int BAR_OF = BAR_PF + SH_WG;
constexpr int BAR_FREE = BAR_OF + SH_WG;
constexpr int BAR_DONE = BAR_FREE + SH_WG;
constexpr int BAR_DONE2 = BAR_DONE + 1;
constexpr int BAR_DF = BAR_DONE2 + 1;
constexpr int BAR_KVF = BAR_DF + SHORT_MAX_STAGES;
constexpr int BAR_KVE = BAR_KVF + SH_MAX_KV_STAGES;
constexpr int NUM_BARS = BAR_KVE + SH_MAX_KV_STAGES;
constexpr int OFF_MISC = NUM_BARS * 8;
static_assert(OFF_MISC + 16 <= SH_BAR_BYTES, "barrier area");

template <int D>
struct ShortGeom {
    static constexpr int ROW_BYTES = D * 2;  // one swizzle panel: 32, 64 or 128 bytes
    static constexpr uint32_t LAYOUT =
        ROW_BYTES == 128 ? kLayoutSw128 : (ROW_BYTES == 64 ? kLayoutSw64 : kLayoutSw32);
    static constexpr uint32_t SBO = 8 * ROW_BYTES;
    static constexpr int Q_BYTES = SHORT_BM * ROW_BYTES;
    static_assert(D == 16 || D == 32 || D == 64, "head dim");
};

template <bool BF16>
__device__ __forceinline__ uint32_t pack2s(float lo, float hi) {
    if constexpr (BF16)
        return cvt_pack_bf16(lo, hi);
    else
        return cvt_pack_f16(lo, hi);
}

struct Item {
    int tile, head, batch;
};

__device__ __forceinline__ Item item_of(int it, int ntile, int h) {
    Item x;
    x.tile = it % ntile;
    const int r = it / ntile;
    x.head = r % h;
    x.batch = r / h;
    return x;
}

// Grouped items: a CTA takes the (batch, group of four heads) pairs c,
// c + grid, c + 2 grid, ... and runs every 32-row query block of each pair
// in turn, so its n-th item is block n % nblk of its (n / nblk)-th pair.
struct GroupItem {
    int batch, group, blk, k;  // k: the pair's index among this CTA's pairs
};

__device__ __forceinline__ GroupItem group_item(int n, int nblk, int hg) {
    GroupItem x;
    x.k = n / nblk;
    x.blk = n - x.k * nblk;
    const int pair = static_cast<int>(blockIdx.x) + x.k * static_cast<int>(gridDim.x);
    x.batch = pair / hg;
    x.group = pair - x.batch * hg;
    return x;
}

// Folds one 32-column chunk of scores into four running maxima. MASK: only
// the first `valid` columns are keys.
template <bool MASK>
__device__ __forceinline__ void chunk_max(const uint32_t (&r)[32], int valid, float (&mx)[4]) {
    const float *s = reinterpret_cast<const float *>(r);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        const float x0 = (!MASK || 2 * e < valid) ? s[2 * e] : -INFINITY;
        const float x1 = (!MASK || 2 * e + 1 < valid) ? s[2 * e + 1] : -INFINITY;
        mx[e & 3] = max3f(mx[e & 3], x0, x1);
    }
}

// P = 2^(s c - m) for one 32-column chunk, added into the packed row sums
// and stored as 16 columns of 16-bit pairs at taddr (two stores of 8).
// MASK: columns from `valid` on are not keys and get exactly 0.
template <bool MASK, bool BF16>
__device__ __forceinline__ void chunk_exp(const uint32_t (&r)[32], int valid, uint64_t c2,
                                          uint64_t nm2, uint64_t (&acc2)[2], uint32_t taddr) {
    const float *s = reinterpret_cast<const float *>(r);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        uint32_t pk[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int k0 = 16 * half + 2 * e;
            float x0, x1;
            f2_split(f2_fma(f2_make(s[k0], s[k0 + 1]), c2, nm2), x0, x1);
            if (MASK) {
                x0 = k0 < valid ? x0 : -INFINITY;
                x1 = k0 + 1 < valid ? x1 : -INFINITY;
            }
            const float p0 = fast_exp2(x0);
            const float p1 = fast_exp2(x1);
            acc2[e & 1] = f2_add(acc2[e & 1], f2_make(p0, p1));
            pk[e] = pack2s<BF16>(p0, p1);
        }
        tmem_st8(taddr + 8 * half, pk);
    }
}

template <bool BF16>
__device__ __forceinline__ float2 unpack2s(uint32_t w) {
    if constexpr (BF16)
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w));
    else
        return __half22float2(*reinterpret_cast<const __half2 *>(&w));
}

// The reference max moved up: the 16-bit P already stored in columns
// [0, cols) is multiplied by alpha (1 for rows that did not move), 16
// columns at a time. Warp-wide. (A rounded P rounded again after the
// scaling: the extra rounding, at most half an ulp of a value below 2^-8
// of the row's new largest P, is far inside the tolerance, and the event
// needs a pair of chunks whose max exceeds every earlier one by 2^8.)
template <bool BF16>
__device__ __forceinline__ void rescale_p(uint32_t tS, int cols, float alpha) {
    tmem_wait_st();  // the P being rescaled was stored by this thread
    for (int c0 = 0; c0 < cols; c0 += 16) {
        uint32_t w[16];
        tmem_ld16(tS + c0, w);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const float2 f = unpack2s<BF16>(w[e]);
            w[e] = pack2s<BF16>(f.x * alpha, f.y * alpha);
        }
        tmem_st16(tS + c0, w);
    }
}

// Plain items, run by lane 0 of warp 0: each item's Q tile, K and V (three
// TMA boxes) into one stage, in that order.
template <int D>
__device__ __forceinline__ void short_producer(const CUtensorMap *tq, const CUtensorMap *tk,
                                               const CUtensorMap *tv, uint32_t sbase,
                                               uint32_t tiles, int items, int ntile,
                                               const ShortArgs &a, const WaitGuard &g) {
    using G = ShortGeom<D>;
    auto bar = [&](int i) { return sbase + 8u * i; };
    const uint32_t bytes = G::Q_BYTES + 2u * a.kv_bytes;
    int n = 0;
    for (int it = blockIdx.x; it < items; it += gridDim.x, ++n) {
        const Item x = item_of(it, ntile, a.h);
        const int st = n % a.nstage;
        if (!mbar_wait(bar(BAR_EMPTY + st), ((n / a.nstage) & 1) ^ 1, g, 20)) break;
        mbar_arrive_expect_tx(bar(BAR_FULL + st), bytes);
        const uint32_t dst = tiles + st * a.stage_bytes;
        tma_load_4d(dst, tq, bar(BAR_FULL + st), 0, x.head, x.tile * SHORT_BM, x.batch);
        tma_load_4d(dst + a.q_bytes, tk, bar(BAR_FULL + st), 0, x.head, 0, x.batch);
        tma_load_4d(dst + a.q_bytes + a.kv_bytes, tv, bar(BAR_FULL + st), 0, x.head, 0, x.batch);
    }
    // Never leave the CTA with a copy still landing in shared memory.
    WaitGuard drain = g;
    uint32_t no_abort = 0;
    drain.abort = &no_abort;
    for (int m = (n > a.nstage ? n - a.nstage : 0); m < n; ++m)
        mbar_wait(bar(BAR_FULL + m % a.nstage), (m / a.nstage) & 1, drain, 21);
}

// Grouped items, run by lane 0 of warp 0: per pair, the group's K and V
// tiles (n_keys rows of 128 bytes each) into a ring of kv stages; per item,
// its 32-row query block of the group (128-byte rows) into the stage's
// staging area. The next pair's K/V is requested right after the current
// pair's first query block, once a kv stage has come free (with three kv
// stages, the one the pair before last used: long done).
// Stage layout (grouped): staging block (32 x 128 bytes), then the
// block-diagonal query tile (128 x 128 bytes); the kv ring follows the
// stages: K tile, then V tile, per kv stage.
__device__ __forceinline__ void group_producer(const CUtensorMap *tq, const CUtensorMap *tk,
                                               const CUtensorMap *tv, uint32_t sbase,
                                               uint32_t tiles, int n_items, int hg,
                                               const ShortArgs &a, const WaitGuard &g) {
    auto bar = [&](int i) { return sbase + 8u * i; };
    const uint32_t kv_base = tiles + a.nstage * a.stage_bytes;
    const int npairs = n_items / a.nblk;
    int kv_n = 0;  // pairs whose K/V have been requested
    auto load_kv = [&](int k) {
        const int ks = k % a.nkv_stage;
        if (!mbar_wait(bar(BAR_KVE + ks), ((k / a.nkv_stage) & 1) ^ 1, g, 28)) return false;
        const int pair = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
        const int bb = pair / hg, gg = pair - (pair / hg) * hg;
        const uint32_t dst = kv_base + ks * a.kv_stage_bytes;
        mbar_arrive_expect_tx(bar(BAR_KVF + ks), 2u * a.kv_bytes);
        tma_load_4d(dst, tk, bar(BAR_KVF + ks), 0, gg, 0, bb);
        tma_load_4d(dst + a.kv_bytes, tv, bar(BAR_KVF + ks), 0, gg, 0, bb);
        ++kv_n;
        return true;
    };
    int n = 0;
    bool ok = npairs > 0 ? load_kv(0) : true;
    for (; ok && n < n_items; ++n) {
        const GroupItem x = group_item(n, a.nblk, hg);
        const int st = n % a.nstage;
        if (!mbar_wait(bar(BAR_EMPTY + st), ((n / a.nstage) & 1) ^ 1, g, 20)) break;
        mbar_arrive_expect_tx(bar(BAR_FULL + st), 32u * 128u);
        tma_load_4d(tiles + st * a.stage_bytes, tq, bar(BAR_FULL + st), 0, x.group, 32 * x.blk,
                    x.batch);
        if (x.blk == 0 && x.k + 1 < npairs) ok = load_kv(x.k + 1);
    }
    // Never leave the CTA with a copy still landing in shared memory.
    WaitGuard drain = g;
    uint32_t no_abort = 0;
    drain.abort = &no_abort;
    for (int m = (n > a.nstage ? n - a.nstage : 0); m < n; ++m)
        mbar_wait(bar(BAR_FULL + m % a.nstage), (m / a.nstage) & 1, drain, 21);
    for (int k = (kv_n > a.nkv_stage ? kv_n - a.nkv_stage : 0); k < kv_n; ++k)
        mbar_wait(bar(BAR_KVF + k % a.nkv_stage), (k / a.nkv_stage) & 1, drain, 29);
}

// Grouped items, run by warp 2: once an item's staging block has landed,
// copy head p's 32 bytes of each of its 32 rows to rows [32p, 32p + 32),
// columns [16p, 16p + 16) of the stage's block-diagonal tile (16 bytes per
// copy, eight copies per thread: one row each), whose other entries stay
// zero; then a cross-proxy fence and one arrival per thread on the tile's
// barrier. Both tiles use the 128-byte swizzle, in which the
// 16-byte chunk c of row r sits at chunk c ^ (r % 8), and the tile's row
// 32p + r has the same r % 8 as the staging row r.
__device__ __forceinline__ void group_copier(uint32_t sbase, uint32_t tiles, int n_items,
                                             const ShortArgs &a, const WaitGuard &g) {
    auto bar = [&](int i) { return sbase + 8u * i; };
    const uint32_t r = threadIdx.x - 64u;  // 0 .. 31: the row of the block
    for (int n = 0; n < n_items; ++n) {
        const int st = n % a.nstage;
        const bool ok = mbar_wait(bar(BAR_FULL + st), (n / a.nstage) & 1, g, 23);
        if (!__all_sync(0xffffffffu, ok)) return;
        const uint32_t stg = tiles + st * a.stage_bytes;
        const uint32_t diag = stg + 32u * 128u;
#pragma unroll
        for (uint32_t c = 0; c < 8; ++c) {  // chunk c: head c / 2
            const uint32_t p = c >> 1;
            const uint32_t chunk = (c ^ (r & 7u)) << 4;
            uint32_t w0, w1, w2, w3;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                         : "r"(stg + r * 128u + chunk));
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                             diag + (32u * p + r) * 128u + chunk),
                         "r"(w0), "r"(w1), "r"(w2), "r"(w3)
                         : "memory");
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(BAR_DF + st));
    }
}

// The MMAs are issued by two threads, each waiting (bounded) on its own
// barriers only: lane 0 of warp 1 issues every QK^T, lane 0 of warp 3 every
// P V. A single thread polling both queues fell behind once every softmax
// warp of an item was busy: it shares its SM sub-partition with three
// softmax warps, and a P V went out up to ~3500 cycles after its P was
// stored. The two streams need no ordering between them beyond the slot
// barriers: QK^T of an item waits for the slot's previous epilogue, which
// follows that item's P V (o_full), and P V waits for P, which follows S.
template <int D, bool GRP>
struct MmaGeom {
    using G = ShortGeom<D>;
    static constexpr uint32_t SBO = GRP ? 1024u : G::SBO;  // 8 rows of 128 bytes when grouped
    static constexpr uint32_t LAYOUT = GRP ? kLayoutSw128 : G::LAYOUT;
    static constexpr uint32_t V_ROW = GRP ? 128u : G::ROW_BYTES;
};

// Waits until every MMA this thread issued has completed (TMEM is released
// after both issuers have done so).
__device__ __forceinline__ void drain_mmas(uint32_t done_bar, const WaitGuard &g, uint32_t site) {
    mma_commit(done_bar);
    WaitGuard drain = g;
    uint32_t no_abort = 0;
    drain.abort = &no_abort;
    mbar_wait(done_bar, 0, drain, site);
}

template <int D, bool BF16, bool GRP>
__device__ __forceinline__ void short_mma_s(uint32_t sbase, uint32_t tiles, uint32_t tmem,
                                            int n_items, const ShortArgs &a,
                                            const WaitGuard &g) {
    using M = MmaGeom<D, GRP>;
    auto bar = [&](int i) { return sbase + 8u * i; };
    // with a negative scale the S MMAs negate Q, so that the softmax always
    // works with a scale >= 0 (the products are the same, negation is exact)
    const uint32_t idesc_s = mma_idesc_f16(SHORT_BM, a.n_keys, BF16, false, false) |
                             (a.scale_log2 < 0.f ? kIdescNegateA : 0u);
    const uint64_t dk = smem_desc(tiles, 16, M::SBO, M::LAYOUT);  // Q and K, K-major
    const uint32_t kv_base = a.nstage * a.stage_bytes;  // grouped: the kv ring, after the stages
    for (int n = 0; n < n_items; ++n) {
        const int sl = n % a.nslot, st = n % a.nstage;
        int ks = 0;
        if constexpr (GRP) {
            // the block-diagonal tile is made; the first block of a pair
            // also waits for the pair's K/V (later blocks follow it)
            const int k = n / a.nblk;
            ks = k % a.nkv_stage;
            if (!mbar_wait(bar(BAR_DF + st), (n / a.nstage) & 1, g, 22)) break;
            if (n == k * a.nblk && !mbar_wait(bar(BAR_KVF + ks), (k / a.nkv_stage) & 1, g, 22))
                break;
        } else {
            if (!mbar_wait(bar(BAR_FULL + st), (n / a.nstage) & 1, g, 22)) break;
        }
        if (n >= a.nslot && !mbar_wait(bar(BAR_FREE + sl), ((n / a.nslot) - 1) & 1, g, 22)) break;
        tc_fence_after();
        const uint32_t tS = tmem + sl * a.slot_cols;
        if constexpr (GRP) {
            static_assert(D == 16, "grouped items: one K = 16 step per head");
            // the p-th MMA takes head p's 16 columns (32 bytes into the
            // 128-byte rows) of the diagonal tile and of K
            const uint64_t qd = dk + ((st * a.stage_bytes + 32u * 128u) >> 4);
            const uint64_t kd = dk + ((kv_base + ks * a.kv_stage_bytes) >> 4);
#pragma unroll
            for (int p = 0; p < 4; ++p) mma_ss(tS, qd + p * 2, kd + p * 2, idesc_s, p > 0 ? 1u : 0u);
            mma_commit(bar(BAR_SF + sl));
            mma_commit(bar(BAR_EMPTY + st));  // the stage is read once QK^T is done
        } else {
            const uint64_t qd = dk + ((st * a.stage_bytes) >> 4);
            const uint64_t kd = qd + (a.q_bytes >> 4);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                mma_ss(tS, qd + kk * 2, kd + kk * 2, idesc_s, kk > 0 ? 1u : 0u);
            mma_commit(bar(BAR_SF + sl));
        }
    }
    drain_mmas(bar(BAR_DONE), g, 25);
}

template <int D, bool BF16, bool GRP>
__device__ __forceinline__ void short_mma_o(uint32_t sbase, uint32_t tiles, uint32_t tmem,
                                            int n_items, const ShortArgs &a,
                                            const WaitGuard &g) {
    using M = MmaGeom<D, GRP>;
    auto bar = [&](int i) { return sbase + 8u * i; };
    // grouped items: P V over the group's four heads side by side, N = 64
    constexpr uint32_t idesc_o = mma_idesc_f16(SHORT_BM, GRP ? 64 : D, BF16, false, true);
    // V, MN-major; its N columns span one swizzle atom, so the leading offset
    // is not stepped through (it is set to the tile size, like a panel stride)
    const uint64_t dv = smem_desc(tiles, a.kv_bytes, M::SBO, M::LAYOUT);
    const uint32_t kv_base = a.nstage * a.stage_bytes;
    const int kv_steps = a.n_keys / 16;
    for (int n = 0; n < n_items; ++n) {
        const int sl = n % a.nslot, st = n % a.nstage;
        // the item's operands, worked out before the wait for its P
        const uint32_t tS = tmem + sl * a.slot_cols;
        int k = 0, ks = 0;
        uint32_t voff;
        if constexpr (GRP) {
            k = n / a.nblk;
            ks = k % a.nkv_stage;
            voff = kv_base + ks * a.kv_stage_bytes + a.kv_bytes;
        } else {
            voff = st * a.stage_bytes + a.q_bytes + a.kv_bytes;
        }
        const uint64_t vd = dv + (voff >> 4);
        if (!mbar_wait(bar(BAR_PF + sl), (n / a.nslot) & 1, g, 24)) break;
        tc_fence_after();
        for (int kk = 0; kk < kv_steps; ++kk)
            mma_ts(tS + a.o_off, tS + kk * 8, vd + ((kk * 16 * M::V_ROW) >> 4), idesc_o,
                   kk > 0 ? 1u : 0u);
        mma_commit(bar(BAR_OF + sl));
        if constexpr (GRP) {
            // the pair's last block releases its K/V
            if (n - k * a.nblk == a.nblk - 1) mma_commit(bar(BAR_KVE + ks));
        } else {
            mma_commit(bar(BAR_EMPTY + st));
        }
    }
    drain_mmas(bar(BAR_DONE2), g, 26);
}

template <int D, bool BF16, bool GRP>
__device__ __forceinline__ void short_softmax(uint32_t sbase, uint32_t tmem, int sl, int q4,
                                              int n_items, int ntile, const ShortArgs &a,
                                              const WaitGuard &g) {
    auto bar = [&](int i) { return sbase + 8u * i; };
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t tS = tmem + sl * a.slot_cols + (static_cast<uint32_t>(q4 * 32) << 16);
    const uint32_t tO = tS + a.o_off;
    // S arrives as sign(scale) * QK^T: with c = |scale| log2 e, the row max
    // of the raw scores is the max of the scaled ones
    const float c = fabsf(a.scale_log2);
    const int nch = a.n_keys / 32;
    // keys of the last 32-column chunk that exist (1..32)
    const int last_valid = a.sk - 32 * (nch - 1);
    const bool o_al32 = (reinterpret_cast<uintptr_t>(a.o) & 31u) == 0;

    int k = 0;
    for (int i = sl; i < n_items; i += a.nslot, ++k) {
        // this warp's 32 rows: (batch, head), first query row, and the
        // column of their O in the slot (their head's 16 of the group's 64
        // when grouped: warp q4 has head q4 of the group)
        int xb, xh, row0, ocol = 0;
        bool warp_live;
        if constexpr (GRP) {
            const GroupItem x = group_item(i, a.nblk, a.h / 4);
            xb = x.batch;
            xh = 4 * x.group + q4;
            row0 = 32 * x.blk;
            ocol = D * q4;
            warp_live = true;
        } else {
            const Item x = item_of(blockIdx.x + i * gridDim.x, ntile, a.h);
            xb = x.batch;
            xh = x.head;
            row0 = x.tile * SHORT_BM + q4 * 32;
            warp_live = row0 < a.sq;
        }
        const int grow = row0 + static_cast<int>(lane);
        const bool ok = mbar_wait(bar(BAR_SF + sl), k & 1, g, 26);
        if (!__all_sync(0xffffffffu, ok)) return;
        tc_fence_after();

        float m_ref = -INFINITY, l = 1.f;
        if (warp_live) {
            // One pass over S, two 32-column chunks per TMEM round trip: the
            // pair's max moves the reference max only past the lazy threshold; then its P is
            // stored into the pair's first 32 columns, whose scores have been
            // read. Only the last chunk can be ragged.
            const uint64_t c2 = f2_make(c, c);
            uint64_t acc2[2] = {0ull, 0ull};
#pragma unroll 1
            for (int ch = 0; ch < nch; ch += 2) {
                {
                    uint32_t r[2][32];
                    tmem_ld32(tS + 32 * ch, r[0]);
                    if (ch + 1 < nch) tmem_ld32(tS + 32 * (ch + 1), r[1]);
                    tmem_wait_ld();
                    float mx[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) mx[q] = -INFINITY;
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int cc = ch + h2;
                        if (cc < nch) {
                            const bool ragged = cc == nch - 1 && last_valid < 32;
                            if (ragged) chunk_max<true>(r[h2], last_valid, mx);
                            else chunk_max<false>(r[h2], 32, mx);
                        }
                    }
                    const float mraw = fmaxf(max3f(mx[0], mx[1], mx[2]), mx[3]);
                    const float m_pair = mraw * c;  // log2 units
                    const bool need = m_pair > m_ref + 8.0f;
                    // 0 on the first pair (nothing stored yet), 1 where kept;
                    // the P already stored is rescaled after this pair's
                    // exponentials, once its scores are out of registers
                    const bool moved = __any_sync(0xffffffffu, need);
                    float alpha = 1.0f;
                    if (moved) {
                        const float m_new = need ? m_pair : m_ref;
                        alpha = fast_exp2(m_ref - m_new);
                        acc2[0] = f2_mul(acc2[0], f2_make(alpha, alpha));
                        acc2[1] = f2_mul(acc2[1], f2_make(alpha, alpha));
                        m_ref = m_new;
                    }
                    const uint64_t nm2 = f2_make(-m_ref, -m_ref);
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int cc = ch + h2;
                        if (cc < nch) {
                            if (cc == nch - 1 && last_valid < 32)
                                chunk_exp<true, BF16>(r[h2], last_valid, c2, nm2, acc2, tS + 16 * cc);
                            else
                                chunk_exp<false, BF16>(r[h2], 32, c2, nm2, acc2, tS + 16 * cc);
                        }
                    }
                    if (moved && ch > 0) rescale_p<BF16>(tS, 16 * ch, alpha);
                }
            }
            tmem_wait_st();
            float a0, a1, a2, a3;
            f2_split(acc2[0], a0, a1);
            f2_split(acc2[1], a2, a3);
            l = (a0 + a1) + (a2 + a3);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_PF + sl));

        // ---------------------------------------------------- epilogue
        // the row's output address and 1 / l, worked out before the wait for O
        constexpr int OCH = D < 32 ? D : 32;
        const bool row_out = warp_live && grow < a.sq;
        const float inv_l = 1.0f / l;
        const int64_t orow =
            ((static_cast<int64_t>(xb) * a.sq + (row_out ? grow : 0)) * a.h + xh) * D;
        uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(a.o) + orow);
        const bool okf = mbar_wait(bar(BAR_OF + sl), k & 1, g, 27);
        if (!__all_sync(0xffffffffu, okf)) return;
        tc_fence_after();
        // O row read out 32 columns at a time (16 at d = 16); the slot goes
        // back to the MMA issuer as soon as the last piece is in registers,
        // before that piece is scaled, packed and stored
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += OCH) {
            uint32_t ov[OCH];
            if (warp_live) {
                if constexpr (OCH == 32)
                    tmem_ld32(tO + ocol + c0, *reinterpret_cast<uint32_t(*)[32]>(ov));
                else
                    tmem_ld16(tO + ocol + c0, *reinterpret_cast<uint32_t(*)[16]>(ov));
                tmem_wait_ld();
            }
            if (c0 + OCH == D) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(BAR_FREE + sl));
            }
            if (row_out) {
#pragma unroll
                for (int e0 = 0; e0 < OCH; e0 += 16) {
                    uint32_t pk[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        pk[e] = pack2s<BF16>(__uint_as_float(ov[e0 + 2 * e]) * inv_l,
                                             __uint_as_float(ov[e0 + 2 * e + 1]) * inv_l);
                    if (o_al32) {
                        st_global_v8(dst + (c0 + e0) / 8, pk);
                    } else {
                        dst[(c0 + e0) / 8] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        dst[(c0 + e0) / 8 + 1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                    }
                }
            }
        }
        if (row_out)
            a.lse[(static_cast<int64_t>(xb) * a.h + xh) * a.sq + grow] =
                (m_ref + __log2f(l)) * 0.69314718055994530942f;
    }
}

// Three slots launch 512 threads at 128 registers; the control warpgroup
// gives some of its share to the softmax warpgroups, whose single pass holds
// two 32-column chunks of scores and their exponentials in flight. Two slots
// (384 threads) launch at 168 and need no rebalancing.
constexpr int kShortRegsControl = 72;
constexpr int kShortRegsSoftmax = 144;
static_assert(4 * kShortRegsControl + 12 * kShortRegsSoftmax <= 16 * 128, "register split");

template <int D, bool BF16, int NWG, bool GRP>
__global__ void __launch_bounds__(128 * (NWG + 1), 1)
    fwd_short_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv, const ShortArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw);
    const uint32_t tiles = sbase + SH_BAR_BYTES;
    auto bar = [&](int i) { return sbase + 8u * i; };

    const int warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    const int ntile = (a.sq + SHORT_BM - 1) / SHORT_BM;
    // grouped: the CTA's (batch, group) pairs times the query blocks of each
    const int units = GRP ? a.b * (a.h / 4) : ntile * a.h * a.b;
    const int n_units =
        blockIdx.x < units ? (units - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
    const int items = units;  // plain items: one per unit
    const int n_items = GRP ? n_units * a.nblk : n_units;

    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + OFF_MISC + 4);
    if (threadIdx.x == 0) {
        for (int i = 0; i < NUM_BARS; ++i) {
            const bool by_warps = (i >= BAR_PF && i < BAR_PF + SH_WG) ||
                                  (i >= BAR_FREE && i < BAR_FREE + SH_WG);
            const bool by_copiers = i >= BAR_DF && i < BAR_DF + SHORT_MAX_STAGES;
            // one arrive per softmax warp; per copying thread (diagonal tiles)
            mbar_init(bar(i), by_warps ? 4u : (by_copiers ? 32u : 1u));
        }
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    if constexpr (GRP) {
        // the zeros of every stage's block-diagonal tile (the copiers only
        // ever write its diagonal blocks), visible to the tensor core
        for (int st = 0; st < a.nstage; ++st)
            for (uint32_t off = 16u * threadIdx.x; off < 128u * 128u; off += 16u * blockDim.x)
                st_shared_zero16(tiles + st * a.stage_bytes + 32u * 128u + off);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitGuard g{abort_flag, a.status, kKernFwd};

    if (warp < 4) {
        if constexpr (NWG == 3) reg_dealloc<kShortRegsControl>();
        if (warp == 0) {
            if (lane == 0 && !(a.flags & kFlagSkipLoads)) {
                if constexpr (GRP)
                    group_producer(&tq, &tk, &tv, sbase, tiles, n_items, a.h / 4, a, g);
                else
                    short_producer<D>(&tq, &tk, &tv, sbase, tiles, items, ntile, a, g);
            }
        } else if (warp == 1) {
            if (lane == 0) short_mma_s<D, BF16, GRP>(sbase, tiles, tmem, n_items, a, g);
        } else if (warp == 3) {
            if (lane == 0) short_mma_o<D, BF16, GRP>(sbase, tiles, tmem, n_items, a, g);
        } else if constexpr (GRP) {
            group_copier(sbase, tiles, n_items, a, g);
        }
    } else {
        if constexpr (NWG == 3) reg_alloc<kShortRegsSoftmax>();
        short_softmax<D, BF16, GRP>(sbase, tmem, (warp - 4) >> 2, warp & 3, n_items, ntile, a,
                                    g);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int D, bool BF16, int NWG, bool GRP>
cudaError_t launch_short_w(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                           const ShortArgs &a, int grid, cudaStream_t stream) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_set[dev]) {
        e = cudaFuncSetAttribute(fwd_short_kernel<D, BF16, NWG, GRP>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, SHORT_SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    fwd_short_kernel<D, BF16, NWG, GRP>
        <<<grid, 128 * (NWG + 1), SHORT_SMEM_BYTES, stream>>>(tq, tk, tv, a);
    return cudaGetLastError();
}

template <int D, bool BF16, bool GRP>
cudaError_t launch_short_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                           const ShortArgs &a, int grid, cudaStream_t stream) {
    switch (a.nslot) {
        case 2: return launch_short_w<D, BF16, 2, GRP>(tq, tk, tv, a, grid, stream);
        case 3: return launch_short_w<D, BF16, 3, GRP>(tq, tk, tv, a, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool short_plan(int sq, int sk, int h, int d, bool grouped_ok, ShortArgs *a) {
    if (sq < 1 || sk < 1 || h < 1 || sk > SHORT_MAX_KEYS || (d != 16 && d != 32 && d != 64))
        return false;
    const int n = (sk + 31) / 32 * 32;
    const int o_off = (n / 2 + 31) / 32 * 32;
    constexpr int avail = SHORT_SMEM_BYTES - 1024 - SH_BAR_BYTES;
    // grouped items at head dim 16 when the heads come in fours
    if (grouped_ok && d == 16 && h % 4 == 0) {
        const int kv_bytes = n * 128;                       // one group K or V tile
        const int stage_bytes = 32 * 128 + 128 * 128;       // staging block + diagonal tile
        int w = n > o_off + 64 ? n : o_off + 64;
        w = (w + 31) / 32 * 32;
        int slots = 512 / w;
        if (slots > SHORT_MAX_SLOTS) slots = SHORT_MAX_SLOTS;
        // three kv stages when four query stages still fit, else two
        const int nkv = 3 * 2 * kv_bytes + 4 * stage_bytes <= avail ? 3 : 2;
        int stages = (avail - nkv * 2 * kv_bytes) / stage_bytes;
        if (stages > SHORT_MAX_STAGES) stages = SHORT_MAX_STAGES;
        if (stages >= 2) {
            if (slots > stages) slots = stages;
            a->n_keys = n;
            a->o_off = o_off;
            a->slot_cols = w;
            a->nslot = slots;
            a->kv_bytes = kv_bytes;
            a->stage_bytes = stage_bytes;
            a->nstage = stages;
            a->grouped = 1;
            a->nblk = (sq + 31) / 32;
            a->kv_stage_bytes = 2 * kv_bytes;
            a->nkv_stage = nkv;
            a->q_bytes = stage_bytes;
            return true;
        }
    }
    const int row_bytes = d * 2;
    int w = n > o_off + d ? n : o_off + d;
    w = (w + 31) / 32 * 32;
    int slots = 512 / w;
    if (slots > SHORT_MAX_SLOTS) slots = SHORT_MAX_SLOTS;
    const int kv_bytes = n * row_bytes;
    const int q_bytes = SHORT_BM * row_bytes;
    const int stage_bytes = q_bytes + 2 * kv_bytes;  // a multiple of 1024
    int stages = avail / stage_bytes;
    if (stages > SHORT_MAX_STAGES) stages = SHORT_MAX_STAGES;
    if (stages < 1) return false;
    // the MMA issuer runs a slot's P V up to slots - 1 items behind its
    // QK^T, so the stage ring must hold at least one item per slot
    if (slots > stages) slots = stages;
    a->n_keys = n;
    a->o_off = o_off;
    a->slot_cols = w;
    a->nslot = slots;
    a->kv_bytes = kv_bytes;
    a->stage_bytes = stage_bytes;
    a->nstage = stages;
    a->grouped = 0;
    a->nblk = 0;
    a->kv_stage_bytes = 0;
    a->nkv_stage = 0;
    a->q_bytes = q_bytes;
    return true;
}

int64_t short_units(const ShortArgs &a, int64_t b, int64_t h) {
    if (a.grouped) return b * (h / 4);
    return b * h * ((a.sq + SHORT_BM - 1) / SHORT_BM);
}

cudaError_t launch_fwd_short(int d, bool bf16, const CUtensorMap &tq, const CUtensorMap &tk,
                             const CUtensorMap &tv, const ShortArgs &a, int grid,
                             cudaStream_t stream) {
#define EXATTN_SHORT_CASE(DD)                                                       \
    case DD:                                                                        \
        return bf16 ? launch_short_t<DD, true, false>(tq, tk, tv, a, grid, stream)  \
                    : launch_short_t<DD, false, false>(tq, tk, tv, a, grid, stream);
    if (a.grouped) {
        if (d != 16) return cudaErrorInvalidValue;
        return bf16 ? launch_short_t<16, true, true>(tq, tk, tv, a, grid, stream)
                    : launch_short_t<16, false, true>(tq, tk, tv, a, grid, stream);
    }
    switch (d) {
        EXATTN_SHORT_CASE(16)
        EXATTN_SHORT_CASE(32)
        EXATTN_SHORT_CASE(64)
        default:
            return cudaErrorInvalidValue;
    }
#undef EXATTN_SHORT_CASE
}

}  // namespace exattn

extern "C" int attn_debug_short_plan(int sq, int sk, int h, int d, int grouped_ok, int *out) {
    exattn::ShortArgs a{};
    if (out == nullptr || !exattn::short_plan(sq, sk, h, d, grouped_ok != 0, &a)) return 0;
    // grouped: the query stages, then the K/V ring; plain: the stages alone
    const int used = a.nstage * a.stage_bytes + (a.grouped ? a.nkv_stage * a.kv_stage_bytes : 0);
    const int v[12] = {a.n_keys,  a.o_off, a.slot_cols, a.nslot,     a.kv_bytes, a.stage_bytes,
                       a.nstage,  a.grouped, a.nblk,    a.nkv_stage, used,
                       exattn::SHORT_SMEM_BYTES - 1024 - exattn::SH_BAR_BYTES};
    for (int i = 0; i < 12; ++i) out[i] = v[i];
    return 1;
}
