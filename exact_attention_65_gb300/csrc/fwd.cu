// Forward exact attention on sm_103a: TMA-staged Q/K/V tiles, S = Q K^T and
// O += P V as tcgen05 MMAs accumulating in tensor memory, and an online
// softmax with one thread per query row.
//
// What is computed follows "Why FlashAttention is fast": the score matrix
// is cut into tiles (section 3.1), the whole QK^T -> softmax -> PV chain
// runs in one kernel with the intermediates on chip (section 3.2), and the
// softmax is done online: a running max and running sum per row, with the
// partial output rescaled whenever the reference max moves (section 3.3).
// The per-row log-sum-exp is emitted beside O.
//
// Persistent CTAs (one per SM, 384 threads) loop over work units; a unit is
// two 128-row query tiles of one (batch, head), and the units are visited
// query block first, so CTAs running at the same time share the head's K/V
// through L2. Roles:
//   warp 0        TMA producer: the unit's Q tiles, then K_j and V_j through
//                 one ring of K/V slots; it runs ahead into the next
//                 unit as soon as the slots free up.
//   warp 1        TMEM owner and MMA issuer (one thread): S_j(t) = Q_t K_j^T
//                 into TMEM, then O_t += P_j(t) V_j with P read from TMEM.
//   warps 2-3     idle.
//   warps 4-7     softmax and epilogue for query tile 0, warps 8-11 for
//                 query tile 1: thread i of warp w owns row 32 (w % 4) + i of
//                 its tile (a warp may only touch its quarter of TMEM lanes).
// Registers are rebalanced per warpgroup with setmaxnreg: warps 0-3 drop to
// 96 per thread and the two softmax warpgroups rise to 200, within the
// 384 x 168 the CTA is launched with.
// The two query tiles ping-pong: while one warpgroup exponentiates its S
// tile, the tensor core works on the other tile's MMAs. A warpgroup hands
// its O accumulator back (o_empty) once it has read it out, so the next
// unit's QK^T MMAs overlap this unit's epilogue.
//
// TMEM (512 columns, fp32): tile t uses columns [256t, 256t+128) for S_j,
// overwritten in place by P_j packed two 16-bit values per column, and
// [256t+128, 256t+128+d) for the O accumulator. tcgen05.mma instructions
// issued by one thread execute in order, so S_{j+1}(t) is only written after
// P_j(t) V_j has read P_j(t) from the same columns.
//
// Lazy rescaling: a row keeps its reference max m until a tile's max
// exceeds it by more than 8 (log2 units). P = 2^(s*c - m) then stays at most
// 2^8, which fp16/bf16 and the fp32 sums hold exactly as well as values
// below 1; the final O/l and LSE = m + log2(l) are the same quantity.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace exattn {
namespace {

// Bit 13 of a kind::f16 instruction descriptor: negate the A operand.
constexpr uint32_t kIdescNegateA = 1u << 13;

template <int D>
struct FwdGeom {
    static constexpr int BM = FWD_BM;
    static constexpr int BN = FWD_BN;
    static constexpr int QT = FWD_QTILES;
    static constexpr int ROW_BYTES = fwd_row_bytes(D);
    static constexpr int PANELS = (D * 2) / ROW_BYTES;
    static constexpr int PANEL_ELEMS = ROW_BYTES / 2;
    static constexpr int Q_PANEL_BYTES = BM * ROW_BYTES;
    static constexpr int KV_PANEL_BYTES = BN * ROW_BYTES;
    static constexpr int Q_TILE_BYTES = BM * D * 2;
    static constexpr int KV_TILE_BYTES = BN * D * 2;
    // One ring of K/V tile slots; items flow K_0, V_0, K_1, V_1, ...
    static constexpr int SLOTS = D == 128 ? 5 : 8;
    // Q buffers (QT tiles each). Measured: one Q buffer and a deeper K/V ring
    // beat two Q buffers and a 3-slot ring at d = 128.
    static constexpr int QBUF = D <= 64 ? 2 : 1;  // next unit's Q loads early where smem allows
    static constexpr int Q_BUF_BYTES = QT * Q_TILE_BYTES;
    static constexpr uint32_t LAYOUT =
        ROW_BYTES == 128 ? kLayoutSw128 : (ROW_BYTES == 64 ? kLayoutSw64 : kLayoutSw32);
    static constexpr uint32_t SBO = 8 * ROW_BYTES;  // bytes between 8-row core-matrix groups
    static constexpr int TMEM_COLS = 512;
    static constexpr int TMEM_TILE_STRIDE = 256;
    static constexpr int TMEM_O_OFF = 128;
    static constexpr int OCH = D < 32 ? D : 32;  // O columns per TMEM access

    static constexpr int OFF_Q = 0;
    static constexpr int OFF_KV = OFF_Q + QBUF * Q_BUF_BYTES;
    static constexpr int OFF_BAR = OFF_KV + SLOTS * KV_TILE_BYTES;
    // barriers: q_full[QBUF] | q_empty[QBUF] | kv_full[SLOTS] |
    //           kv_empty[SLOTS] | s_full[QT] | p_full[QT] | o_full[QT] |
    //           o_empty[QT] | done | v_land | v_fix
    static constexpr int BAR_QF = 0;              // [QBUF]
    static constexpr int BAR_QE = BAR_QF + QBUF;  // [QBUF]
    static constexpr int BAR_KVF = BAR_QE + QBUF;
    static constexpr int BAR_KVE = BAR_KVF + SLOTS;
    static constexpr int BAR_SF = BAR_KVE + SLOTS;
    static constexpr int BAR_PF = BAR_SF + QT;
    static constexpr int BAR_OF = BAR_PF + QT;
    static constexpr int BAR_OE = BAR_OF + QT;
    static constexpr int BAR_DONE = BAR_OE + QT;
    static constexpr int BAR_VLAND = BAR_DONE + 1;  // paged: last V tile landed (MMA -> zeroing)
    static constexpr int BAR_VFIX = BAR_VLAND + 1;  // paged: its stale rows zeroed (zeroing -> MMA)
    static constexpr int NUM_BARS = BAR_VFIX + 1;
    // The kernel for units with one live query tile puts S of odd key tiles
    // in the second tile's S columns and uses that tile's barriers, idle
    // there: its S full and P full barriers, and its O full barrier for one
    // completed by every P V (an O rescale waits for the one before it).
    static constexpr int BAR_SF2 = BAR_SF + 1;
    static constexpr int BAR_PF2 = BAR_PF + 1;
    static constexpr int BAR_PVD = BAR_OF + 1;
    static_assert(QT == 2, "the one-tile kernel borrows the second tile's barriers");
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int USED = OFF_MISC + 16;
    // Keep one CTA per SM: it owns all 512 TMEM columns.
    static constexpr int MIN_SMEM = 120 * 1024;
    static constexpr int SMEM_BYTES = (USED > MIN_SMEM ? USED : MIN_SMEM) + 1024;
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static_assert(D % 16 == 0 && D >= 16 && D <= 128, "head dim");
};

// Per-thread register budgets after the rebalance: 4 warps at kRegsControl
// plus 8 at kRegsSoftmax may not exceed 12 warps at the launch's 168.
constexpr int kRegsLaunch = 168;
constexpr int kRegsControl = 96;  // below this the MMA issuer spills
constexpr int kRegsSoftmax = 200;
static_assert(4 * kRegsControl + 8 * kRegsSoftmax <= 12 * kRegsLaunch, "register split");
static_assert(FWD_THREADS == 12 * 32, "three warpgroups");

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (BF16)
        return cvt_pack_bf16(lo, hi);
    else
        return cvt_pack_f16(lo, hi);
}

// A work unit: query rows [m0, m0 + 256) of one (batch, head) against key
// tiles [kv0, kv0 + nkv) (all of them unless the keys are split); n_qt of its
// two 128-row tiles hold rows below sq.
struct Unit {
    int m0, head, batch, n_qt, split, kv0, nkv;
    int sk;  // keys of this unit's sequence (a.sk unless the cache is paged)
};

// Units are numbered query block first, then split, head and batch. SPLIT
// picks the kernel's compiled form: 0 the plain forward, 1 the causal forward
// over all keys of a head, 2 key ranges (split-KV decode, paged caches) with
// the mask a run-time choice; each keeps only the code it needs.
template <int SPLIT, bool PAGED>
__device__ __forceinline__ Unit unit_of(int u, int nqb, int nkv_all, const FwdArgs &a) {
    Unit x;
    int qb = u % nqb;
    int r = u / nqb;
    // Causal units grow with the query block. Run longest first across all
    // (batch, head) pairs, each CTA's strided share mixes long and short
    // units whatever the grid. (Reversing every other group's query blocks
    // instead keeps a head's units together, but when the grid is a multiple
    // of the query blocks per head it hands each CTA one block index: b4 s512
    // h32 43.7 against 30 us, b16 s1024 h16 157 against 101 us.)
    const bool causal = SPLIT == 1 || (SPLIT == 2 && a.causal);
    if (causal) {
        if (SPLIT == 1 || a.longest_first) {
            const int per = (SPLIT == 2 ? a.splits : 1) * a.h * a.b;  // units per query block
            qb = nqb - 1 - u / per;
            r = u % per;
        } else if (r & 1) {
            qb = nqb - 1 - qb;
        }
    }
    x.split = 0;
    x.kv0 = 0;
    x.nkv = nkv_all;
    x.sk = a.sk;
    if constexpr (SPLIT == 2) {
        x.split = r % a.splits;
        r /= a.splits;
    }
    x.head = r % a.h;
    x.batch = r / a.h;
    if constexpr (SPLIT == 2) {
        if constexpr (PAGED) {  // the sequence's own length, on the device
            x.sk = min(max(__ldg(a.seqlens + x.batch), 0), a.sk);
            nkv_all = (x.sk + FWD_BN - 1) / FWD_BN;
        }
        x.kv0 = x.split * a.tiles_per_split;
        x.nkv = max(0, min(a.tiles_per_split, nkv_all - x.kv0));
    }
    x.m0 = qb * (FWD_BM * FWD_QTILES);
    x.n_qt = min(FWD_QTILES, (a.sq - x.m0 + FWD_BM - 1) / FWD_BM);
    if constexpr (SPLIT != 0) {
        if (causal) {
            // the unit's last row sees keys up to last + sk - sq: later key
            // tiles are not needed (none at all if that is below 0)
            const int last = min(x.m0 + FWD_BM * FWD_QTILES, a.sq) - 1;
            const int kmax = last + x.sk - a.sq;
            const int tiles = kmax < 0 ? 0 : kmax / FWD_BN + 1;
            x.nkv = max(0, min(x.nkv, tiles - x.kv0));
        }
    }
    return x;
}

template <int D, int SPLIT, bool PAGED>
__device__ __forceinline__ void fwd_producer(const CUtensorMap *tq, const CUtensorMap *tk,
                                             const CUtensorMap *tv, uint32_t sbase, int nqb,
                                             int units, int nkv, const FwdArgs &a,
                                             const WaitGuard &g) {
    using G = FwdGeom<D>;
    auto bar = [&](int i) { return sbase + G::OFF_BAR + 8u * i; };
    // K/V are re-read by every query block of the head; with one query block
    // they are read once, and kept out of the way in L2 instead
    const uint64_t keep = nqb > 1 ? policy_evict_last() : policy_evict_first();

    int q_issued = 0, n_issued = 0;  // n counts ring items (K and V tiles)
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        const Unit x = unit_of<SPLIT, PAGED>(u, nqb, nkv, a);
        // A Q buffer is free once every S MMA of the unit two back has completed.
        const int qb = q_issued % G::QBUF;
        if (!mbar_wait(bar(G::BAR_QE + qb), ((q_issued / G::QBUF) & 1) ^ 1, g, 1)) break;
        mbar_arrive_expect_tx(bar(G::BAR_QF + qb), x.n_qt * G::Q_TILE_BYTES);
        for (int t = 0; t < x.n_qt; ++t)
            for (int p = 0; p < G::PANELS; ++p)
                tma_load_4d(sbase + G::OFF_Q + qb * G::Q_BUF_BYTES + t * G::Q_TILE_BYTES +
                                p * G::Q_PANEL_BYTES,
                            tq, bar(G::BAR_QF + qb), p * G::PANEL_ELEMS, x.head, x.m0 + t * G::BM,
                            x.batch);
        ++q_issued;
        for (int i = 0; i < 2 * x.nkv; ++i) {  // K_j at i = 2j, V_j at i = 2j + 1
            const int s = n_issued % G::SLOTS;
            const uint32_t ph = (n_issued / G::SLOTS) & 1;
            if (!mbar_wait(bar(G::BAR_KVE + s), ph ^ 1, g, 2)) {
                ok = false;
                break;
            }
            mbar_arrive_expect_tx(bar(G::BAR_KVF + s), G::KV_TILE_BYTES);
            const CUtensorMap *map = (i & 1) ? tv : tk;
            const uint32_t dst = sbase + G::OFF_KV + s * G::KV_TILE_BYTES;
            const int row0 = (x.kv0 + (i >> 1)) * G::BN;
            for (int p = 0; p < G::PANELS; ++p)
                tma_load_4d_hint(dst + p * G::KV_PANEL_BYTES, map, bar(G::BAR_KVF + s),
                                 p * G::PANEL_ELEMS, x.head, row0, x.batch, keep);
            ++n_issued;
        }
    }
    // Never leave the CTA with a copy still landing in shared memory: wait
    // (bounded, even after an abort) for the last load issued into each slot.
    WaitGuard drain = g;
    uint32_t no_abort = 0;
    drain.abort = &no_abort;
    for (int n = (q_issued > G::QBUF ? q_issued - G::QBUF : 0); n < q_issued; ++n)
        mbar_wait(bar(G::BAR_QF + n % G::QBUF), (n / G::QBUF) & 1, drain, 9);
    for (int n = (n_issued > G::SLOTS ? n_issued - G::SLOTS : 0); n < n_issued; ++n)
        mbar_wait(bar(G::BAR_KVF + n % G::SLOTS), (n / G::SLOTS) & 1, drain, 10);
}

// The producer for paged caches, run by the whole of warp 0: lane 0 waits
// for the slots and arms their barriers, and the K/V tiles are gathered as
// boxes of box_rows rows (each inside one page), one box per lane, so that
// the block-table lookups and TMA issues of a tile run side by side instead
// of one after another (a tile of 16-key pages is 8 boxes per panel). A box
// wholly past the sequence's end is addressed past the last pool page, so
// TMA fills it with zeros; rows past the end inside the last box hold stale
// data (masked for K, zeroed for V before the P V MMA).
template <int D, int SPLIT, bool PAGED>
__device__ __forceinline__ void fwd_producer_paged(const CUtensorMap *tq, const CUtensorMap *tk,
                                                   const CUtensorMap *tv, uint32_t sbase, int nqb,
                                                   int units, int nkv, const FwdArgs &a,
                                                   const WaitGuard &g) {
    using G = FwdGeom<D>;
    auto bar = [&](int i) { return sbase + G::OFF_BAR + 8u * i; };
    const uint32_t lane = threadIdx.x & 31;
    const uint64_t keep = nqb > 1 ? policy_evict_last() : policy_evict_first();
    const int nbox = G::BN / a.box_rows;  // 1 .. 8

    int q_issued = 0, n_issued = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        const Unit x = unit_of<SPLIT, PAGED>(u, nqb, nkv, a);
        const int qb = q_issued % G::QBUF;
        bool got = true;
        if (lane == 0) {
            got = mbar_wait(bar(G::BAR_QE + qb), ((q_issued / G::QBUF) & 1) ^ 1, g, 1);
            if (got) {
                mbar_arrive_expect_tx(bar(G::BAR_QF + qb), x.n_qt * G::Q_TILE_BYTES);
                for (int t = 0; t < x.n_qt; ++t)
                    for (int p = 0; p < G::PANELS; ++p)
                        tma_load_4d(sbase + G::OFF_Q + qb * G::Q_BUF_BYTES + t * G::Q_TILE_BYTES +
                                        p * G::Q_PANEL_BYTES,
                                    tq, bar(G::BAR_QF + qb), p * G::PANEL_ELEMS, x.head,
                                    x.m0 + t * G::BM, x.batch);
            }
        }
        if (!__shfl_sync(0xffffffffu, got, 0)) break;
        ++q_issued;
        for (int i = 0; i < 2 * x.nkv; ++i) {  // K_j at i = 2j, V_j at i = 2j + 1
            const int s = n_issued % G::SLOTS;
            const uint32_t ph = (n_issued / G::SLOTS) & 1;
            // this lane's box: its page is looked up before the slot is waited for
            const int key = (x.kv0 + (i >> 1)) * G::BN + static_cast<int>(lane) * a.box_rows;
            int page = a.num_pages, prow = 0;
            if (static_cast<int>(lane) < nbox && key < x.sk) {
                const int lp = key / a.page_size;
                page = min(max(__ldg(a.block_table + static_cast<int64_t>(x.batch) * a.max_pages + lp),
                               0),
                           a.num_pages - 1);
                prow = key - lp * a.page_size;
            }
            bool free_slot = true;
            if (lane == 0) {
                free_slot = mbar_wait(bar(G::BAR_KVE + s), ph ^ 1, g, 2);
                if (free_slot) mbar_arrive_expect_tx(bar(G::BAR_KVF + s), G::KV_TILE_BYTES);
            }
            if (!__shfl_sync(0xffffffffu, free_slot, 0)) {
                ok = false;
                break;
            }
            if (static_cast<int>(lane) < nbox) {
                const CUtensorMap *map = (i & 1) ? tv : tk;
                const uint32_t dst = sbase + G::OFF_KV + s * G::KV_TILE_BYTES +
                                     lane * a.box_rows * G::ROW_BYTES;
                for (int p = 0; p < G::PANELS; ++p)
                    tma_load_4d_hint(dst + p * G::KV_PANEL_BYTES, map, bar(G::BAR_KVF + s),
                                     p * G::PANEL_ELEMS, x.head, prow, page, keep);
            }
            __syncwarp();
            ++n_issued;
        }
    }
    // Never leave the CTA with a copy still landing in shared memory.
    if (lane == 0) {
        WaitGuard drain = g;
        uint32_t no_abort = 0;
        drain.abort = &no_abort;
        for (int n = (q_issued > G::QBUF ? q_issued - G::QBUF : 0); n < q_issued; ++n)
            mbar_wait(bar(G::BAR_QF + n % G::QBUF), (n / G::QBUF) & 1, drain, 9);
        for (int n = (n_issued > G::SLOTS ? n_issued - G::SLOTS : 0); n < n_issued; ++n)
            mbar_wait(bar(G::BAR_KVF + n % G::SLOTS), (n / G::SLOTS) & 1, drain, 10);
    }
}

// Paged caches: a unit's last K/V tile can end inside the sequence's last
// page, whose rows past the end hold stale data. P is exactly 0 there, but the
// tensor core still multiplies those V rows (0 * NaN is NaN), so warps 2-3
// zero them in shared memory (whole swizzled rows: a row's bytes stay in its
// own 16-byte-chunk group under every swizzle mode). The MMA issuer, which
// consumes the ring in order, tells them when that V tile has landed
// (BAR_VLAND; waiting on the ring's own barrier from here could match an
// older phase of the same parity), and they hand the tile back through
// BAR_VFIX before its P V reads it.
template <bool PAGED>
__device__ __forceinline__ bool unit_needs_v_fix(const Unit &x) {
    return PAGED && x.nkv > 0 && (x.kv0 + x.nkv) * FWD_BN > x.sk;
}

template <int D, int SPLIT, bool PAGED>
__device__ __forceinline__ void fwd_fix_v(uint32_t sbase, int nqb, int units, int nkv,
                                          const FwdArgs &a, const WaitGuard &g) {
    using G = FwdGeom<D>;
    auto bar = [&](int i) { return sbase + 8u * i + G::OFF_BAR; };
    const int t = threadIdx.x - 64;  // warps 2-3
    const uint32_t lane = threadIdx.x & 31;
    constexpr int CPR = G::ROW_BYTES / 16;  // 16-byte chunks per row and panel
    int kv_base = 0;
    int fix_cnt = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const Unit x = unit_of<SPLIT, PAGED>(u, nqb, nkv, a);
        if (unit_needs_v_fix<PAGED>(x)) {
            const int nv = 2 * (kv_base + x.nkv - 1) + 1;  // ring item of the last V tile
            const int slot = nv % G::SLOTS;
            // The issuer has seen the tile land and holds the slot until the
            // hand-back, so the ring barrier's current phase is this item's.
            bool ok = mbar_wait(bar(G::BAR_VLAND), fix_cnt & 1, g, 15);
            ok = ok && mbar_wait(bar(G::BAR_KVF + slot), (nv / G::SLOTS) & 1, g, 16);
            ++fix_cnt;
            if (!__all_sync(0xffffffffu, ok)) return;
            const int valid = x.sk - (x.kv0 + x.nkv - 1) * G::BN;  // 1 .. BN - 1
            const int per_panel = (G::BN - valid) * CPR;
            const uint32_t base = sbase + G::OFF_KV + slot * G::KV_TILE_BYTES;
            for (int c = t; c < per_panel * G::PANELS; c += 64) {
                const int p = c / per_panel;
                const int rem = c - p * per_panel;
                st_shared_zero16(base + p * G::KV_PANEL_BYTES + (valid + rem / CPR) * G::ROW_BYTES +
                                 (rem % CPR) * 16);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(G::BAR_VFIX));
        }
        kv_base += x.nkv;
    }
}

template <int D, bool BF16, int SPLIT, bool PAGED, bool ONE>
__device__ __forceinline__ void fwd_mma(uint32_t sbase, uint32_t tmem, int nqb, int units,
                                        int nkv, const FwdArgs &a, const WaitGuard &g) {
    using G = FwdGeom<D>;
    auto bar = [&](int i) { return sbase + G::OFF_BAR + 8u * i; };
    // with a negative scale the S MMAs negate Q, so that the softmax always
    // works with a scale >= 0 (the products are the same, negation is exact)
    const uint32_t idesc_s = mma_idesc_f16(G::BM, G::BN, BF16, false, false) |
                             (a.scale_log2 < 0.f ? kIdescNegateA : 0u);
    constexpr uint32_t idesc_o = mma_idesc_f16(G::BM, D, BF16, false, true);
    // This one thread issues every MMA of the CTA and is on the critical path,
    // so descriptors are built once here: the start-address field is the low
    // 14 bits of (address >> 4), so an offset of x bytes within shared memory
    // is added as x >> 4 without touching the other fields.
    const uint64_t dq = smem_desc(sbase + G::OFF_Q, 16, G::SBO, G::LAYOUT);    // Q, K-major
    const uint64_t dk = smem_desc(sbase + G::OFF_KV, 16, G::SBO, G::LAYOUT);   // K, K-major
    const uint64_t dv =
        smem_desc(sbase + G::OFF_KV, G::KV_PANEL_BYTES, G::SBO, G::LAYOUT);  // V, MN-major

    int it_u = 0;     // units processed by this CTA
    int kv_base = 0;  // K/V tiles consumed before the current unit
    int p_cnt[G::QT] = {};  // P phases consumed per query tile
    int o_cnt[G::QT] = {};  // units finished per query tile
    int fix_cnt = 0;        // paged V tiles handed over by the zeroing warps
    int p2_cnt = 0;         // P phases of odd key tiles in one-tile units
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x, ++it_u) {
        const Unit x = unit_of<SPLIT, PAGED>(u, nqb, nkv, a);
        const int qbuf = it_u % G::QBUF;
        if (!mbar_wait(bar(G::BAR_QF + qbuf), (it_u / G::QBUF) & 1, g, 4)) break;
        if constexpr (ONE) {
            // One live query tile: S of key tile j goes to the S columns of
            // tile (j & 1), so S_{j+1} is made while the softmax works on
            // S_j, and O (tile 0's) accumulates P_j V_j from either. S_{j+2}
            // is issued right after P_j V_j, which has read the columns it
            // overwrites (the tensor core runs a thread's MMAs in order).
            const uint32_t tO = tmem + G::TMEM_O_OFF;
            auto issue_s = [&](int j) {
                const int nk = 2 * (kv_base + j), ks = nk % G::SLOTS;
                if (!mbar_wait(bar(G::BAR_KVF + ks), (nk / G::SLOTS) & 1, g, 5)) return false;
                tc_fence_after();
                const uint32_t tS = tmem + (j & 1) * G::TMEM_TILE_STRIDE;
                const uint64_t qdesc = dq + ((qbuf * G::Q_BUF_BYTES) >> 4);
                const uint64_t kdesc = dk + ((ks * G::KV_TILE_BYTES) >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const int p = (kk * 16) / G::PANEL_ELEMS;
                    const int off = ((kk * 16) % G::PANEL_ELEMS) * 2;
                    mma_ss(tS, qdesc + ((p * G::Q_PANEL_BYTES + off) >> 4),
                           kdesc + ((p * G::KV_PANEL_BYTES + off) >> 4), idesc_s, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar((j & 1) ? G::BAR_SF2 : G::BAR_SF));
                mma_commit(bar(G::BAR_KVE + ks));                           // last read of K_j
                if (j == x.nkv - 1) mma_commit(bar(G::BAR_QE + qbuf));     // ... and of this Q
                return true;
            };
            if (x.nkv > 0) ok = issue_s(0);
            if (ok && x.nkv > 1) ok = issue_s(1);
            for (int j = 0; ok && j < x.nkv; ++j) {
                const int nv = 2 * (kv_base + j) + 1, vs = nv % G::SLOTS;
                if (!mbar_wait(bar(G::BAR_KVF + vs), (nv / G::SLOTS) & 1, g, 6)) {
                    ok = false;
                    break;
                }
                if (j == x.nkv - 1 && unit_needs_v_fix<PAGED>(x)) {
                    // a paged unit's last V tile has landed; wait for its
                    // stale rows to be zeroed
                    mbar_arrive(bar(G::BAR_VLAND));
                    if (!mbar_wait(bar(G::BAR_VFIX), fix_cnt & 1, g, 11)) {
                        ok = false;
                        break;
                    }
                    ++fix_cnt;
                }
                // the first P V overwrites O: the previous unit's epilogue
                // must have read it out
                if (j == 0 && !mbar_wait(bar(G::BAR_OE), (o_cnt[0] & 1) ^ 1, g, 7)) {
                    ok = false;
                    break;
                }
                const bool odd = j & 1;
                if (!mbar_wait(bar(odd ? G::BAR_PF2 : G::BAR_PF), (odd ? p2_cnt : p_cnt[0]) & 1, g,
                               8)) {
                    ok = false;
                    break;
                }
                if (odd)
                    ++p2_cnt;
                else
                    ++p_cnt[0];
                tc_fence_after();
                const uint32_t tP = tmem + (j & 1) * G::TMEM_TILE_STRIDE;
                const uint64_t vdesc = dv + ((vs * G::KV_TILE_BYTES) >> 4);
#pragma unroll
                for (int kk = 0; kk < G::BN / 16; ++kk)
                    mma_ts(tO, tP + kk * 8, vdesc + ((kk * 16 * G::ROW_BYTES) >> 4), idesc_o,
                           (j > 0 || kk > 0) ? 1u : 0u);
                mma_commit(bar(G::BAR_KVE + vs));  // last read of V_j
                mma_commit(bar(G::BAR_PVD));
                if (j == x.nkv - 1) mma_commit(bar(G::BAR_OF));
                if (j + 2 < x.nkv) ok = issue_s(j + 2);
            }
            if (!ok) break;
            if (x.nkv == 0) {  // causal: a unit that sees no key
                mma_commit(bar(G::BAR_QE + qbuf));
                mma_commit(bar(G::BAR_OF));
            }
            kv_base += x.nkv;
            ++o_cnt[0];
            continue;
        }
        // The issue order keeps the tensor core's short instruction queue fed:
        // every barrier wait or commit sits right after a group of MMAs, while
        // those are still queued, never in a clump between two groups.
        for (int j = 0; ok && j <= x.nkv; ++j) {
            // ring items: K_j is item 2 (kv_base + j), V_{j-1} the item before it
            const int nk = 2 * (kv_base + j), nv = nk - 1;
            const int ks = nk % G::SLOTS, vs = nv % G::SLOTS;
            // a paged unit's last V tile, once its stale rows are zeroed
            if (j == x.nkv && unit_needs_v_fix<PAGED>(x)) {
                if (!mbar_wait(bar(G::BAR_VFIX), fix_cnt & 1, g, 11)) {
                    ok = false;
                    break;
                }
                ++fix_cnt;
            }
            for (int t = 0; t < x.n_qt; ++t) {
                const uint32_t tS = tmem + t * G::TMEM_TILE_STRIDE;
                const uint32_t tO = tS + G::TMEM_O_OFF;
                if (j > 0) {
                    // The first P V of a unit overwrites O_t: the previous unit's
                    // epilogue must have read it out.
                    if (j == 1 && !mbar_wait(bar(G::BAR_OE + t), (o_cnt[t] & 1) ^ 1, g, 7)) {
                        ok = false;
                        break;
                    }
                    // O_t += P_{j-1}(t) V_{j-1}; P sits in the S columns, 16 keys
                    // per 8 columns. V_{j-1} was waited for at the end of step j-1.
                    if (!mbar_wait(bar(G::BAR_PF + t), p_cnt[t] & 1, g, 8)) {
                        ok = false;
                        break;
                    }
                    ++p_cnt[t];
                    tc_fence_after();
                    const uint64_t vdesc = dv + ((vs * G::KV_TILE_BYTES) >> 4);
#pragma unroll
                    for (int kk = 0; kk < G::BN / 16; ++kk)
                        mma_ts(tO, tS + kk * 8, vdesc + ((kk * 16 * G::ROW_BYTES) >> 4), idesc_o,
                               (j > 1 || kk > 0) ? 1u : 0u);
                    if (t == x.n_qt - 1) mma_commit(bar(G::BAR_KVE + vs));  // last read of V_{j-1}
                }
                if (j < x.nkv) {
                    if (t == 0 &&
                        !mbar_wait(bar(G::BAR_KVF + ks), (nk / G::SLOTS) & 1, g, 5)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // S_j(t) = Q_t K_j^T, 16 head-dim elements per instruction.
                    const uint64_t qdesc = dq + ((qbuf * G::Q_BUF_BYTES + t * G::Q_TILE_BYTES) >> 4);
                    const uint64_t kdesc = dk + ((ks * G::KV_TILE_BYTES) >> 4);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const int p = (kk * 16) / G::PANEL_ELEMS;
                        const int off = ((kk * 16) % G::PANEL_ELEMS) * 2;
                        mma_ss(tS, qdesc + ((p * G::Q_PANEL_BYTES + off) >> 4),
                               kdesc + ((p * G::KV_PANEL_BYTES + off) >> 4), idesc_s,
                               kk > 0 ? 1u : 0u);
                    }
                    mma_commit(bar(G::BAR_SF + t));
                    if (t == x.n_qt - 1) {
                        mma_commit(bar(G::BAR_KVE + ks));                  // last read of K_j
                        if (j == x.nkv - 1) mma_commit(bar(G::BAR_QE + qbuf));  // ... and of this Q
                    }
                } else {
                    mma_commit(bar(G::BAR_OF + t));
                }
            }
            if (!ok) break;
            // V_j for the next step, waited for while the S MMAs above are queued
            if (j < x.nkv &&
                !mbar_wait(bar(G::BAR_KVF + (nk + 1) % G::SLOTS), ((nk + 1) / G::SLOTS) & 1, g, 6)) {
                ok = false;
                break;
            }
            // a paged unit's last V tile has landed: the zeroing warps may go
            if (j == x.nkv - 1 && unit_needs_v_fix<PAGED>(x)) mbar_arrive(bar(G::BAR_VLAND));
        }
        // a unit with no key tile (causal) still frees its Q buffer
        if constexpr (SPLIT)
            if (x.nkv == 0) mma_commit(bar(G::BAR_QE + qbuf));
        kv_base += x.nkv;
        for (int t = 0; t < x.n_qt; ++t) ++o_cnt[t];
    }
    // No MMA may still be running when TMEM is released.
    mma_commit(bar(G::BAR_DONE));
    WaitGuard drain = g;
    uint32_t no_abort = 0;
    drain.abort = &no_abort;
    mbar_wait(bar(G::BAR_DONE), 0, drain, 12);
}

template <int D, bool BF16, int SPLIT, bool PAGED, bool ONE>
__device__ __forceinline__ void fwd_softmax(uint32_t sbase, uint32_t tmem, int t, int q4, int nqb,
                                            int units, int nkv, const FwdArgs &a,
                                            const WaitGuard &g) {
    using G = FwdGeom<D>;
    auto bar = [&](int i) { return sbase + G::OFF_BAR + 8u * i; };
    const uint32_t lane = threadIdx.x & 31;
    const int row = q4 * 32 + lane;
    const uint32_t tS0 = tmem + t * G::TMEM_TILE_STRIDE + (static_cast<uint32_t>(q4 * 32) << 16);
    const uint32_t tO = tS0 + G::TMEM_O_OFF;
    // S arrives as sign(scale) * QK^T (the S MMAs negate Q for a negative
    // scale): with c = |scale| log2 e, the row max of the raw scores is the
    // max of the scaled ones
    const float c = fabsf(a.scale_log2);
    int s_cnt = 0, o_cnt = 0;
    // one-tile units (tile 0's warpgroup only): S phases of odd key tiles,
    // and P V products issued so far
    int s2_cnt = 0, pv_done = 0;

    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const Unit x = unit_of<SPLIT, PAGED>(u, nqb, nkv, a);
        if (t >= x.n_qt) continue;
        constexpr bool single = ONE;
        const int tile_row0 = x.m0 + t * G::BM;
        const int grow = tile_row0 + row;
        // A warp whose 32 rows all lie past sq skips the math but keeps the
        // barrier protocol.
        const bool warp_live = tile_row0 + q4 * 32 < a.sq;

        float m_ref = -INFINITY;  // reference max, log2 units
        float l = 0.f;            // running sum of 2^(s*c - m_ref)
        bool alive = true;
        for (int j = 0; j < x.nkv; ++j) {
            // S_j: in one-tile units odd key tiles use the second tile's S
            // columns and barriers
            const bool alt = single && (j & 1);
            const uint32_t tS = alt ? tS0 + G::TMEM_TILE_STRIDE : tS0;
            const bool ok = mbar_wait(bar(alt ? G::BAR_SF2 : G::BAR_SF + t),
                                      (alt ? s2_cnt : s_cnt) & 1, g, 13);
            if (alt)
                ++s2_cnt;
            else
                ++s_cnt;
            if (!__all_sync(0xffffffffu, ok)) {
                alive = false;
                break;
            }
            tc_fence_after();
            if (warp_live) {
                // keys of this tile the row may use: inside [0, sk) and, with the
                // causal mask, at most grow + sk - sq. Loads and chunk skips
                // follow the warp's largest count (tcgen05.ld is warp-wide).
                int valid = x.sk - (x.kv0 + j) * G::BN;
                int vmax = valid;
                bool ragged = valid < G::BN;
                if constexpr (SPLIT != 0) {
                    if (SPLIT == 1 || a.causal) {
                        valid = min(valid, grow + x.sk - a.sq + 1 - (x.kv0 + j) * G::BN);
                        vmax = __reduce_max_sync(0xffffffffu, valid);
                        ragged = __any_sync(0xffffffffu, valid < G::BN);
                    }
                }
                uint32_t sr[G::BN];
                const float *s = reinterpret_cast<const float *>(sr);
                // row max of the scores
                float mx[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) mx[i] = -INFINITY;
                if (!ragged) {
                    // the max of the first 64 scores runs while the rest load
                    tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
                    tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
                    tmem_wait_ld();
                    tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
                    tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
                        if (part == 1) tmem_wait_ld();
#pragma unroll
                        for (int i = part * G::BN / 4; i < (part + 1) * G::BN / 4; ++i)
                            mx[i & 3] = max3f(mx[i & 3], s[2 * i], s[2 * i + 1]);
                    }
                } else {
#pragma unroll
                    for (int c0 = 0; c0 < G::BN; c0 += 32) {
                        if (c0 < vmax)
                            tmem_ld32(tS + c0, *reinterpret_cast<uint32_t(*)[32]>(&sr[c0]));
                    }
                    tmem_wait_ld();
                    // whole 32-key chunks past sk are skipped (a warp-uniform branch)
#pragma unroll
                    for (int c0 = 0; c0 < G::BN; c0 += 32) {
                        if (c0 < vmax) {
#pragma unroll
                            for (int i = c0; i < c0 + 32; ++i) {
                                if (i < valid) mx[i & 3] = fmaxf(mx[i & 3], s[i]);
                            }
                        }
                    }
                }
                const float mraw = fmaxf(max3f(mx[0], mx[1], mx[2]), mx[3]);
                const float m_tile = mraw * c;

                const bool need = m_tile > m_ref + 8.0f;
                const float m_new = need ? m_tile : m_ref;
                // 1 if kept, 0 on the first tile; a row that has seen no key yet
                // (causal) keeps m = -inf and alpha 1
                const float alpha =
                    (SPLIT && m_new == -INFINITY) ? 1.0f : fast_exp2(m_ref - m_new);
                m_ref = m_new;

                // O must be rescaled (rare once the running max settles) before
                // the MMA issuer accumulates P_j V_j into it. The rescale runs
                // after P is stored, when the scores are no longer held in
                // registers, and before P is handed over.
                const bool rescale = j > 0 && __any_sync(0xffffffffu, need);

                // P = 2^(s*c - m_ref), packed in pairs into the S columns, 64 keys
                // at a time; keys past sk get exactly 0 (their V rows are TMA
                // zero fill).
                const float neg_m = -m_ref;
                const uint64_t c2 = f2_make(c, c), nm2 = f2_make(neg_m, neg_m);
                uint64_t acc2[2] = {0ull, 0ull};  // packed partial row sums (0.0f bits)
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t pk[G::BN / 4];
                    if (!ragged) {
#pragma unroll
                        for (int i = 0; i < G::BN / 4; ++i) {
                            const int k0 = half * (G::BN / 2) + 2 * i;
                            float x0, x1;
                            // x = s * c - m for two keys in one packed FMA
                            f2_split(f2_fma(f2_make(s[k0], s[k0 + 1]), c2, nm2), x0, x1);
                            const float p0 = fast_exp2(x0);
                            const float p1 = fast_exp2(x1);
                            acc2[i & 1] = f2_add(acc2[i & 1], f2_make(p0, p1));
                            pk[i] = pack2<BF16>(p0, p1);
                        }
                    } else {
                        // last key tile: keys past sk are masked to exactly 0; whole
                        // 32-key chunks past sk are zero without exponentiating (a
                        // warp-uniform branch)
#pragma unroll
                        for (int ch = 0; ch < 2; ++ch) {
                            if (half * (G::BN / 2) + ch * 32 < vmax) {
#pragma unroll
                                for (int i = ch * 16; i < ch * 16 + 16; ++i) {
                                    const int k0 = half * (G::BN / 2) + 2 * i;
                                    float x0, x1;
                                    f2_split(f2_fma(f2_make(s[k0], s[k0 + 1]), c2, nm2), x0, x1);
                                    x0 = (k0 < valid) ? x0 : -INFINITY;
                                    x1 = (k0 + 1 < valid) ? x1 : -INFINITY;
                                    const float p0 = fast_exp2(x0);
                                    const float p1 = fast_exp2(x1);
                                    acc2[i & 1] = f2_add(acc2[i & 1], f2_make(p0, p1));
                                    pk[i] = pack2<BF16>(p0, p1);
                                }
                            } else {
#pragma unroll
                                for (int i = ch * 16; i < ch * 16 + 16; ++i) pk[i] = 0u;
                            }
                        }
                    }
                    tmem_st32(tS + half * (G::BN / 4), pk);
                }
                if (rescale) {
                    // O row *= alpha once P_{j-1} V_{j-1} has completed: S_j's
                    // commit covers it where S_j was issued after it; a one-tile
                    // unit issues S_j earlier and waits for that P V's own
                    // barrier (at most one phase ahead of this wait: the next
                    // P V needs this P_j). 16 columns at a time keeps this path
                    // spill-free.
                    if (single) {
                        const bool okv = mbar_wait(bar(G::BAR_PVD), (pv_done + j - 1) & 1, g, 15);
                        if (!__all_sync(0xffffffffu, okv)) {
                            alive = false;
                            break;
                        }
                        tc_fence_after();
                    }
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += 16) {
                        uint32_t ov[16];
                        tmem_ld16(tO + c0, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                        tmem_st16(tO + c0, ov);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(alt ? G::BAR_PF2 : G::BAR_PF + t));
                float a0, a1, a2, a3;
                f2_split(acc2[0], a0, a1);
                f2_split(acc2[1], a2, a3);
                l = l * alpha + ((a0 + a1) + (a2 + a3));
            } else {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(alt ? G::BAR_PF2 : G::BAR_PF + t));
            }
        }
        if (!alive) return;
        if (single) pv_done += x.nkv;

        // ---------------------------------------------------- epilogue
        // Read O_t a chunk at a time, normalise, and store: packed to 16 bits
        // into O, or as fp32 into this split's O_i; then hand the accumulator
        // back to the MMA issuer. The epilogue sits between this unit's last
        // P and the next unit's first softmax on these warps, so what needs
        // no O (1 / l, the addresses) is worked out before the wait for it.
        // A row that saw no key (causal) has l = 0: O = 0, LSE = -inf.
        const bool empty_row = SPLIT && !(l > 0.0f);
        const float inv_l = empty_row ? 0.0f : 1.0f / l;
        const bool row_out = warp_live && grow < a.sq;
        // fp32 partials only with more than one split (key ranges with one
        // split, paged or several-row decode calls, write O and LSE)
        const bool part = SPLIT == 2 && a.splits > 1;
        // Rows start at multiples of 2d bytes (>= 32); only the base of O may
        // be merely 16-byte aligned. The fp32 partials are allocated here.
        const bool o_al32 = (reinterpret_cast<uintptr_t>(a.o) & 31u) == 0;
        const int64_t orow =
            ((static_cast<int64_t>(part ? x.split * a.b + x.batch : x.batch) * a.sq +
              (row_out ? grow : 0)) * a.h + x.head) * D;
        uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(a.o) + orow);
        float *dst_part = a.o_part + orow;
        const bool ok = mbar_wait(bar(G::BAR_OF + t), o_cnt & 1, g, 14);
        ++o_cnt;
        if (!__all_sync(0xffffffffu, ok)) return;
        tc_fence_after();
        if (warp_live) {
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += G::OCH) {
                uint32_t ov[G::OCH];
                if constexpr (G::OCH == 32)
                    tmem_ld32(tO + c0, *reinterpret_cast<uint32_t(*)[32]>(ov));
                else
                    tmem_ld16(tO + c0, *reinterpret_cast<uint32_t(*)[16]>(ov));
                tmem_wait_ld();
                if (part && row_out) {
#pragma unroll
                    for (int i = 0; i < G::OCH; ++i)
                        ov[i] = empty_row ? 0u : __float_as_uint(__uint_as_float(ov[i]) * inv_l);
#pragma unroll
                    for (int i = 0; i < G::OCH / 8; ++i)
                        st_global_v8(dst_part + c0 + 8 * i,
                                     *reinterpret_cast<const uint32_t(*)[8]>(&ov[8 * i]));
                } else if (row_out) {
                    uint32_t pk[G::OCH / 2];
#pragma unroll
                    for (int i = 0; i < G::OCH / 2; ++i)
                        pk[i] = empty_row ? 0u
                                          : pack2<BF16>(__uint_as_float(ov[2 * i]) * inv_l,
                                                        __uint_as_float(ov[2 * i + 1]) * inv_l);
                    if (o_al32) {
                        // whole 32-byte sectors: 16 columns per store
#pragma unroll
                        for (int i = 0; i < G::OCH / 16; ++i)
                            st_global_v8(dst + c0 / 8 + 2 * i,
                                         *reinterpret_cast<const uint32_t(*)[8]>(&pk[8 * i]));
                    } else {
#pragma unroll
                        for (int i = 0; i < G::OCH / 8; ++i)
                            dst[c0 / 8 + i] =
                                make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                    }
                }
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(G::BAR_OE + t));
        if (row_out) {
            const float lse =
                empty_row ? -INFINITY : (m_ref + __log2f(l)) * 0.69314718055994530942f;
            if (part)
                a.lse_part[((static_cast<int64_t>(x.split) * a.b + x.batch) * a.h + x.head) * a.sq +
                           grow] = lse;
            else
                a.lse[(static_cast<int64_t>(x.batch) * a.h + x.head) * a.sq + grow] = lse;
        }
    }
}

template <int D, bool BF16, int SPLIT, bool PAGED, bool ONE>
__global__ void __launch_bounds__(FWD_THREADS, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, const FwdArgs a) {
    using G = FwdGeom<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw);
    auto bar = [&](int i) { return sbase + G::OFF_BAR + 8u * i; };

    const int warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    const int nqb = (a.sq + G::BM * G::QT - 1) / (G::BM * G::QT);
    const int units = nqb * a.splits * a.h * a.b;
    const int nkv = (a.sk + G::BN - 1) / G::BN;  // key tiles in all

    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + G::OFF_MISC);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + G::OFF_MISC + 4);

    if (threadIdx.x == 0) {
        for (int i = 0; i < G::NUM_BARS; ++i) {
            uint32_t count = 1;
            // one arrive per softmax warp
            if ((i >= G::BAR_PF && i < G::BAR_PF + G::QT) ||
                (i >= G::BAR_OE && i < G::BAR_OE + G::QT))
                count = 4;
            if (i == G::BAR_VFIX) count = 2;  // one arrive per zeroing warp
            mbar_init(bar(i), count);
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
        tmem_alloc(smem_u32(tmem_slot), G::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitGuard g{abort_flag, a.status, kKernFwd};

    if (warp < 4) {
        reg_dealloc<kRegsControl>();
        if (warp == 0) {
            if constexpr (PAGED) {
                if (!(a.flags & kFlagSkipLoads))
                    fwd_producer_paged<D, SPLIT, PAGED>(&tq, &tk, &tv, sbase, nqb, units, nkv, a, g);
            } else {
                if (lane == 0 && !(a.flags & kFlagSkipLoads))
                    fwd_producer<D, SPLIT, PAGED>(&tq, &tk, &tv, sbase, nqb, units, nkv, a, g);
            }
        } else if (warp == 1) {
            if (lane == 0) fwd_mma<D, BF16, SPLIT, PAGED, ONE>(sbase, tmem, nqb, units, nkv, a, g);
        } else if (PAGED && !(a.flags & kFlagSkipLoads)) {
            fwd_fix_v<D, SPLIT, PAGED>(sbase, nqb, units, nkv, a, g);
        }
    } else {
        reg_alloc<kRegsSoftmax>();
        fwd_softmax<D, BF16, SPLIT, PAGED, ONE>(sbase, tmem, (warp - 4) >> 2, warp & 3, nqb, units,
                                                nkv, a, g);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, G::TMEM_COLS);
}

template <int D, bool BF16, int SPLIT, bool PAGED, bool ONE>
cudaError_t launch_fwd_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                         const FwdArgs &a, cudaStream_t stream) {
    using G = FwdGeom<D>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_set[dev]) {
        e = cudaFuncSetAttribute(fwd_kernel<D, BF16, SPLIT, PAGED, ONE>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const int64_t nqb = (a.sq + G::BM * G::QT - 1) / (G::BM * G::QT);
    const int64_t units = nqb * a.splits * a.h * a.b;
    // Units of equal length: as few CTAs as the number of waves needs (256
    // units on 152 SMs: 128 CTAs of two units, not 104 of two and 48 of one),
    // so fewer of them compete for DRAM while all start at once (b4 s512 h32:
    // +1-2%). Causal units differ in length and are dealt longest first over
    // one CTA per SM (b2 s4096 h16 was 7% slower on the smaller grid).
    const int64_t waves = (units + a.num_sms - 1) / a.num_sms;
    const int64_t ctas =
        a.causal ? (units < a.num_sms ? units : a.num_sms) : (units + waves - 1) / waves;
    fwd_kernel<D, BF16, SPLIT, PAGED, ONE>
        <<<static_cast<unsigned>(ctas), FWD_THREADS, G::SMEM_BYTES, stream>>>(tq, tk, tv, a);
    return cudaGetLastError();
}

// At most 128 query rows against more than one key tile: every unit has one
// live query tile, and the kernel compiled for that case (double-buffered S)
// runs (b1 h16 sk32768 with 10 rows: 55.6 -> 49.7 us; b8 h48 sk8192: 285 ->
// 241 us). With a single key tile there is nothing to overlap (b64 s100 h16:
// 32.8 -> 33.9 us), so the two-tile kernel keeps those. The two paths are
// separate kernels: compiled into one, the two-tile calls lost about 6 us
// per launch (b4 s512 h32: 26.6 -> 32.8 us) though they never ran the other.
template <int D, bool BF16, int SPLIT, bool PAGED>
cudaError_t launch_fwd_o(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                         const FwdArgs &a, cudaStream_t stream) {
    return a.sq <= FWD_BM && a.sk > FWD_BN
               ? launch_fwd_t<D, BF16, SPLIT, PAGED, true>(tq, tk, tv, a, stream)
               : launch_fwd_t<D, BF16, SPLIT, PAGED, false>(tq, tk, tv, a, stream);
}

template <int D, bool BF16>
cudaError_t launch_fwd_d(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                         const FwdArgs &a, cudaStream_t stream) {
    // four instantiations: the plain forward, the causal forward (one key
    // range, no partials), key ranges (with or without the mask), and key
    // ranges over a paged cache; each keeps only the code it needs (the
    // causal forward on the key-range kernel: b8 s256 h32 d128 26.6 against
    // 24.6 us, b2 s1024 h48 47.4 against 45.0)
    if (a.block_table) return launch_fwd_o<D, BF16, 2, true>(tq, tk, tv, a, stream);
    if (a.splits > 1) return launch_fwd_o<D, BF16, 2, false>(tq, tk, tv, a, stream);
    return a.causal ? launch_fwd_o<D, BF16, 1, false>(tq, tk, tv, a, stream)
                    : launch_fwd_o<D, BF16, 0, false>(tq, tk, tv, a, stream);
}

}  // namespace

cudaError_t launch_fwd(int d, bool bf16, const CUtensorMap &tq, const CUtensorMap &tk,
                       const CUtensorMap &tv, const FwdArgs &a, cudaStream_t stream) {
#define EXATTN_FWD_CASE(DD)                                               \
    case DD:                                                              \
        return bf16 ? launch_fwd_d<DD, true>(tq, tk, tv, a, stream)       \
                    : launch_fwd_d<DD, false>(tq, tk, tv, a, stream);
    switch (d) {
        EXATTN_FWD_CASE(16)
        EXATTN_FWD_CASE(32)
        EXATTN_FWD_CASE(64)
        EXATTN_FWD_CASE(128)
        default:
            return cudaErrorInvalidValue;
    }
#undef EXATTN_FWD_CASE
}

}  // namespace exattn
