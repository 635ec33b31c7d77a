// Backward of exact attention for short sequences and small heads: the
// shapes of the flash-attn timing issue ("2.6.3 is faster than 2.7.0 for
// flash-attn v2 CUDA fwd/bwd": head dim 16, sequences of 50 to 300), where
// the tile kernels of bwd.cu spend most of their time on padding (a 150-key
// problem is two 128-key tiles, one holding 22 keys) and on per-unit set-up.
//
// What is computed is the chain rule of the forward's definition, as in
// bwd.cu: with S = scale Q K^T, P = exp(S - LSE) (the forward's LSE), and
// D = rowsum(dO * O) (bwd_dot_kernel),
//     dV = P^T dO,   dP = dO V^T,   dS = P * (dP - D),
//     dQ = scale dS K,   dK = scale dS^T Q.
//
// A work item is one (batch, head) with all of its keys (at most 160) in one
// row of S, and its query rows in one or two 128-row tiles. Per query tile:
//   S = Q_t K^T and dP = dO_t V^T into TMEM (one MMA each per 16 of d);
//   the elementwise warps (one query row per TMEM lane) make P and dS; dS goes
//   back into S's columns (16-bit, the A operand of dQ = dS K, from TMEM),
//   and P and dS go to shared memory as rows of keys: read as MN-major A
//   operands they are P^T and dS^T, so dV += P^T dO_t and dK += dS^T Q_t
//   accumulate in TMEM over the item's query tiles (one 128-key M tile per
//   128 keys);
//   dQ of the tile is complete at once (all keys in one row) and is written
//   out; dK and dV are written after the item's last tile. No atomics, no
//   second pass.
//
// Persistent CTAs (one per SM) take items round-robin:
//   warp 0        TMA producer (lane 0): Q, dO, K, V of an item into a stage
//                 (two stages at d = 16, one at d = 32); then the whole warp
//                 stages the item's LSE and D rows in shared memory ahead of
//                 their use (the elementwise warps would otherwise start
//                 each item with a global load of them).
//   warp 1        TMEM owner; issues S, dP and dQ MMAs (one thread).
//   warp 2        issues the dK MMAs (one thread).
//   warp 3        issues the dV MMAs (one thread): a tile's dQ, dK and dV
//                 and the next tile's S and dP go out side by side rather
//                 than one after another.
//   warps 4-11    elementwise: group g (warps 4 + 4g .. 7 + 4g) holds all
//                 128 lanes and takes the 16-key chunks c with c % 2 == g;
//                 group g also writes dK and dV of key M tile g.
// TMEM columns: S [0, N), dP [N, 2N) (N = sk rounded up to 32), dQ, then
// dV and dK of each key M tile, each region 32 columns wide.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace exattn {
namespace {

constexpr int SB_THREADS = 384;
constexpr int SB_EW_WARPS = 8;
constexpr int SB_QT = 128;                        // rows of a query tile (TMEM lanes)
constexpr int SB_PANEL_BYTES = SB_QT * 128;       // 64 keys of 128 query rows, 16-bit
constexpr int SB_PDS_BYTES = 4 * SB_PANEL_BYTES;  // keys 0..255: an M tile reads two whole panels
constexpr int SB_MAX_N = 160;                     // TMEM: 2 N + 32 (dQ) + 2 x 2 x 32 (dV, dK)
constexpr int SB_COL_W = 32;                      // columns of a dQ / dV / dK region
static_assert(2 * SB_MAX_N + SB_COL_W + 2 * 2 * SB_COL_W <= 512, "TMEM columns of the widest item");

template <int D>
struct SbGeom {
    static_assert(D == 16 || D == 32, "head dim");
    static constexpr int RB = D * 2;  // bytes of one row: one swizzle atom wide
    static constexpr uint32_t LAYOUT = RB == 64 ? kLayoutSw64 : kLayoutSw32;
    static constexpr uint32_t SBO = 8 * RB;
    static constexpr int TQ_BYTES = SBWD_MAX_Q * RB;  // Q or dO of an item
    static constexpr int TK_BYTES = SBWD_MAX_K * RB;  // K or V
    static constexpr int STAGE_BYTES = 2 * TQ_BYTES + 2 * TK_BYTES;  // Q | dO | K | V
    static constexpr int STAGES = D == 16 ? 2 : 1;
    static constexpr int OFF_P = STAGES * STAGE_BYTES;
    static constexpr int OFF_DS = OFF_P + SB_PDS_BYTES;
    // per stage: the item's LSE (log2 units) and D, SBWD_MAX_Q floats each
    static constexpr int OFF_LD = OFF_DS + SB_PDS_BYTES;
    static constexpr int OFF_BAR = OFF_LD + STAGES * 2 * SBWD_MAX_Q * 4;
    static constexpr int BAR_INF = 0;              // [2] an item's inputs landed
    static constexpr int BAR_INE = BAR_INF + 2;    // [2] its last MMAs (all 3 issuers) read them
    static constexpr int BAR_SF = BAR_INE + 2;     // a tile's S and dP in TMEM
    static constexpr int BAR_PF = BAR_SF + 1;      // its P and dS written (8 warps)
    static constexpr int BAR_PFREE = BAR_PF + 1;   // its dV and dK MMAs have read them (2)
    static constexpr int BAR_QF = BAR_PFREE + 1;   // its dQ in TMEM
    static constexpr int BAR_QE = BAR_QF + 1;      // dQ read out (8 warps)
    static constexpr int BAR_KVF = BAR_QE + 1;     // the item's dK and dV in TMEM (2)
    static constexpr int BAR_KVE = BAR_KVF + 1;    // read out (8 warps)
    static constexpr int BAR_LDF = BAR_KVE + 1;    // [2] an item's LSE and D staged (warp 0)
    static constexpr int BAR_DONE = BAR_LDF + 2;   // [3] each issuer's MMAs complete
    static constexpr int NUM_BARS = BAR_DONE + 3;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
    static_assert(OFF_P % 1024 == 0, "P and dS panels on swizzle-atom boundaries");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

// Per-call layout, the same in every thread.
struct SbPlan {
    int n;      // key columns of S: sk rounded up to 32
    int nmk;    // 128-key M tiles of dK / dV
    int nqt;    // 128-row query tiles
    int c_dp, c_dq, c_dv, c_dk;  // TMEM columns
};

__device__ __forceinline__ SbPlan sb_plan(const BwdArgs &a) {
    SbPlan p;
    p.n = (a.sk + 31) / 32 * 32;
    p.nmk = p.n > 128 ? 2 : 1;
    p.nqt = (a.sq + SB_QT - 1) / SB_QT;
    p.c_dp = p.n;
    p.c_dq = 2 * p.n;
    p.c_dv = p.c_dq + SB_COL_W;
    p.c_dk = p.c_dv + p.nmk * SB_COL_W;
    return p;
}

template <bool BF16>
__device__ __forceinline__ uint32_t sb_pack(float lo, float hi) {
    if constexpr (BF16)
        return cvt_pack_bf16(lo, hi);
    else
        return cvt_pack_f16(lo, hi);
}

// Warp 0. Lane 0 waits for an item's stage and loads its Q, dO, K and V;
// then the warp writes LSE * log2(e) and D of every query row of the item
// into the stage (rows past sq get LSE = +inf, hence P = 0, and D = 0).
template <int D>
__device__ __forceinline__ void sb_producer(const CUtensorMap *tq, const CUtensorMap *tk,
                                            const CUtensorMap *tv, const CUtensorMap *tdo,
                                            uint8_t *smem, uint32_t sbase, int items,
                                            const SbPlan &p, const BwdArgs &a,
                                            const WaitGuard &g) {
    using G = SbGeom<D>;
    auto bar = [&](int i) { return sbase + G::OFF_BAR + 8u * i; };
    constexpr float kLog2e = 1.4426950408889634f;
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t bytes = 2u * (p.nqt * SB_QT) * G::RB + 2u * p.n * G::RB;
    const int rows = p.nqt * SB_QT;
    int n = 0;
    for (int it = blockIdx.x; it < items; it += gridDim.x, ++n) {
        const int head = it % a.h, batch = it / a.h;
        const int st = n % G::STAGES;
        bool ok = true;
        if (lane == 0) {
            ok = mbar_wait(bar(G::BAR_INE + st), ((n / G::STAGES) & 1) ^ 1, g, 40);
            if (ok) {
                mbar_arrive_expect_tx(bar(G::BAR_INF + st), bytes);
                const uint32_t dst = sbase + st * G::STAGE_BYTES;
                tma_load_4d(dst, tq, bar(G::BAR_INF + st), 0, head, 0, batch);
                tma_load_4d(dst + G::TQ_BYTES, tdo, bar(G::BAR_INF + st), 0, head, 0, batch);
                tma_load_4d(dst + 2 * G::TQ_BYTES, tk, bar(G::BAR_INF + st), 0, head, 0, batch);
                tma_load_4d(dst + 2 * G::TQ_BYTES + G::TK_BYTES, tv, bar(G::BAR_INF + st), 0,
                            head, 0, batch);
            }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        const int64_t base = static_cast<int64_t>(it) * a.sq;  // (batch, head) = it
        float *ld = reinterpret_cast<float *>(smem + G::OFF_LD) + st * 2 * SBWD_MAX_Q;
        for (int r = lane; r < rows; r += 32) {
            const bool v = r < a.sq;
            ld[r] = v ? a.lse[base + r] * kLog2e : INFINITY;
            ld[SBWD_MAX_Q + r] = v ? a.dvec[base + r] : 0.f;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(G::BAR_LDF + st));
    }
    // never leave the CTA with a copy still landing in shared memory
    if (lane == 0) {
        WaitGuard drain = g;
        uint32_t no_abort = 0;
        drain.abort = &no_abort;
        for (int m = (n > G::STAGES ? n - G::STAGES : 0); m < n; ++m)
            mbar_wait(bar(G::BAR_INF + m % G::STAGES), (m / G::STAGES) & 1, drain, 41);
    }
}

// dQ = dS K over STEPS steps of 16 keys, one straight-line run of MMAs: A is
// dS in S's columns (keys 16 kk .. 16 kk + 15 packed into the first 8 of
// their 16 columns), B is K MN-major.
template <int D, int STEPS>
__device__ __forceinline__ void sb_issue_dq(uint32_t t_dq, uint32_t t_s, uint64_t kmn,
                                            uint32_t idesc) {
#pragma unroll
    for (int kk = 0; kk < STEPS; ++kk)
        mma_ts(t_dq, t_s + kk * 16, kmn + ((kk * 16 * SbGeom<D>::RB) >> 4), idesc,
               kk > 0 ? 1u : 0u);
}

template <int D>
__device__ __forceinline__ void sb_issue_dq_n(int steps, uint32_t t_dq, uint32_t t_s,
                                              uint64_t kmn, uint32_t idesc) {
    switch (steps) {  // keys rounded up to 32: 2, 4, ..., 10 steps
        case 2: sb_issue_dq<D, 2>(t_dq, t_s, kmn, idesc); break;
        case 4: sb_issue_dq<D, 4>(t_dq, t_s, kmn, idesc); break;
        case 6: sb_issue_dq<D, 6>(t_dq, t_s, kmn, idesc); break;
        case 8: sb_issue_dq<D, 8>(t_dq, t_s, kmn, idesc); break;
        default: sb_issue_dq<D, 10>(t_dq, t_s, kmn, idesc); break;
    }
}

// dV += P^T dO_t (or dK += dS^T Q_t) for key M tile mt over the tile's
// first 16 STEPS query rows (rows past sq hold P = dS = 0 and are skipped),
// one straight-line run; acc0 = 0 overwrites (the item's first tile). a is
// the P (or dS) panel pair of the M tile, b dO_t (or Q_t).
template <int D, int STEPS>
__device__ __forceinline__ void sb_issue_kv(uint32_t t_acc, uint64_t a, uint64_t b, uint32_t idesc,
                                            uint32_t acc0) {
#pragma unroll
    for (int kk = 0; kk < STEPS; ++kk)
        mma_ss(t_acc, a + ((kk * 2048) >> 4), b + ((kk * 16 * SbGeom<D>::RB) >> 4), idesc,
               (acc0 || kk > 0) ? 1u : 0u);
}

template <int D>
__device__ __forceinline__ void sb_issue_kv_n(int steps, uint32_t t_acc, uint64_t a, uint64_t b,
                                              uint32_t idesc, uint32_t acc0) {
    switch (steps) {
        case 1: sb_issue_kv<D, 1>(t_acc, a, b, idesc, acc0); break;
        case 2: sb_issue_kv<D, 2>(t_acc, a, b, idesc, acc0); break;
        case 3: sb_issue_kv<D, 3>(t_acc, a, b, idesc, acc0); break;
        case 4: sb_issue_kv<D, 4>(t_acc, a, b, idesc, acc0); break;
        case 5: sb_issue_kv<D, 5>(t_acc, a, b, idesc, acc0); break;
        case 6: sb_issue_kv<D, 6>(t_acc, a, b, idesc, acc0); break;
        case 7: sb_issue_kv<D, 7>(t_acc, a, b, idesc, acc0); break;
        default: sb_issue_kv<D, 8>(t_acc, a, b, idesc, acc0); break;
    }
}

// Waits until every MMA this thread issued has completed (TMEM is released
// after both issuers have done so).
__device__ __forceinline__ void sb_drain(uint32_t done_bar, const WaitGuard &g, uint32_t site) {
    mma_commit(done_bar);
    WaitGuard drain = g;
    uint32_t no_abort = 0;
    drain.abort = &no_abort;
    mbar_wait(done_bar, 0, drain, site);
}

// The MMAs are issued by three threads. Warp 1: per tile S and dP, then
// (once P and dS are made) dQ, then the next tile's S and dP; warp 3 the dV
// MMAs and warp 2 the dK MMAs of each tile, which read P and dS from the
// shared-memory panels and release them (p_free, once both have). One thread
// issuing all of them sent a tile's 10 dQ and 32 dV / dK MMAs (N = 16) one
// after the other, and the next tile's S and dP only after those. Nothing
// orders the streams but the barriers: the panels are rewritten only after
// p_free, S and dP only after warp 1's own dQ has read dS out of S's
// columns, and the accumulators are disjoint.
template <int D, bool BF16>
__device__ __forceinline__ void sb_mma_sq(uint32_t sbase, uint32_t tmem, int n_items,
                                          const SbPlan &p, const WaitGuard &g) {
    using G = SbGeom<D>;
    auto bar = [&](int i) { return sbase + G::OFF_BAR + 8u * i; };
    const uint32_t idesc_s = mma_idesc_f16(SB_QT, p.n, BF16, false, false);
    constexpr uint32_t idesc_q = mma_idesc_f16(SB_QT, D, BF16, false, true);  // A TMEM, B MN-major
    // stage 0's K-major and MN-major views
    const uint64_t kmaj = smem_desc(sbase, 16, G::SBO, G::LAYOUT);
    const uint64_t mnmaj = smem_desc(sbase, G::TQ_BYTES, G::SBO, G::LAYOUT);
    const uint32_t t_s = tmem, t_dp = tmem + p.c_dp, t_dq = tmem + p.c_dq;
    int n_tile = 0;
    for (int i = 0; i < n_items; ++i) {
        const int st = i % G::STAGES;
        if (!mbar_wait(bar(G::BAR_INF + st), (i / G::STAGES) & 1, g, 42)) break;
        const uint32_t so = (st * G::STAGE_BYTES) >> 4;  // the stage's descriptor offset
        const uint32_t o_do = G::TQ_BYTES >> 4, o_k = (2 * G::TQ_BYTES) >> 4,
                       o_v = (2 * G::TQ_BYTES + G::TK_BYTES) >> 4;
        bool ok = true;
        for (int qt = 0; qt < p.nqt; ++qt, ++n_tile) {
            const uint32_t oq = (qt * SB_QT * G::RB) >> 4;  // the tile's rows of Q / dO
            // S = Q_t K^T, dP = dO_t V^T (the previous tile's dQ MMA has read
            // dS out of S's columns: same thread, in order)
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                mma_ss(t_s, kmaj + so + oq + kk * 2, kmaj + so + o_k + kk * 2, idesc_s,
                       kk > 0 ? 1u : 0u);
                mma_ss(t_dp, kmaj + so + o_do + oq + kk * 2, kmaj + so + o_v + kk * 2, idesc_s,
                       kk > 0 ? 1u : 0u);
            }
            mma_commit(bar(G::BAR_SF));
            if (!mbar_wait(bar(G::BAR_PF), n_tile & 1, g, 43)) {
                ok = false;
                break;
            }
            // dQ = dS K into a free accumulator
            if (n_tile > 0 && !mbar_wait(bar(G::BAR_QE), (n_tile - 1) & 1, g, 44)) {
                ok = false;
                break;
            }
            tc_fence_after();
            sb_issue_dq_n<D>(p.n / 16, t_dq, t_s, mnmaj + so + o_k, idesc_q);
            mma_commit(bar(G::BAR_QF));
        }
        if (!ok) break;
        mma_commit(bar(G::BAR_INE + st));
    }
    sb_drain(bar(G::BAR_DONE), g, 46);
}

// DK = false: dV += P^T dO_t; DK = true: dK += dS^T Q_t.
template <int D, bool BF16, bool DK>
__device__ __forceinline__ void sb_mma_kv(uint32_t sbase, uint32_t tmem, int n_items,
                                          const SbPlan &p, int sq, const WaitGuard &g) {
    using G = SbGeom<D>;
    auto bar = [&](int i) { return sbase + G::OFF_BAR + 8u * i; };
    constexpr uint32_t idesc_kv = mma_idesc_f16(SB_QT, D, BF16, true, true);  // A, B MN-major
    // stage 0's MN-major view; the P or dS panels (MN-major A: the leading
    // offset steps 64 keys, the stride offset 8 query rows)
    const uint64_t mnmaj = smem_desc(sbase, G::TQ_BYTES, G::SBO, G::LAYOUT);
    const uint64_t adesc =
        smem_desc(sbase + (DK ? G::OFF_DS : G::OFF_P), SB_PANEL_BYTES, 1024, kLayoutSw128);
    const uint32_t t_acc = tmem + (DK ? p.c_dk : p.c_dv);
    int n_tile = 0;
    for (int i = 0; i < n_items; ++i) {
        const int st = i % G::STAGES;
        // B: Q_t for dK, dO_t for dV
        const uint32_t ob = (st * G::STAGE_BYTES + (DK ? 0 : G::TQ_BYTES)) >> 4;
        bool ok = true;
        for (int qt = 0; qt < p.nqt; ++qt, ++n_tile) {
            const uint32_t oq = (qt * SB_QT * G::RB) >> 4;
            if (!mbar_wait(bar(G::BAR_PF), n_tile & 1, g, DK ? 55 : 54)) {
                ok = false;
                break;
            }
            // per 128-key M tile, 16 query rows per MMA; the item's first
            // tile overwrites what the previous item's epilogue has read out
            if (qt == 0 && i > 0 && !mbar_wait(bar(G::BAR_KVE), (i - 1) & 1, g, 45)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int rows = min(SB_QT, sq - qt * SB_QT);  // the tile's query rows
            const int ksteps = (rows + 15) / 16;
            for (int mt = 0; mt < p.nmk; ++mt)
                sb_issue_kv_n<D>(ksteps, t_acc + mt * SB_COL_W,
                                 adesc + ((2 * mt * SB_PANEL_BYTES) >> 4), mnmaj + ob + oq, idesc_kv,
                                 qt > 0 ? 1u : 0u);
            mma_commit(bar(G::BAR_PFREE));
        }
        if (!ok) break;
        mma_commit(bar(G::BAR_INE + st));
        mma_commit(bar(G::BAR_KVF));
    }
    sb_drain(bar(G::BAR_DONE + (DK ? 2 : 1)), g, DK ? 56 : 53);
}

// Stores COLS fp32 TMEM columns of this thread's lane, times mul, as 16-bit.
template <int COLS, bool BF16>
__device__ __forceinline__ void sb_store_row(uint32_t taddr, float mul, uint16_t *dst, bool out) {
#pragma unroll
    for (int c0 = 0; c0 < COLS; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(taddr + c0, v);
        tmem_wait_ld();
        if (out) {
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                pk[i] = sb_pack<BF16>(__uint_as_float(v[2 * i]) * mul,
                                      __uint_as_float(v[2 * i + 1]) * mul);
            uint4 *d4 = reinterpret_cast<uint4 *>(dst + c0);
            d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
    }
}

template <int D, bool BF16>
__device__ __forceinline__ void sb_elementwise(uint8_t *smem, uint32_t sbase, uint32_t tmem,
                                               int q4, int grp, int n_items, const SbPlan &p,
                                               const BwdArgs &a, const WaitGuard &g) {
    using G = SbGeom<D>;
    auto bar = [&](int i) { return sbase + G::OFF_BAR + 8u * i; };
    const uint32_t lane = threadIdx.x & 31;
    const int row = q4 * 32 + lane;  // TMEM lane: a query row of the tile (a key row for dK, dV)
    const uint32_t lanes = static_cast<uint32_t>(q4 * 32) << 16;
    const float c = a.scale_log2;
    const int nch16 = p.n / 16;  // 16-key chunks (even: n is a multiple of 32)
    // this thread's rows of the P and dS panels (row of 128 bytes, 16-byte
    // chunks XOR-swizzled by the row's low three bits)
    uint8_t *prow = smem + G::OFF_P + row * 128;
    uint8_t *dsrow = smem + G::OFF_DS + row * 128;
    const int sw = row & 7;
    int n_tile = 0;
    for (int i = 0; i < n_items; ++i) {
        const int it = blockIdx.x + i * gridDim.x;
        const int head = it % a.h, batch = it / a.h;
        const int st = i % G::STAGES;
        const bool okl = mbar_wait(bar(G::BAR_LDF + st), (i / G::STAGES) & 1, g, 52);
        if (!__all_sync(0xffffffffu, okl)) return;
        const float *ld = reinterpret_cast<const float *>(smem + G::OFF_LD) + st * 2 * SBWD_MAX_Q;
        for (int qt = 0; qt < p.nqt; ++qt, ++n_tile) {
            const int grow = qt * SB_QT + row;
            const bool valid = grow < a.sq;
            // rows past sq: LSE = +inf makes P = 0, and dO (TMA zero fill) dP = 0
            const float lse2 = ld[grow];
            const float drow = ld[SBWD_MAX_Q + grow];
            const bool oks = mbar_wait(bar(G::BAR_SF), n_tile & 1, g, 47);
            if (!__all_sync(0xffffffffu, oks)) return;
            // the previous tile's dV / dK MMAs have read the P and dS panels
            if (n_tile > 0) {
                const bool okf = mbar_wait(bar(G::BAR_PFREE), (n_tile - 1) & 1, g, 48);
                if (!__all_sync(0xffffffffu, okf)) return;
            }
            tc_fence_after();
            // a warp whose 32 rows are all past sq has nothing the MMAs read
            // (they stop at the tile's last 16-row step holding a query row)
            const bool live = q4 * 32 < a.sq - qt * SB_QT;
            // 16-key chunks j = grp, grp + 2, ...: the next chunk's TMEM loads
            // are in flight while this one is worked on
            const uint32_t t_s = tmem + lanes, t_dp = tmem + lanes + p.c_dp;
            auto work = [&](const uint32_t (&sv)[16], const uint32_t (&pv)[16], int j) {
                uint32_t pp[8], pd[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int k = 16 * j + 2 * e;
                    float p0 = fast_exp2(__uint_as_float(sv[2 * e]) * c - lse2);
                    float p1 = fast_exp2(__uint_as_float(sv[2 * e + 1]) * c - lse2);
                    p0 = k < a.sk ? p0 : 0.f;  // keys past sk (TMA zero fill) take no part
                    p1 = k + 1 < a.sk ? p1 : 0.f;
                    pp[e] = sb_pack<BF16>(p0, p1);
                    pd[e] = sb_pack<BF16>(p0 * (__uint_as_float(pv[2 * e]) - drow),
                                          p1 * (__uint_as_float(pv[2 * e + 1]) - drow));
                }
                // dS of the chunk's 16 keys into its first 8 columns (read
                // already, by this thread): the A operand of dQ = dS K
                tmem_st8(t_s + 16 * j, pd);
                // P and dS rows into the panels: keys 16 j .. 16 j + 15 are
                // 16-byte chunks 2 (j & 3), + 1 of panel j / 4
                const int pan = (j >> 2) * SB_PANEL_BYTES;
                const int c0 = (j & 3) * 2;
                const int o0 = pan + ((c0 ^ sw) << 4), o1 = pan + (((c0 + 1) ^ sw) << 4);
                *reinterpret_cast<uint4 *>(prow + o0) = make_uint4(pp[0], pp[1], pp[2], pp[3]);
                *reinterpret_cast<uint4 *>(prow + o1) = make_uint4(pp[4], pp[5], pp[6], pp[7]);
                *reinterpret_cast<uint4 *>(dsrow + o0) = make_uint4(pd[0], pd[1], pd[2], pd[3]);
                *reinterpret_cast<uint4 *>(dsrow + o1) = make_uint4(pd[4], pd[5], pd[6], pd[7]);
            };
            if (live) {
                uint32_t sa[16], pa[16], sb[16], pb[16];
                int j = grp;
                tmem_ld16(t_s + 16 * j, sa);
                tmem_ld16(t_dp + 16 * j, pa);
                tmem_wait_ld();
#pragma unroll 1
                for (; j < nch16; j += 4) {
                    if (j + 2 < nch16) {
                        tmem_ld16(t_s + 16 * (j + 2), sb);
                        tmem_ld16(t_dp + 16 * (j + 2), pb);
                    }
                    work(sa, pa, j);
                    if (j + 2 >= nch16) break;
                    tmem_wait_ld();
                    if (j + 4 < nch16) {
                        tmem_ld16(t_s + 16 * (j + 4), sa);
                        tmem_ld16(t_dp + 16 * (j + 4), pa);
                    }
                    work(sb, pb, j + 2);
                    tmem_wait_ld();
                }
            }
            fence_proxy_async_smem();  // the panels, for the tensor core
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(G::BAR_PF));

            // dQ of the tile: each group stores 16 of its columns (d = 16:
            // group 0 alone)
            const bool okq = mbar_wait(bar(G::BAR_QF), n_tile & 1, g, 49);
            if (!__all_sync(0xffffffffu, okq)) return;
            tc_fence_after();
            if (grp * 16 < D) {
                uint16_t *dst = reinterpret_cast<uint16_t *>(a.dq) +
                                ((static_cast<int64_t>(batch) * a.sq + (valid ? grow : 0)) * a.h +
                                 head) * D + grp * 16;
                sb_store_row<16, BF16>(tmem + lanes + p.c_dq + grp * 16, a.scale, dst, valid);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(G::BAR_QE));
        }
        // dK and dV of the item: group g stores key M tile g
        const bool okk = mbar_wait(bar(G::BAR_KVF), i & 1, g, 50);
        if (!__all_sync(0xffffffffu, okk)) return;
        tc_fence_after();
        if (grp < p.nmk) {
            const int key = grp * SB_QT + row;
            const bool out = key < a.sk;
            const int64_t off =
                ((static_cast<int64_t>(batch) * a.sk + (out ? key : 0)) * a.h + head) * D;
            sb_store_row<D, BF16>(tmem + lanes + p.c_dv + grp * SB_COL_W, 1.0f,
                                  reinterpret_cast<uint16_t *>(a.dv) + off, out);
            sb_store_row<D, BF16>(tmem + lanes + p.c_dk + grp * SB_COL_W, a.scale,
                                  reinterpret_cast<uint16_t *>(a.dk) + off, out);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(G::BAR_KVE));
    }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(SB_THREADS, 1)
    bwd_short_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv,
                     const __grid_constant__ CUtensorMap tdo, const BwdArgs a) {
    using G = SbGeom<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw);
    auto bar = [&](int i) { return sbase + G::OFF_BAR + 8u * i; };

    const int warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    const int items = a.b * a.h;
    const int n_items =
        static_cast<int>(blockIdx.x) < items ? (items - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
    const SbPlan p = sb_plan(a);

    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + G::OFF_MISC);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + G::OFF_MISC + 4);
    if (threadIdx.x == 0) {
        for (int i = 0; i < G::NUM_BARS; ++i) {
            const bool by_warps = i == G::BAR_PF || i == G::BAR_QE || i == G::BAR_KVE;
            // commits of all three issuers (the stages), of the dV and dK
            // issuers (the panels, the item's dK and dV); BAR_LDF: one
            // arrive by warp 0's lane 0
            const uint32_t n_arrive = by_warps ? static_cast<uint32_t>(SB_EW_WARPS)
                                      : (i == G::BAR_INE || i == G::BAR_INE + 1) ? 3u
                                      : (i == G::BAR_PFREE || i == G::BAR_KVF)   ? 2u
                                                                                 : 1u;
            mbar_init(bar(i), n_arrive);
        }
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        tma_prefetch_desc(&tdo);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitGuard g{abort_flag, a.status, kKernBwd};

    if (warp == 0) {
        if (!(a.flags & kFlagSkipLoads))
            sb_producer<D>(&tq, &tk, &tv, &tdo, smem, sbase, items, p, a, g);
    } else if (warp == 1) {
        if (lane == 0) sb_mma_sq<D, BF16>(sbase, tmem, n_items, p, g);
    } else if (warp == 2) {
        if (lane == 0) sb_mma_kv<D, BF16, true>(sbase, tmem, n_items, p, a.sq, g);
    } else if (warp == 3) {
        if (lane == 0) sb_mma_kv<D, BF16, false>(sbase, tmem, n_items, p, a.sq, g);
    } else if (warp >= 4) {
        sb_elementwise<D, BF16>(smem, sbase, tmem, warp & 3, (warp - 4) >> 2, n_items, p, a, g);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int D, bool BF16>
cudaError_t launch_sb_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                        const CUtensorMap &tdo, const BwdArgs &a, cudaStream_t stream) {
    using G = SbGeom<D>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_set[dev]) {
        e = cudaFuncSetAttribute(bwd_short_kernel<D, BF16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const int64_t items = static_cast<int64_t>(a.b) * a.h;
    const int64_t grid = items < a.num_sms ? items : a.num_sms;
    bwd_short_kernel<D, BF16>
        <<<static_cast<unsigned>(grid), SB_THREADS, G::SMEM_BYTES, stream>>>(tq, tk, tv, tdo, a);
    return cudaGetLastError();
}

}  // namespace

bool bwd_short_plan(int sq, int sk, int d, bool causal) {
    if (causal || (d != 16 && d != 32)) return false;
    if (sq < 1 || sq > SBWD_MAX_Q || sk < 1) return false;
    const int n = (sk + 31) / 32 * 32;
    return n <= SB_MAX_N;
}

cudaError_t launch_bwd_short(int d, bool bf16, const CUtensorMap &tq, const CUtensorMap &tk,
                             const CUtensorMap &tv, const CUtensorMap &tdo, const BwdArgs &a,
                             cudaStream_t stream) {
    cudaError_t e = launch_bwd_dot(d, bf16, a, stream);
    if (e != cudaSuccess) return e;
    switch (d) {
        case 16:
            return bf16 ? launch_sb_t<16, true>(tq, tk, tv, tdo, a, stream)
                        : launch_sb_t<16, false>(tq, tk, tv, tdo, a, stream);
        case 32:
            return bf16 ? launch_sb_t<32, true>(tq, tk, tv, tdo, a, stream)
                        : launch_sb_t<32, false>(tq, tk, tv, tdo, a, stream);
        default:
            return cudaErrorInvalidValue;
    }
}

}  // namespace exattn
