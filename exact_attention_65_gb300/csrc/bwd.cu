// Backward pass of exact attention on sm_103a: dQ, dK, dV from Q, K, V, the
// forward's O and LSE, and the upstream gradient dO.
//
// The pages time a backward pass (the flash-attn timing issue) but do not
// write one out; what is computed is the chain rule of the forward's
// definition. With S = scale * Q K^T, P = softmax(S) by rows (recomputed
// from the saved LSE: P = exp(S - LSE)), O = P V:
//     dV = P^T dO,   dP = dO V^T,   D = rowsum(dO * O) = rowsum(P * dP),
//     dS = P * (dP - D),   dQ = scale * dS K,   dK = scale * dS^T Q.
// Nothing of size s^2 goes to HBM: each score tile is recomputed on chip,
// as in the forward ("Why FlashAttention is fast", section 3.2).
//
// Three kernels:
//   bwd_dot_kernel   D = rowsum(dO * O), fp32 [b, h, sq].
//   bwd_kernel<DQ>   one unit = a 128-row query tile; it keeps Q and dO in
//                    shared memory, streams K_j and V_j, and accumulates
//                    dQ += dS K_j in TMEM.
//   bwd_kernel<DKV>  one unit = a 128-key tile; it keeps K and V, streams
//                    Q_i and dO_i, and accumulates dV += P^T dO_i and
//                    dK += dS^T Q_i in TMEM.
// Computing dQ in its own pass (recomputing S and dP once more) avoids
// accumulating it across CTAs with atomics.
//
// Both are persistent kernels with the forward's roles: warp 0 is the TMA
// producer (the unit's fixed pair of tiles, then a ring of streamed tiles),
// one thread of warp 1 issues the tcgen05 MMAs, warps 4-11 hold one TMEM lane
// (one row of the tile) per thread in two groups that split the columns, and
// do the elementwise work. For each step the MMAs write the score tile and
// the dP tile to TMEM; the warps turn them into 16-bit P and dS written back
// in place, a 64-column half at a time; then the accumulating MMAs read them
// from TMEM, the first half's while the warps work on the second.
//
// TMEM columns: [0, 128) score tile (then P or dS), [128, 256) dP tile (then
// dS in the dK/dV kernel), [256, 256 + d) dQ or dV, [384, 384 + d) dK; the
// dQ kernel keeps Q and dO as 16-bit MMA operands in [384, 384 + d).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace exattn {
namespace {

constexpr int kBwdDQ = 0;   // query-tile units: dQ
constexpr int kBwdDKV = 1;  // key-tile units: dK and dV
// warp 0 producer, warp 1 MMA issuer, warps 2-3 idle, warps 4-11 elementwise
// (two groups of four: each group holds all 128 TMEM lanes, and group g takes
// columns [32g, 32g + 32) of every 64-column half of the score tile)
constexpr int kBwdThreads = 384;
constexpr int kBwdComputeWarps = 8;

template <int D>
struct BwdGeom {
    static constexpr int BT = 128;  // rows of every tile
    static constexpr int HN = 64;   // a step's score tile is made and used in two halves of HN columns
    static constexpr int ROW_BYTES = fwd_row_bytes(D);
    static constexpr int PANELS = (D * 2) / ROW_BYTES;
    static constexpr int PANEL_ELEMS = ROW_BYTES / 2;
    static constexpr int PANEL_BYTES = BT * ROW_BYTES;
    static constexpr int TILE_BYTES = BT * D * 2;
    static constexpr int SLOTS = D == 128 ? 4 : 8;  // streamed tiles, two per step
    static constexpr uint32_t LAYOUT =
        ROW_BYTES == 128 ? kLayoutSw128 : (ROW_BYTES == 64 ? kLayoutSw64 : kLayoutSw32);
    static constexpr uint32_t SBO = 8 * ROW_BYTES;
    static constexpr int TMEM_COLS = 512;
    static constexpr int T_S = 0, T_P = 128, T_A0 = 256, T_A1 = 384;
    // dQ kernel: the fixed Q and dO tiles as 16-bit MMA A operands in TMEM
    static constexpr int T_Q = 384, T_DO = T_Q + D / 2;
    static_assert(T_DO + D / 2 <= TMEM_COLS, "TMEM budget");

    static constexpr int OFF_FIX = 0;                       // the unit's two fixed tiles
    static constexpr int OFF_RING = 2 * TILE_BYTES;
    static constexpr int OFF_BAR = OFF_RING + SLOTS * TILE_BYTES;
    // barriers: fix_full | fix_empty | ring_full[SLOTS] | ring_empty[SLOTS] |
    //           s_full[2] | p_full[2] | acc_full | acc_empty | ld[2] | done
    static constexpr int BAR_FF = 0;
    static constexpr int BAR_FE = 1;
    static constexpr int BAR_RF = 2;
    static constexpr int BAR_RE = BAR_RF + SLOTS;
    static constexpr int BAR_SF = BAR_RE + SLOTS;  // [2]: a half's S and dP written
    static constexpr int BAR_PF = BAR_SF + 2;      // [2]: a half's P / dS written back
    static constexpr int BAR_AF = BAR_PF + 2;
    static constexpr int BAR_AE = BAR_AF + 1;
    static constexpr int BAR_LD = BAR_AE + 1;  // [2]: a step's LSE and D staged (dK/dV kernel)
    static constexpr int BAR_DONE = BAR_LD + 2;
    static constexpr int NUM_BARS = BAR_DONE + 1;
    // per step parity: LSE * log2(e) of the step's 128 query rows, then their D
    static constexpr int OFF_LD = (OFF_BAR + NUM_BARS * 8 + 15) & ~15;  // read as float4
    static constexpr int OFF_MISC = OFF_LD + 2 * 2 * BT * 4;
    static constexpr int USED = OFF_MISC + 16;
    static constexpr int MIN_SMEM = 120 * 1024;  // one CTA per SM: it owns all of TMEM
    static constexpr int SMEM_BYTES = (USED > MIN_SMEM ? USED : MIN_SMEM) + 1024;
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

template <bool BF16>
__device__ __forceinline__ uint32_t pack2b(float lo, float hi) {
    if constexpr (BF16)
        return cvt_pack_bf16(lo, hi);
    else
        return cvt_pack_f16(lo, hi);
}

template <bool BF16>
__device__ __forceinline__ float to_f32(uint16_t bits) {
    if constexpr (BF16)
        return __uint_as_float(static_cast<uint32_t>(bits) << 16);
    else
        return __half2float(__ushort_as_half(bits));
}

// D[b, h, i] = sum_t dO[b, i, h, t] * O[b, i, h, t] in fp32; d/8 lanes per row.
template <int D, bool BF16>
__global__ void __launch_bounds__(256)
    bwd_dot_kernel(const uint16_t *__restrict__ o, const uint16_t *__restrict__ dout,
                   float *__restrict__ dvec, int b, int sq, int h) {
    constexpr int LPR = D / 8;
    constexpr int RPW = 32 / LPR;
    const int lane = threadIdx.x & 31;
    const int64_t rows = static_cast<int64_t>(b) * sq * h;
    const int64_t r = (static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5)) *
                          RPW + lane / LPR;
    const int sub = lane % LPR;
    float acc = 0.f;
    if (r < rows) {
        const uint4 wo = *reinterpret_cast<const uint4 *>(o + r * D + sub * 8);
        const uint4 wd = *reinterpret_cast<const uint4 *>(dout + r * D + sub * 8);
        const uint32_t uo[4] = {wo.x, wo.y, wo.z, wo.w};
        const uint32_t ud[4] = {wd.x, wd.y, wd.z, wd.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc = fmaf(to_f32<BF16>(static_cast<uint16_t>(uo[i] & 0xffffu)),
                       to_f32<BF16>(static_cast<uint16_t>(ud[i] & 0xffffu)), acc);
            acc = fmaf(to_f32<BF16>(static_cast<uint16_t>(uo[i] >> 16)),
                       to_f32<BF16>(static_cast<uint16_t>(ud[i] >> 16)), acc);
        }
    }
#pragma unroll
    for (int off = LPR / 2; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (r < rows && sub == 0) {
        // r = (batch * sq + i) * h + head  ->  [b, h, sq]
        const int head = static_cast<int>(r % h);
        const int64_t bi = r / h;
        const int i = static_cast<int>(bi % sq);
        const int64_t batch = bi / sq;
        dvec[(batch * h + head) * sq + i] = acc;
    }
}

// A unit: tile `tile` (128 rows) of one (batch, head); its rows are query
// rows (dQ kernel) or key rows (dK/dV kernel).
struct BUnit {
    int tile, head, batch;
};

// Without a mask the tiles of one (batch, head) are neighbours, so CTAs
// running at the same time share its streamed tiles in L2. Under the causal
// mask units differ in length (a query tile's grows with its index, a key
// tile's shrinks), and a grid that is a multiple of the tile count would keep
// each CTA on one tile index; there units run longest first across all
// (batch, head) pairs, so the round-robin over CTAs deals each a mix.
template <int MODE, bool CAUSAL>
__device__ __forceinline__ BUnit bunit_of(int u, int ntiles, const BwdArgs &a) {
    BUnit x;
    int r;
    if constexpr (CAUSAL) {
        const int bh = a.b * a.h;
        const int rank = u / bh;
        r = u - rank * bh;
        x.tile = MODE == kBwdDQ ? ntiles - 1 - rank : rank;
    } else {
        x.tile = u % ntiles;
        r = u / ntiles;
    }
    x.head = r % a.h;
    x.batch = r / a.h;
    return x;
}

// The streamed tiles a unit visits: first .. first + count - 1 of nsteps_all.
// With the causal mask (query row i sees key k only if k <= i + sk - sq) a
// query tile stops at its last row's last visible key tile, and a key tile
// starts at the first query tile that can see any of its keys; a unit with
// nothing left (count 0) writes zeros.
template <int MODE, bool CAUSAL>
__device__ __forceinline__ void unit_steps(const BUnit &x, int nsteps_all, const BwdArgs &a,
                                           int &first, int &count) {
    first = 0;
    count = nsteps_all;
    if constexpr (CAUSAL) {
        const int off = a.sk - a.sq;
        if constexpr (MODE == kBwdDQ) {
            const int last = min(x.tile * 128 + 127, a.sq - 1);
            const int kmax = last + off;
            count = kmax < 0 ? 0 : min(nsteps_all, kmax / 128 + 1);
        } else {
            const int q0 = x.tile * 128 - off;  // first query row seeing the tile's first key
            first = q0 <= 0 ? 0 : min(q0 / 128, nsteps_all);
            count = nsteps_all - first;
        }
    }
}

template <int D, int MODE, bool CAUSAL>
__device__ __forceinline__ void bwd_producer(const CUtensorMap *tq, const CUtensorMap *tk,
                                             const CUtensorMap *tv, const CUtensorMap *tdo,
                                             uint32_t sbase, int ntiles, int nsteps, int units,
                                             const BwdArgs &a, const WaitGuard &g) {
    using G = BwdGeom<D>;
    auto bar = [&](int i) { return sbase + G::OFF_BAR + 8u * i; };
    // the unit's fixed pair and the streamed pair of each step
    const CUtensorMap *fa = MODE == kBwdDQ ? tq : tk;
    const CUtensorMap *fb = MODE == kBwdDQ ? tdo : tv;
    const CUtensorMap *sa = MODE == kBwdDQ ? tk : tq;
    const CUtensorMap *sb = MODE == kBwdDQ ? tv : tdo;
    const uint64_t keep = policy_evict_last();  // streamed tiles are re-read by other units
    int it_u = 0, n_issued = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x, ++it_u) {
        const BUnit x = bunit_of<MODE, CAUSAL>(u, ntiles, a);
        int first, count;
        unit_steps<MODE, CAUSAL>(x, nsteps, a, first, count);
        if (!mbar_wait(bar(G::BAR_FE), (it_u & 1) ^ 1, g, 1)) break;
        mbar_arrive_expect_tx(bar(G::BAR_FF), 2 * G::TILE_BYTES);
        for (int p = 0; p < G::PANELS; ++p) {
            tma_load_4d(sbase + G::OFF_FIX + p * G::PANEL_BYTES, fa, bar(G::BAR_FF),
                        p * G::PANEL_ELEMS, x.head, x.tile * G::BT, x.batch);
            tma_load_4d(sbase + G::OFF_FIX + G::TILE_BYTES + p * G::PANEL_BYTES, fb, bar(G::BAR_FF),
                        p * G::PANEL_ELEMS, x.head, x.tile * G::BT, x.batch);
        }
        for (int i = 0; i < 2 * count; ++i) {  // step j: item 2j from sa, 2j + 1 from sb
            const int s = n_issued % G::SLOTS;
            if (!mbar_wait(bar(G::BAR_RE + s), ((n_issued / G::SLOTS) & 1) ^ 1, g, 2)) {
                ok = false;
                break;
            }
            mbar_arrive_expect_tx(bar(G::BAR_RF + s), G::TILE_BYTES);
            const CUtensorMap *map = (i & 1) ? sb : sa;
            for (int p = 0; p < G::PANELS; ++p)
                tma_load_4d_hint(sbase + G::OFF_RING + s * G::TILE_BYTES + p * G::PANEL_BYTES, map,
                                 bar(G::BAR_RF + s), p * G::PANEL_ELEMS, x.head,
                                 (first + (i >> 1)) * G::BT, x.batch, keep);
            ++n_issued;
        }
    }
    // wait (bounded, even after an abort) for the copies still landing
    WaitGuard drain = g;
    uint32_t no_abort = 0;
    drain.abort = &no_abort;
    if (it_u > 0) mbar_wait(bar(G::BAR_FF), (it_u - 1) & 1, drain, 9);
    for (int n = (n_issued > G::SLOTS ? n_issued - G::SLOTS : 0); n < n_issued; ++n)
        mbar_wait(bar(G::BAR_RF + n % G::SLOTS), (n / G::SLOTS) & 1, drain, 10);
}

template <int D, int MODE, bool BF16, bool CAUSAL>
__device__ __forceinline__ void bwd_mma(uint32_t sbase, uint32_t tmem, int ntiles, int nsteps,
                                        int units, const BwdArgs &a, const WaitGuard &g) {
    using G = BwdGeom<D>;
    auto bar = [&](int i) { return sbase + G::OFF_BAR + 8u * i; };
    // Width of the S / dP MMAs. A 128 x 64 MMA takes about as long on the
    // tensor core as a 128 x 128 one, so S and dP are made whole; the warps
    // still hand P / dS over a half at a time, and the first half's
    // accumulation runs while they work on the second.
    constexpr bool kFull = true;
    constexpr uint32_t idesc_half = mma_idesc_f16(G::BT, kFull ? G::BT : G::HN, BF16, false, false);
    constexpr uint32_t idesc_acc = mma_idesc_f16(G::BT, D, BF16, false, true);      // 128 x d, B MN-major
    // K-major and MN-major descriptors of the fixed tiles and of ring slot 0
    const uint64_t fix_k = smem_desc(sbase + G::OFF_FIX, 16, G::SBO, G::LAYOUT);
    const uint64_t ring_k = smem_desc(sbase + G::OFF_RING, 16, G::SBO, G::LAYOUT);
    const uint64_t ring_mn = smem_desc(sbase + G::OFF_RING, G::PANEL_BYTES, G::SBO, G::LAYOUT);
    constexpr uint32_t tile16 = G::TILE_BYTES >> 4;
    // HN rows into a tile: a whole number of swizzle atoms (8 rows each)
    constexpr uint32_t half16 = (G::HN * G::ROW_BYTES) >> 4;

    // Half h of a step's S and dP (or both halves at once): the fixed tiles
    // (A, 128 rows) times rows [h HN, (h+1) HN) of the streamed pair (B,
    // K-major), over the head dim.
    // (dQ kernel: A = Q and dO from TMEM, copied there once per unit, so
    // that only B is read from shared memory; dK/dV kernel: A = K and V from
    // shared memory, TMEM being full.)
    auto issue_sdp = [&](int sa, int sb, int h) {
        const uint32_t row16 = kFull ? 0u : h * half16;
        const uint32_t col = kFull ? 0u : h * G::HN;
        const uint64_t ba = ring_k + sa * tile16 + row16;
        const uint64_t bb = ring_k + sb * tile16 + row16;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const int p = (kk * 16) / G::PANEL_ELEMS;
            const int off = ((kk * 16) % G::PANEL_ELEMS) * 2;
            const uint32_t o16 = (p * G::PANEL_BYTES + off) >> 4;
            if constexpr (MODE == kBwdDQ)
                mma_ts(tmem + G::T_S + col, tmem + G::T_Q + kk * 8, ba + o16, idesc_half,
                       kk > 0 ? 1u : 0u);
            else
                mma_ss(tmem + G::T_S + col, fix_k + o16, ba + o16, idesc_half, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const int p = (kk * 16) / G::PANEL_ELEMS;
            const int off = ((kk * 16) % G::PANEL_ELEMS) * 2;
            const uint32_t o16 = (p * G::PANEL_BYTES + off) >> 4;
            if constexpr (MODE == kBwdDQ)
                mma_ts(tmem + G::T_P + col, tmem + G::T_DO + kk * 8, bb + o16, idesc_half,
                       kk > 0 ? 1u : 0u);
            else
                mma_ss(tmem + G::T_P + col, fix_k + tile16 + o16, bb + o16, idesc_half,
                       kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(G::BAR_SF + h));
        if (kFull) mma_commit(bar(G::BAR_SF + 1));  // both halves are there
    };
    // acc (+)= A[TMEM: 128 rows x HN, 16-bit] times B[HN rows x d, MN-major],
    // 16 rows of B per MMA. The warp group that made columns [32g, 32g + 32)
    // of the half packed them into the half's columns [32g, 32g + 16).
    auto mma_acc_half = [&](uint32_t dst, uint32_t a_tmem, uint64_t bdesc_mn, bool first) {
#pragma unroll
        for (int kk = 0; kk < G::HN / 16; ++kk)
            mma_ts(dst, a_tmem + (kk >> 1) * 32 + (kk & 1) * 8,
                   bdesc_mn + ((kk * 16 * G::ROW_BYTES) >> 4), idesc_acc,
                   (!first || kk > 0) ? 1u : 0u);
    };
    // ring slots of global step gs, waited for until loaded
    auto wait_ring = [&](int gs, int &sa, int &sb) {
        const int na = 2 * gs, nb = na + 1;
        sa = na % G::SLOTS;
        sb = nb % G::SLOTS;
        return mbar_wait(bar(G::BAR_RF + sa), (na / G::SLOTS) & 1, g, 5) &&
               mbar_wait(bar(G::BAR_RF + sb), (nb / G::SLOTS) & 1, g, 6);
    };

    // Software pipeline over half steps. For half h of step j the issuer
    // waits for the warps' P / dS of (j, h), queues the accumulation of
    // (j, h) and then S / dP of (j + 1, h) into the same columns (the tensor
    // core runs in order, so the accumulation has read them first; with
    // whole-width S / dP, after the second half). The tensor core works on
    // one half while the warps work on the other.
    int it_u = 0, base = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x, ++it_u) {
        if (!mbar_wait(bar(G::BAR_FF), it_u & 1, g, 4)) break;
        int first, count;
        unit_steps<MODE, CAUSAL>(bunit_of<MODE, CAUSAL>(u, ntiles, a), nsteps, a, first, count);
        if (count == 0) {  // nothing to accumulate: free the fixed tiles, hand over
            mma_commit(bar(G::BAR_FE));
            mma_commit(bar(G::BAR_AF));
            continue;
        }
        if constexpr (MODE == kBwdDQ) {
            // Q and dO into TMEM, 16 head-dim columns per copy, after the last
            // S / dP MMAs of the previous unit (same thread, in order); then
            // their shared-memory tiles are free for the next unit's loads.
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int p = (kk * 16) / G::PANEL_ELEMS;
                const int off = ((kk * 16) % G::PANEL_ELEMS) * 2;
                const uint32_t o16 = (p * G::PANEL_BYTES + off) >> 4;
                tmem_cp_128x256b(tmem + G::T_Q + kk * 8, fix_k + o16);
                tmem_cp_128x256b(tmem + G::T_DO + kk * 8, fix_k + tile16 + o16);
            }
            mma_commit(bar(G::BAR_FE));
        }
        int sa = 0, sb = 0;
        if (!wait_ring(base, sa, sb)) {
            ok = false;
            break;
        }
        tc_fence_after();
        issue_sdp(sa, sb, 0);
        if (!kFull) issue_sdp(sa, sb, 1);
        for (int j = 0; ok && j < count; ++j) {
            const int gs = base + j;
            int na = 0, nb = 0;  // ring slots of step j + 1
            for (int h = 0; h < 2; ++h) {
                if (!mbar_wait(bar(G::BAR_PF + h), gs & 1, g, 8)) {
                    ok = false;
                    break;
                }
                // The first accumulation of a unit overwrites the accumulators:
                // the previous unit's epilogue must have read them out.
                if (j == 0 && h == 0 && !mbar_wait(bar(G::BAR_AE), (it_u & 1) ^ 1, g, 7)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const bool first_acc = j == 0 && h == 0;
                const uint32_t col = h * G::HN;
                if constexpr (MODE == kBwdDQ) {
                    // dQ += dS K_j (rows of K_j in this half)
                    mma_acc_half(tmem + G::T_A0, tmem + G::T_S + col, ring_mn + sa * tile16 + h * half16,
                                 first_acc);
                } else {
                    // dV += P^T dO_i, dK += dS^T Q_i (query rows of this half)
                    mma_acc_half(tmem + G::T_A0, tmem + G::T_S + col, ring_mn + sb * tile16 + h * half16,
                                 first_acc);
                    mma_acc_half(tmem + G::T_A1, tmem + G::T_P + col, ring_mn + sa * tile16 + h * half16,
                                 first_acc);
                }
                if (h == 1) {  // step j's streamed tiles are read for the last time
                    mma_commit(bar(G::BAR_RE + sa));
                    mma_commit(bar(G::BAR_RE + sb));
                }
                if (j + 1 < count && (!kFull || h == 1)) {
                    if (h == 0 || kFull) {
                        if (!wait_ring(gs + 1, na, nb)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    issue_sdp(na, nb, kFull ? 0 : h);
                }
            }
            if (!ok) break;
            sa = na;
            sb = nb;
        }
        if (!ok) break;
        if constexpr (MODE == kBwdDKV) mma_commit(bar(G::BAR_FE));
        mma_commit(bar(G::BAR_AF));
        base += count;
    }
    mma_commit(bar(G::BAR_DONE));
    WaitGuard drain = g;
    uint32_t no_abort = 0;
    drain.abort = &no_abort;
    mbar_wait(bar(G::BAR_DONE), 0, drain, 12);
}

// Store `cols` columns (multiple of 16) of one fp32 TMEM row, scaled, as
// 16-bit values at dst.
template <int COLS, bool BF16>
__device__ __forceinline__ void store_row(uint32_t taddr, float mul, uint16_t *dst, bool out,
                                          bool zero) {
#pragma unroll
    for (int c0 = 0; c0 < COLS; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(taddr + c0, v);
        tmem_wait_ld();
        if (out) {
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                pk[i] = zero ? 0u
                             : pack2b<BF16>(__uint_as_float(v[2 * i]) * mul,
                                            __uint_as_float(v[2 * i + 1]) * mul);
            uint4 *d4 = reinterpret_cast<uint4 *>(dst + c0);
            d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
    }
}

template <int D, int MODE, bool BF16, bool CAUSAL>
__device__ __forceinline__ void bwd_compute(uint8_t *smem, uint32_t sbase, uint32_t tmem, int q4, int cg,
                                            int ntiles, int nsteps, int units, const BwdArgs &a,
                                            const WaitGuard &g) {
    using G = BwdGeom<D>;
    auto bar = [&](int i) { return sbase + G::OFF_BAR + 8u * i; };
    const uint32_t lane = threadIdx.x & 31;
    const int row = q4 * 32 + lane;  // TMEM lane = row of the unit's tile
    const uint32_t lanes = static_cast<uint32_t>(q4 * 32) << 16;
    const float c = a.scale_log2;
    constexpr float kLog2e = 1.4426950408889634f;
    int it_u = 0, step = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++it_u) {
        const BUnit x = bunit_of<MODE, CAUSAL>(u, ntiles, a);
        int first, count;
        unit_steps<MODE, CAUSAL>(x, nsteps, a, first, count);
        const int grow = x.tile * G::BT + row;
        const int64_t bh = static_cast<int64_t>(x.batch) * a.h + x.head;
        // dQ kernel: this row's LSE (log2 units) and D; rows past sq take no part
        float lse2 = INFINITY, drow = 0.f;
        if constexpr (MODE == kBwdDQ) {
            if (grow < a.sq) {
                lse2 = a.lse[bh * a.sq + grow] * kLog2e;
                drow = a.dvec[bh * a.sq + grow];
            }
        }
        for (int j = 0; j < count; ++j, ++step) {
            const int tj = first + j;  // the streamed tile of this step
            const float *ldbuf = nullptr;
            if constexpr (MODE == kBwdDKV) {
                // Stage the step's LSE (log2 units) and D: thread `row` takes query
                // row j*128 + row. Double-buffered by step parity; the buffer is
                // rewritten two steps later, after every warp has passed the
                // barrier of the step in between.
                // (group 0 stages, both groups read)
                float *buf = reinterpret_cast<float *>(smem + G::OFF_LD) + (step & 1) * 2 * G::BT;
                if (cg == 0) {
                    const int qr = tj * G::BT + row;
                    buf[row] = qr < a.sq ? a.lse[bh * a.sq + qr] * kLog2e : INFINITY;
                    buf[G::BT + row] = qr < a.sq ? a.dvec[bh * a.sq + qr] : 0.f;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(G::BAR_LD + (step & 1)));
                }
                const bool okl = mbar_wait(bar(G::BAR_LD + (step & 1)), (step >> 1) & 1, g, 15);
                if (!__all_sync(0xffffffffu, okl)) return;
                ldbuf = buf;
            }
            // the score tile in two halves of HN columns, as the MMAs make them
            for (int h = 0; h < 2; ++h) {
                const bool ok = mbar_wait(bar(G::BAR_SF + h), step & 1, g, 13);
                if (!__all_sync(0xffffffffu, ok)) return;
                tc_fence_after();
                const int hc = h * G::HN;  // first column of the half
                if constexpr (MODE == kBwdDQ) {
                    // row = query row; columns = keys tj*128 + hc .. : P = 2^(s c - lse2),
                    // dS = P (dP - D); keys past sk (TMA zero fill) take no part.
                    // (causal: the row's own last visible key)
                    const int kv = (CAUSAL ? min(a.sk, grow + a.sk - a.sq + 1) : a.sk) - tj * G::BT - hc;
                    {
                        const int c0 = 32 * cg;  // this group's columns of the half
                        uint32_t sv[32], pv[32];
                        tmem_ld32(tmem + lanes + G::T_S + hc + c0, sv);
                        tmem_ld32(tmem + lanes + G::T_P + hc + c0, pv);
                        tmem_wait_ld();
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int k = c0 + 2 * i;
                            float p0 = fast_exp2(__uint_as_float(sv[2 * i]) * c - lse2);
                            float p1 = fast_exp2(__uint_as_float(sv[2 * i + 1]) * c - lse2);
                            p0 = k < kv ? p0 : 0.f;
                            p1 = k + 1 < kv ? p1 : 0.f;
                            pk[i] = pack2b<BF16>(p0 * (__uint_as_float(pv[2 * i]) - drow),
                                                 p1 * (__uint_as_float(pv[2 * i + 1]) - drow));
                        }
                        // dS of the half's keys c0 .. c0+31 into its columns c0 .. c0+15
                        // (read already, by this thread)
                        tmem_st16(tmem + lanes + G::T_S + hc + c0, pk);
                    }
                } else {
                    // row = key row; columns = query rows tj*128 + hc .. with their
                    // own LSE and D, staged for the step in shared memory (query rows
                    // past sq get LSE = +inf, hence P = 0, and D = 0).
                    const float4 *ld4 = reinterpret_cast<const float4 *>(ldbuf);
                    // causal: this key row is seen by the tile's query columns >= cmin
                    const int cmin = CAUSAL ? grow - (a.sk - a.sq) - tj * G::BT : -1;
                    {
                        const int c0 = 32 * cg;  // this group's columns of the half
                        uint32_t sv[32], pv[32];
                        tmem_ld32(tmem + lanes + G::T_S + hc + c0, sv);
                        tmem_ld32(tmem + lanes + G::T_P + hc + c0, pv);
                        tmem_wait_ld();
                        uint32_t pp[16], pd[16];
#pragma unroll
                        for (int q = 0; q < 8; ++q) {  // four columns per shared-memory read
                            const float4 l4 = ld4[((hc + c0) >> 2) + q];
                            const float4 d4 = ld4[(G::BT >> 2) + ((hc + c0) >> 2) + q];
                            const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
                            const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
                            float pr[4], dr[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int i = 4 * q + e;
                                pr[e] = fast_exp2(__uint_as_float(sv[i]) * c - lv[e]);
                                if constexpr (CAUSAL) pr[e] = (hc + c0 + i >= cmin) ? pr[e] : 0.f;
                                dr[e] = pr[e] * (__uint_as_float(pv[i]) - dv[e]);
                            }
                            pp[2 * q] = pack2b<BF16>(pr[0], pr[1]);
                            pp[2 * q + 1] = pack2b<BF16>(pr[2], pr[3]);
                            pd[2 * q] = pack2b<BF16>(dr[0], dr[1]);
                            pd[2 * q + 1] = pack2b<BF16>(dr[2], dr[3]);
                        }
                        // P^T and dS^T of the half's columns c0 .. c0+31 into its
                        // columns c0 .. c0+15 (read already, by this thread)
                        tmem_st16(tmem + lanes + G::T_S + hc + c0, pp);
                        tmem_st16(tmem + lanes + G::T_P + hc + c0, pd);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(G::BAR_PF + h));
            }
        }

        // ---------------------------------------------------- epilogue
        const bool ok = mbar_wait(bar(G::BAR_AF), it_u & 1, g, 14);
        if (!__all_sync(0xffffffffu, ok)) return;
        tc_fence_after();
        const float scale = a.scale;
        // each group stores half of the columns (d = 16: group 0 all of them)
        constexpr int EC = D >= 32 ? D / 2 : D;
        const int e0 = D >= 32 ? cg * EC : 0;
        const bool mine = D >= 32 || cg == 0;
        if constexpr (MODE == kBwdDQ) {
            const bool out = grow < a.sq;
            uint16_t *dst = reinterpret_cast<uint16_t *>(a.dq) +
                            ((static_cast<int64_t>(x.batch) * a.sq + (out ? grow : 0)) * a.h + x.head) * D;
            if (mine) store_row<EC, BF16>(tmem + lanes + G::T_A0 + e0, scale, dst + e0, out, count == 0);
        } else {
            const bool out = grow < a.sk;
            const int64_t off =
                ((static_cast<int64_t>(x.batch) * a.sk + (out ? grow : 0)) * a.h + x.head) * D + e0;
            if (mine) {
                store_row<EC, BF16>(tmem + lanes + G::T_A0 + e0, 1.0f,
                                    reinterpret_cast<uint16_t *>(a.dv) + off, out, count == 0);
                store_row<EC, BF16>(tmem + lanes + G::T_A1 + e0, scale,
                                    reinterpret_cast<uint16_t *>(a.dk) + off, out, count == 0);
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(G::BAR_AE));
    }
}

template <int D, int MODE, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
               const BwdArgs a) {
    using G = BwdGeom<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw);
    auto bar = [&](int i) { return sbase + G::OFF_BAR + 8u * i; };

    const int warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    const int nq_t = (a.sq + G::BT - 1) / G::BT;
    const int nk_t = (a.sk + G::BT - 1) / G::BT;
    const int ntiles = MODE == kBwdDQ ? nq_t : nk_t;   // tiles that make units
    const int nsteps = MODE == kBwdDQ ? nk_t : nq_t;   // streamed tiles per unit
    const int units = ntiles * a.h * a.b;

    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + G::OFF_MISC);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + G::OFF_MISC + 4);
    if (threadIdx.x == 0) {
        for (int i = 0; i < G::NUM_BARS; ++i)
            mbar_init(bar(i), (i == G::BAR_PF || i == G::BAR_PF + 1 || i == G::BAR_AE)
                                  ? static_cast<uint32_t>(kBwdComputeWarps)  // one per compute warp
                                  : (i == G::BAR_LD || i == G::BAR_LD + 1) ? 4u  // the staging group
                                                                           : 1u);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), G::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitGuard g{abort_flag, a.status, kKernBwd};

    if (warp == 0) {
        if (lane == 0 && !(a.flags & kFlagSkipLoads)) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            tma_prefetch_desc(&tv);
            tma_prefetch_desc(&tdo);
            bwd_producer<D, MODE, CAUSAL>(&tq, &tk, &tv, &tdo, sbase, ntiles, nsteps, units, a, g);
        }
    } else if (warp == 1) {
        if (lane == 0) bwd_mma<D, MODE, BF16, CAUSAL>(sbase, tmem, ntiles, nsteps, units, a, g);
    } else if (warp >= 4 && warp < 4 + kBwdComputeWarps) {
        bwd_compute<D, MODE, BF16, CAUSAL>(smem, sbase, tmem, warp & 3, (warp - 4) >> 2, ntiles,
                                           nsteps, units, a, g);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, G::TMEM_COLS);
}

template <int D, int MODE, bool BF16, bool CAUSAL>
cudaError_t launch_bwd_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                         const CUtensorMap &tdo, const BwdArgs &a, int max_ctas,
                         cudaStream_t stream) {
    using G = BwdGeom<D>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_set[dev]) {
        e = cudaFuncSetAttribute(bwd_kernel<D, MODE, BF16, CAUSAL>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const int64_t ntiles = MODE == kBwdDQ ? (a.sq + G::BT - 1) / G::BT : (a.sk + G::BT - 1) / G::BT;
    const int64_t units = ntiles * a.h * a.b;
    const int64_t ctas = units < max_ctas ? units : max_ctas;
    bwd_kernel<D, MODE, BF16, CAUSAL>
        <<<static_cast<unsigned>(ctas), kBwdThreads, G::SMEM_BYTES, stream>>>(tq, tk, tv, tdo, a);
    return cudaGetLastError();
}

template <int D, bool BF16, bool CAUSAL>
cudaError_t launch_bwd_tiles(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                             const CUtensorMap &tdo, const BwdArgs &a, cudaStream_t stream,
                             cudaStream_t side) {
    using G = BwdGeom<D>;
    if (side == nullptr) {
        cudaError_t e = launch_bwd_t<D, kBwdDKV, BF16, CAUSAL>(tq, tk, tv, tdo, a, a.num_sms, stream);
        if (e != cudaSuccess) return e;
        return launch_bwd_t<D, kBwdDQ, BF16, CAUSAL>(tq, tk, tv, tdo, a, a.num_sms, stream);
    }
    // SM shares in proportion to the work: a key-tile step (four products)
    // costs about 1.1 times a query-tile step (three, two of them reading
    // their A operand from TMEM)
    const int64_t u_kv = (a.sk + G::BT - 1) / G::BT * a.h * a.b;
    const int64_t u_q = (a.sq + G::BT - 1) / G::BT * a.h * a.b;
    const double w_kv = 1.1 * static_cast<double>(u_kv) * a.sq, w_q = static_cast<double>(u_q) * a.sk;
    int c_kv = static_cast<int>(a.num_sms * w_kv / (w_kv + w_q) + 0.5);
    c_kv = c_kv < 1 ? 1 : (c_kv > a.num_sms - 1 ? a.num_sms - 1 : c_kv);
    int c_q = a.num_sms - c_kv;
    if (u_kv + u_q <= a.num_sms) {  // every unit has an SM of its own
        c_kv = static_cast<int>(u_kv);
        c_q = static_cast<int>(u_q);
    }
    cudaEvent_t ev_d = nullptr, ev_q = nullptr;
    cudaError_t e = cudaEventCreateWithFlags(&ev_d, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev_q, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventRecord(ev_d, stream);            // D is made
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side, ev_d, 0);
    if (e == cudaSuccess) e = launch_bwd_t<D, kBwdDKV, BF16, CAUSAL>(tq, tk, tv, tdo, a, c_kv, stream);
    if (e == cudaSuccess) e = launch_bwd_t<D, kBwdDQ, BF16, CAUSAL>(tq, tk, tv, tdo, a, c_q, side);
    // join: work queued on `stream` afterwards waits for dQ as well
    if (e == cudaSuccess) e = cudaEventRecord(ev_q, side);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, ev_q, 0);
    if (ev_d) cudaEventDestroy(ev_d);
    if (ev_q) cudaEventDestroy(ev_q);
    return e;
}

// D = rowsum(dO * O), fp32 [b, h, sq]
template <int D, bool BF16>
cudaError_t launch_dot_d(const BwdArgs &a, cudaStream_t stream) {
    constexpr int RPW = 32 / (D / 8);
    const int64_t rows = static_cast<int64_t>(a.b) * a.sq * a.h;
    const int64_t warps = (rows + RPW - 1) / RPW;
    bwd_dot_kernel<D, BF16><<<static_cast<unsigned>((warps + 7) / 8), 256, 0, stream>>>(
        static_cast<const uint16_t *>(a.o), static_cast<const uint16_t *>(a.dout), a.dvec, a.b,
        a.sq, a.h);
    return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_bwd_d(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                         const CUtensorMap &tdo, const BwdArgs &a, cudaStream_t stream,
                         cudaStream_t side) {
    // D, then dK/dV and dQ
    cudaError_t e = launch_dot_d<D, BF16>(a, stream);
    if (e != cudaSuccess) return e;
    return a.causal ? launch_bwd_tiles<D, BF16, true>(tq, tk, tv, tdo, a, stream, side)
                    : launch_bwd_tiles<D, BF16, false>(tq, tk, tv, tdo, a, stream, side);
}

}  // namespace

cudaError_t launch_bwd_dot(int d, bool bf16, const BwdArgs &a, cudaStream_t stream) {
    switch (d) {
        case 16: return bf16 ? launch_dot_d<16, true>(a, stream) : launch_dot_d<16, false>(a, stream);
        case 32: return bf16 ? launch_dot_d<32, true>(a, stream) : launch_dot_d<32, false>(a, stream);
        case 64: return bf16 ? launch_dot_d<64, true>(a, stream) : launch_dot_d<64, false>(a, stream);
        case 128:
            return bf16 ? launch_dot_d<128, true>(a, stream) : launch_dot_d<128, false>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_bwd(int d, bool bf16, const CUtensorMap &tq, const CUtensorMap &tk,
                       const CUtensorMap &tv, const CUtensorMap &tdo, const BwdArgs &a,
                       cudaStream_t stream, cudaStream_t side) {
#define EXATTN_BWD_CASE(DD)                                                      \
    case DD:                                                                     \
        return bf16 ? launch_bwd_d<DD, true>(tq, tk, tv, tdo, a, stream, side)   \
                    : launch_bwd_d<DD, false>(tq, tk, tv, tdo, a, stream, side);
    switch (d) {
        EXATTN_BWD_CASE(16)
        EXATTN_BWD_CASE(32)
        EXATTN_BWD_CASE(64)
        EXATTN_BWD_CASE(128)
        default:
            return cudaErrorInvalidValue;
    }
#undef EXATTN_BWD_CASE
}

}  // namespace exattn
