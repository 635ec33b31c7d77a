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
// its keys. Persistent CTAs (one per SM) deal their items to two or three
// TMEM slots, so several items are in flight per SM and the latency chain of each
// (loads, QK^T, softmax, PV, store) overlaps the others':
//   warp 0        TMA producer: Q tile, K and V of the item into a ring of
//                 shared-memory stages.
//   warp 1        TMEM owner and MMA issuer (one thread): S = Q K^T into the
//                 item's slot, later O = P V into the same slot.
//   warps 2-3     idle.
//   warps 4..     one softmax warpgroup per slot (the kernel is compiled
//                 for 2 and 3 slots); warpgroup g owns slot g, and thread i
//                 of warp w owns row 32 (w % 4) + i of its tile.
// TMEM slot g spans columns [g W, g W + W): S in [0, N) (N = sk rounded up
// to 32), overwritten by P two 16-bit keys per column in [0, N/2), and the
// O accumulator in [o_off, o_off + d) once S has been read.
// The softmax reads S once, 64 columns at a time, with the lazy reference
// max of the general forward: the first 64 columns set it, and a later pair
// of chunks whose max exceeds it by more than 8 (log2 units) moves it and
// rescales the P already stored (rare). So no thread holds a whole score
// row and each chunk costs one TMEM round trip.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace exattn {
namespace {

constexpr int SH_WG = SHORT_MAX_SLOTS;          // most softmax warpgroups
constexpr int SH_MAX_CHUNKS = SHORT_MAX_KEYS / 32;
constexpr int SH_BAR_BYTES = 1024;             // barriers and flags, before the tiles

// barriers: full[stages] | empty[stages] | s_full[slots] | p_full[slots] |
//           o_full[slots] | free[slots] | done
constexpr int BAR_FULL = 0;
constexpr int BAR_EMPTY = BAR_FULL + SHORT_MAX_STAGES;
constexpr int BAR_SF = BAR_EMPTY + SHORT_MAX_STAGES;
constexpr int BAR_PF = BAR_SF + SH_WG;
constexpr int BAR_OF = BAR_PF + SH_WG;
constexpr int BAR_FREE = BAR_OF + SH_WG;
constexpr int BAR_DONE = BAR_FREE + SH_WG;
constexpr int NUM_BARS = BAR_DONE + 1;
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

// Folds one 32-column chunk of raw scores into four running maxima (minima
// when scale < 0). MASK: only the first `valid` columns are keys.
template <bool MASK, bool POS>
__device__ __forceinline__ void chunk_extreme(const uint32_t (&r)[32], int valid, float (&mx)[4]) {
    const float *s = reinterpret_cast<const float *>(r);
    const float pad = POS ? -INFINITY : INFINITY;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        const float x0 = (!MASK || 2 * e < valid) ? s[2 * e] : pad;
        const float x1 = (!MASK || 2 * e + 1 < valid) ? s[2 * e + 1] : pad;
        mx[e & 3] = POS ? max3f(mx[e & 3], x0, x1) : min3f(mx[e & 3], x0, x1);
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
        tma_load_4d(dst + G::Q_BYTES, tk, bar(BAR_FULL + st), 0, x.head, 0, x.batch);
        tma_load_4d(dst + G::Q_BYTES + a.kv_bytes, tv, bar(BAR_FULL + st), 0, x.head, 0, x.batch);
    }
    // Never leave the CTA with a copy still landing in shared memory.
    WaitGuard drain = g;
    uint32_t no_abort = 0;
    drain.abort = &no_abort;
    for (int m = (n > a.nstage ? n - a.nstage : 0); m < n; ++m)
        mbar_wait(bar(BAR_FULL + m % a.nstage), (m / a.nstage) & 1, drain, 21);
}

template <int D, bool BF16>
__device__ __forceinline__ void short_mma(uint32_t sbase, uint32_t tiles, uint32_t tmem,
                                          int n_items, const ShortArgs &a, const WaitGuard &g) {
    using G = ShortGeom<D>;
    auto bar = [&](int i) { return sbase + 8u * i; };
    const uint32_t idesc_s = mma_idesc_f16(SHORT_BM, a.n_keys, BF16, false, false);
    constexpr uint32_t idesc_o = mma_idesc_f16(SHORT_BM, D, BF16, false, true);
    const uint64_t dk = smem_desc(tiles, 16, G::SBO, G::LAYOUT);  // Q and K, K-major
    // V, MN-major; d spans one swizzle atom, so the leading offset is not
    // stepped through (it is set to the tile size, like a panel stride)
    const uint64_t dv = smem_desc(tiles, a.kv_bytes, G::SBO, G::LAYOUT);
    const int kv_steps = a.n_keys / 16;
    // Two queues in item order: QK^T for the next item whose stage has landed
    // and whose slot the epilogue of the item nslot back has handed back, and
    // P V for the oldest item whose P is stored. Polled without blocking, so
    // neither queue waits behind the other's barrier; the wait is bounded
    // like every other (no progress for the bound, or a CTA-wide abort).
    int s_next = 0, p_next = 0;
    uint64_t t0 = global_timer_ns();
    uint32_t polls = 0;
    while (p_next < n_items) {
        bool progressed = false;
        if (s_next < n_items && s_next - p_next < a.nslot) {
            const int sl = s_next % a.nslot, st = s_next % a.nstage;
            if (mbar_test_wait(bar(BAR_FULL + st), (s_next / a.nstage) & 1) &&
                (s_next < a.nslot ||
                 mbar_test_wait(bar(BAR_FREE + sl), ((s_next / a.nslot) - 1) & 1))) {
                tc_fence_after();
                const uint32_t tS = tmem + sl * a.slot_cols;
                const uint64_t qd = dk + ((st * a.stage_bytes) >> 4);
                const uint64_t kd = qd + (G::Q_BYTES >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(tS, qd + kk * 2, kd + kk * 2, idesc_s, kk > 0 ? 1u : 0u);
                mma_commit(bar(BAR_SF + sl));
                ++s_next;
                progressed = true;
            }
        }
        if (p_next < s_next) {
            const int sl = p_next % a.nslot, st = p_next % a.nstage;
            if (mbar_test_wait(bar(BAR_PF + sl), (p_next / a.nslot) & 1)) {
                tc_fence_after();
                const uint32_t tS = tmem + sl * a.slot_cols;
                const uint64_t vd = dv + ((st * a.stage_bytes + G::Q_BYTES + a.kv_bytes) >> 4);
                for (int kk = 0; kk < kv_steps; ++kk)
                    mma_ts(tS + a.o_off, tS + kk * 8, vd + ((kk * 16 * G::ROW_BYTES) >> 4), idesc_o,
                           kk > 0 ? 1u : 0u);
                mma_commit(bar(BAR_OF + sl));
                mma_commit(bar(BAR_EMPTY + st));
                ++p_next;
                progressed = true;
            }
        }
        if (progressed) {
            t0 = global_timer_ns();
            polls = 0;
        } else if ((++polls & 15u) == 0u) {
            if (*g.abort) break;
            if (global_timer_ns() - t0 > kWaitTimeoutNs || polls >= kWaitMaxPolls) {
                *g.abort = 1u;
                atomicCAS(g.status, 0u, (g.kernel << 8) | 22u);
                break;
            }
        }
    }
    // No MMA may still be running when TMEM is released.
    mma_commit(bar(BAR_DONE));
    WaitGuard drain = g;
    uint32_t no_abort = 0;
    drain.abort = &no_abort;
    mbar_wait(bar(BAR_DONE), 0, drain, 25);
}

template <int D, bool BF16>
__device__ __forceinline__ void short_softmax(uint32_t sbase, uint32_t tmem, int sl, int q4,
                                              int n_items, int ntile, const ShortArgs &a,
                                              const WaitGuard &g) {
    auto bar = [&](int i) { return sbase + 8u * i; };
    const uint32_t lane = threadIdx.x & 31;
    const int row = q4 * 32 + lane;
    const uint32_t tS = tmem + sl * a.slot_cols + (static_cast<uint32_t>(q4 * 32) << 16);
    const uint32_t tO = tS + a.o_off;
    const float c = a.scale_log2;
    const bool c_pos = c >= 0.f;
    const int nch = a.n_keys / 32;
    // keys of the last 32-column chunk that exist (1..32)
    const int last_valid = a.sk - 32 * (nch - 1);
    const bool o_al32 = (reinterpret_cast<uintptr_t>(a.o) & 31u) == 0;

    int k = 0;
    for (int i = sl; i < n_items; i += a.nslot, ++k) {
        const Item x = item_of(blockIdx.x + i * gridDim.x, ntile, a.h);
        const int grow = x.tile * SHORT_BM + row;
        const bool warp_live = x.tile * SHORT_BM + q4 * 32 < a.sq;
        const bool ok = mbar_wait(bar(BAR_SF + sl), k & 1, g, 26);
        if (!__all_sync(0xffffffffu, ok)) return;
        tc_fence_after();

        float m_ref = -INFINITY, l = 1.f;
        if (warp_live) {
            // One pass over S, two 32-column chunks per TMEM round trip: the
            // pair's max (of the raw scores, their min if scale < 0) moves the
            // reference max only past the lazy threshold; then its P is
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
                    for (int q = 0; q < 4; ++q) mx[q] = c_pos ? -INFINITY : INFINITY;
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int cc = ch + h2;
                        if (cc < nch) {
                            const bool ragged = cc == nch - 1 && last_valid < 32;
                            if (c_pos) {
                                if (ragged) chunk_extreme<true, true>(r[h2], last_valid, mx);
                                else chunk_extreme<false, true>(r[h2], 32, mx);
                            } else {
                                if (ragged) chunk_extreme<true, false>(r[h2], last_valid, mx);
                                else chunk_extreme<false, false>(r[h2], 32, mx);
                            }
                        }
                    }
                    const float mraw = c_pos ? fmaxf(max3f(mx[0], mx[1], mx[2]), mx[3])
                                             : fminf(min3f(mx[0], mx[1], mx[2]), mx[3]);
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
        const bool okf = mbar_wait(bar(BAR_OF + sl), k & 1, g, 27);
        if (!__all_sync(0xffffffffu, okf)) return;
        tc_fence_after();
        // O row read out 32 columns at a time (16 at d = 16); the slot goes
        // back to the MMA issuer as soon as the last piece is in registers,
        // before that piece is scaled, packed and stored
        constexpr int OCH = D < 32 ? D : 32;
        const bool row_out = warp_live && grow < a.sq;
        const float inv_l = 1.0f / l;
        const int64_t orow =
            ((static_cast<int64_t>(x.batch) * a.sq + (row_out ? grow : 0)) * a.h + x.head) * D;
        uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(a.o) + orow);
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += OCH) {
            uint32_t ov[OCH];
            if (warp_live) {
                if constexpr (OCH == 32)
                    tmem_ld32(tO + c0, *reinterpret_cast<uint32_t(*)[32]>(ov));
                else
                    tmem_ld16(tO + c0, *reinterpret_cast<uint32_t(*)[16]>(ov));
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
            a.lse[(static_cast<int64_t>(x.batch) * a.h + x.head) * a.sq + grow] =
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

template <int D, bool BF16, int NWG>
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
    const int items = ntile * a.h * a.b;
    const int n_items =
        blockIdx.x < items ? (items - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;

    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + OFF_MISC + 4);
    if (threadIdx.x == 0) {
        for (int i = 0; i < NUM_BARS; ++i) {
            const bool by_warps = (i >= BAR_PF && i < BAR_PF + SH_WG) ||
                                  (i >= BAR_FREE && i < BAR_FREE + SH_WG);
            mbar_init(bar(i), by_warps ? 4u : 1u);  // one arrive per softmax warp
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
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitGuard g{abort_flag, a.status, kKernFwd};

    if (warp < 4) {
        if constexpr (NWG == 3) reg_dealloc<kShortRegsControl>();
        if (warp == 0) {
            if (lane == 0 && !(a.flags & kFlagSkipLoads))
                short_producer<D>(&tq, &tk, &tv, sbase, tiles, items, ntile, a, g);
        } else if (warp == 1) {
            if (lane == 0) short_mma<D, BF16>(sbase, tiles, tmem, n_items, a, g);
        }
    } else {
        if constexpr (NWG == 3) reg_alloc<kShortRegsSoftmax>();
        short_softmax<D, BF16>(sbase, tmem, (warp - 4) >> 2, warp & 3, n_items, ntile, a, g);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int D, bool BF16, int NWG>
cudaError_t launch_short_w(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                           const ShortArgs &a, int grid, cudaStream_t stream) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_set[dev]) {
        e = cudaFuncSetAttribute(fwd_short_kernel<D, BF16, NWG>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, SHORT_SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    fwd_short_kernel<D, BF16, NWG>
        <<<grid, 128 * (NWG + 1), SHORT_SMEM_BYTES, stream>>>(tq, tk, tv, a);
    return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_short_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                           const ShortArgs &a, int grid, cudaStream_t stream) {
    switch (a.nslot) {
        case 2: return launch_short_w<D, BF16, 2>(tq, tk, tv, a, grid, stream);
        case 3: return launch_short_w<D, BF16, 3>(tq, tk, tv, a, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool short_plan(int sk, int d, ShortArgs *a) {
    if (sk < 1 || sk > SHORT_MAX_KEYS || (d != 16 && d != 32 && d != 64)) return false;
    const int n = (sk + 31) / 32 * 32;
    const int row_bytes = d * 2;
    const int o_off = (n / 2 + 31) / 32 * 32;
    int w = n > o_off + d ? n : o_off + d;
    w = (w + 31) / 32 * 32;
    int slots = 512 / w;
    if (slots > SHORT_MAX_SLOTS) slots = SHORT_MAX_SLOTS;
    const int kv_bytes = n * row_bytes;
    const int stage_bytes = SHORT_BM * row_bytes + 2 * kv_bytes;  // a multiple of 1024
    int stages = (SHORT_SMEM_BYTES - 1024 - SH_BAR_BYTES) / stage_bytes;
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
    return true;
}

cudaError_t launch_fwd_short(int d, bool bf16, const CUtensorMap &tq, const CUtensorMap &tk,
                             const CUtensorMap &tv, const ShortArgs &a, int grid,
                             cudaStream_t stream) {
#define EXATTN_SHORT_CASE(DD)                                                \
    case DD:                                                                 \
        return bf16 ? launch_short_t<DD, true>(tq, tk, tv, a, grid, stream)  \
                    : launch_short_t<DD, false>(tq, tk, tv, a, grid, stream);
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
