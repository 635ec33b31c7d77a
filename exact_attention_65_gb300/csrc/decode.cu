// Split-KV decode ("flash-decoding") on sm_103a.
//
// Stage 1 (decode_split_kernel): the keys of one (batch, head) are cut into
// `splits` ranges of whole key blocks; one CTA per (split, head, batch,
// query block) streams its range of K and V through a TMA ring and runs the
// online softmax over it, writing its own O_i and LSE_i. With a single
// split it writes the final O and LSE directly.
//
// Stage 2: the reduce stated in the flash-decoding issue ("where is flash
// decoding second stage (reduce) code?"), with the max split LSE taken out
// first:
//     M = max_i LSE_i, LSE = M + ln sum_i exp(LSE_i - M),
//     O = sum_i exp(LSE_i - LSE) * O_i.
// It runs in the split kernel itself: each split CTA counts its arrival on
// a per-(batch, query block, head) counter after its partials are written,
// and the one that arrives last reduces them (no CTA waits for another). A
// separate combine_kernel does the same when no counters are given.
//
// Decode does about one multiply-add per byte of K and V, so it is bound by
// HBM bandwidth, not by math (the same issue: its speed is close to a
// memcpy, and it is split along seqlen_k only so that enough CTAs issue
// loads). The dot products therefore run on the CUDA cores in fp32; the
// design effort goes into keeping many bytes in flight: each CTA keeps
// STAGES blocks of 16 KB of K and of V requested ahead through TMA.
//
// CTA layout (288 threads): warps 0-7 consume, warp 8 is the TMA producer.
// A key row of d elements is read by d/8 lanes, 16 bytes each; a warp
// covers 32/(d/8) rows per pass and 4 passes per block. Every lane group
// keeps its own running (max, sum, output) state; the states are merged
// through shared memory at the end of the split.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace exattn {
namespace {

// ST stages of K/V blocks in flight. One split per (batch, head) streams a
// long range per CTA and gains from a fourth stage (b8 h48 sk8192: 277 ->
// 256 us); split launches, whose CTAs all start at once, lose from it.
template <int D, int ST>
struct DecGeom {
    static constexpr int LPR = D / 8;           // lanes per key row
    static constexpr int RPP = 32 / LPR;        // rows per warp pass
    static constexpr int NCW = 8;               // consumer warps
    static constexpr int THREADS = 32 * (NCW + 1);
    static constexpr int BN = dec_block_rows(D);  // key rows per block
    static constexpr int BOX_ROWS = dec_box_rows(D);
    static constexpr int BOXES = BN / BOX_ROWS;
    static constexpr int ROWS_PER_WARP = BN / NCW;
    static constexpr int PASSES = ROWS_PER_WARP / RPP;
    static constexpr int GROUPS = NCW * RPP;    // independent softmax states per query
    static constexpr int STAGES = ST;
    static constexpr int BLOCK_BYTES = BN * D * 2;
    static constexpr int STAGE_BYTES = 2 * BLOCK_BYTES;  // K block then V block
    static constexpr int OFF_BAR = STAGES * STAGE_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES;          // full[S] | empty[S]
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 128;
    static_assert(BLOCK_BYTES == DEC_BLOCK_BYTES, "block size");
    static_assert(PASSES * RPP * NCW == BN, "block coverage");
};

template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4 &w, float (&x)[8]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (BF16) {
            __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162 *>(&u[i]);
            float2 f = __bfloat1622float2(h);
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
        } else {
            __half2 h = *reinterpret_cast<const __half2 *>(&u[i]);
            float2 f = __half22float2(h);
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
        }
    }
}

template <bool BF16>
__device__ __forceinline__ uint16_t to_elem(float x) {
    if constexpr (BF16) {
        __nv_bfloat16 v = __float2bfloat16_rn(x);
        return *reinterpret_cast<uint16_t *>(&v);
    } else {
        __half v = __float2half_rn(x);
        return *reinterpret_cast<uint16_t *>(&v);
    }
}

__device__ __forceinline__ void consumer_sync(int nthreads) {
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// Barrier over the consumer warps that also ORs a predicate across them,
// so a decision taken after it is the same in every consumer warp.
__device__ __forceinline__ bool consumer_sync_any(bool pred, int nthreads) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(nthreads)
        : "memory");
    return r != 0;
}

template <int D, int ST, int QR, bool BF16, bool PAGED, typename Full, typename Empty>
__device__ __forceinline__ void decode_consume(uint8_t *smem, Full full, Empty empty, int warp,
                                               int lane, int split, int head, int batch, int q0,
                                               int nq, int blk0, int blk1, int row_end,
                                               const DecodeArgs &a, const WaitGuard &g) {
    using G = DecGeom<D, ST>;
    volatile uint32_t *abort_flag = g.abort;
    const int grp = lane / G::LPR;  // row slot within a pass
    const int sub = lane % G::LPR;  // which 8 elements of the row
    float q[QR][8];
#pragma unroll
    for (int qi = 0; qi < QR; ++qi) {
        if (qi < nq) {
            const uint16_t *qp = reinterpret_cast<const uint16_t *>(a.q) +
                                 ((static_cast<int64_t>(batch) * a.sq + q0 + qi) * a.h + head) * D +
                                 sub * 8;
            unpack8<BF16>(*reinterpret_cast<const uint4 *>(qp), q[qi]);
#pragma unroll
            for (int e = 0; e < 8; ++e) q[qi][e] *= a.scale_log2;  // scores come out in log2 units
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) q[qi][e] = 0.f;
        }
    }
    float m[QR], l[QR], o[QR][8];
#pragma unroll
    for (int qi = 0; qi < QR; ++qi) {
        m[qi] = -INFINITY;
        l[qi] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) o[qi][e] = 0.f;
    }

    bool alive = true;
    int it = 0;
    for (int blk = blk0; blk < blk1; ++blk, ++it) {
        const int s = it % G::STAGES;
        bool ok = mbar_wait(full(s), (it / G::STAGES) & 1, g, 3);
        if (!__all_sync(0xffffffffu, ok)) {
            alive = false;
            break;
        }
        const uint8_t *kb = smem + s * G::STAGE_BYTES;
        const uint8_t *vb = kb + G::BLOCK_BYTES;
        const bool tail = PAGED && (blk + 1) * G::BN > row_end;
        float x[G::PASSES][QR];
#pragma unroll
        for (int p = 0; p < G::PASSES; ++p) {
            const int r = warp * G::ROWS_PER_WARP + p * G::RPP + grp;
            float kf[8];
            unpack8<BF16>(*reinterpret_cast<const uint4 *>(kb + r * D * 2 + sub * 16), kf);
#pragma unroll
            for (int qi = 0; qi < QR; ++qi) {
                float acc = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc = fmaf(q[qi][e], kf[e], acc);
                x[p][qi] = acc;
            }
        }
#pragma unroll
        for (int off = G::LPR / 2; off >= 1; off >>= 1)
#pragma unroll
            for (int p = 0; p < G::PASSES; ++p)
#pragma unroll
                for (int qi = 0; qi < QR; ++qi)
                    x[p][qi] += __shfl_xor_sync(0xffffffffu, x[p][qi], off);
        // keys past the end of the split (zero-filled by TMA) do not take part
#pragma unroll
        for (int p = 0; p < G::PASSES; ++p) {
            const int grow = blk * G::BN + warp * G::ROWS_PER_WARP + p * G::RPP + grp;
            if (grow >= row_end)
#pragma unroll
                for (int qi = 0; qi < QR; ++qi) x[p][qi] = -INFINITY;
        }
        float pw[G::PASSES][QR];
#pragma unroll
        for (int qi = 0; qi < QR; ++qi) {
            float mb = x[0][qi];
#pragma unroll
            for (int p = 1; p < G::PASSES; ++p) mb = fmaxf(mb, x[p][qi]);
            const float m_new = fmaxf(m[qi], mb);
            if (m_new == -INFINITY) {  // nothing valid seen yet by this lane group
#pragma unroll
                for (int p = 0; p < G::PASSES; ++p) pw[p][qi] = 0.f;
                continue;
            }
            const float alpha = fast_exp2(m[qi] - m_new);
            float ps = 0.f;
#pragma unroll
            for (int p = 0; p < G::PASSES; ++p) {
                pw[p][qi] = fast_exp2(x[p][qi] - m_new);
                ps += pw[p][qi];
            }
            l[qi] = l[qi] * alpha + ps;
#pragma unroll
            for (int e = 0; e < 8; ++e) o[qi][e] *= alpha;
            m[qi] = m_new;
        }
#pragma unroll
        for (int p = 0; p < G::PASSES; ++p) {
            const int r = warp * G::ROWS_PER_WARP + p * G::RPP + grp;
            float vf[8];
            unpack8<BF16>(*reinterpret_cast<const uint4 *>(vb + r * D * 2 + sub * 16), vf);
            // Rows past the split's last key weigh 0; a paged cache's last page
            // holds stale data there, which must not reach O even as 0 * NaN.
            // Only the split's last block can hold such rows. (A contiguous
            // cache has TMA zero fill there.)
            if constexpr (PAGED) {
                if (tail && blk * G::BN + r >= row_end)
#pragma unroll
                    for (int e = 0; e < 8; ++e) vf[e] = 0.f;
            }
#pragma unroll
            for (int qi = 0; qi < QR; ++qi)
#pragma unroll
                for (int e = 0; e < 8; ++e) o[qi][e] = fmaf(pw[p][qi], vf[e], o[qi][e]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(s));
    }

    // The reduce grid may begin launching now; it waits for this grid to
    // complete before it reads any partial.
    griddep_launch_dependents();

    // ---------------------------------------- merge the lane-group states
    // All consumers are past their last read of the ring before it is reused,
    // and all of them agree on whether the split was abandoned.
    if (consumer_sync_any(!alive || *abort_flag != 0u, G::NCW * 32)) return;
    float *red_m = reinterpret_cast<float *>(smem);                 // [QR][GROUPS]
    float *red_l = red_m + QR * G::GROUPS;                          // [QR][GROUPS]
    float *red_w = red_l + QR * G::GROUPS;                          // [QR][GROUPS] weights
    float *red_lse = red_w + QR * G::GROUPS;                        // [QR]
    float *red_o = red_lse + 4 * ((QR + 3) / 4);                    // [QR][GROUPS][D]
    const int gidx = warp * G::RPP + grp;
#pragma unroll
    for (int qi = 0; qi < QR; ++qi) {
        if (sub == 0) {
            red_m[qi * G::GROUPS + gidx] = m[qi];
            red_l[qi * G::GROUPS + gidx] = l[qi];
        }
        float4 *dst = reinterpret_cast<float4 *>(red_o + (qi * G::GROUPS + gidx) * D + sub * 8);
        dst[0] = make_float4(o[qi][0], o[qi][1], o[qi][2], o[qi][3]);
        dst[1] = make_float4(o[qi][4], o[qi][5], o[qi][6], o[qi][7]);
    }
    consumer_sync(G::NCW * 32);
    // one warp per query row: global max, total sum, per-group weights, LSE
    if (warp < nq) {
        const int qi = warp;
        float mx = -INFINITY;
        for (int gi = lane; gi < G::GROUPS; gi += 32) mx = fmaxf(mx, red_m[qi * G::GROUPS + gi]);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        float tot = 0.f;
        for (int gi = lane; gi < G::GROUPS; gi += 32) {
            const float mg = red_m[qi * G::GROUPS + gi];
            tot += (mg == -INFINITY) ? 0.f : red_l[qi * G::GROUPS + gi] * fast_exp2(mg - mx);
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
        const bool empty_split = (mx == -INFINITY);
        const float inv = empty_split ? 0.f : 1.0f / tot;
        for (int gi = lane; gi < G::GROUPS; gi += 32) {
            const float mg = red_m[qi * G::GROUPS + gi];
            red_w[qi * G::GROUPS + gi] = (mg == -INFINITY) ? 0.f : fast_exp2(mg - mx) * inv;
        }
        if (lane == 0)
            red_lse[qi] = empty_split ? -INFINITY : (mx + __log2f(tot)) * 0.69314718055994530942f;
    }
    consumer_sync(G::NCW * 32);
    for (int idx = threadIdx.x; idx < nq * D; idx += G::NCW * 32) {
        const int qi = idx / D, dd = idx % D;
        float acc = 0.f;
        for (int gi = 0; gi < G::GROUPS; ++gi)
            acc = fmaf(red_w[qi * G::GROUPS + gi], red_o[(qi * G::GROUPS + gi) * D + dd], acc);
        const int qrow = q0 + qi;
        if (a.splits == 1) {
            uint16_t *op = reinterpret_cast<uint16_t *>(a.o);
            op[((static_cast<int64_t>(batch) * a.sq + qrow) * a.h + head) * D + dd] = to_elem<BF16>(acc);
        } else {
            a.o_part[((((static_cast<int64_t>(split) * a.b + batch) * a.sq + qrow) * a.h + head) * D) +
                     dd] = acc;
        }
    }
    if (threadIdx.x < nq) {
        const int qrow = q0 + threadIdx.x;
        const float v = red_lse[threadIdx.x];
        if (a.splits == 1)
            a.lse[(static_cast<int64_t>(batch) * a.h + head) * a.sq + qrow] = v;
        else
            a.lse_part[((static_cast<int64_t>(split) * a.b + batch) * a.h + head) * a.sq + qrow] = v;
    }
}

// Many splits: lane i holds LSE_i of the splits i, i+32, ...; every load is
// independent of the ones before it, so the warp keeps many in flight
// instead of paying one memory latency per split. Returns LSE; acc gets O.
template <int D>
__device__ __forceinline__ float combine_many(const float *__restrict__ lse_part,
                                              const float *__restrict__ src, int64_t lse_idx,
                                              int64_t lse_stride, int64_t o_stride, int splits,
                                              int lane, float (&acc)[D >= 32 ? D / 32 : 1]) {
    constexpr int PER = D >= 32 ? D / 32 : 1;
    constexpr float kLog2e = 1.4426950408889634f;
    float mx = -INFINITY;
#pragma unroll 4
    for (int i = lane; i < splits; i += 32) mx = fmaxf(mx, __ldcg(lse_part + i * lse_stride + lse_idx));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float tot = 0.f;
#pragma unroll 4
    for (int i = lane; i < splits; i += 32) {
        const float li = __ldcg(lse_part + i * lse_stride + lse_idx);
        tot += (li == -INFINITY) ? 0.f : fast_exp2((li - mx) * kLog2e);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
    const float L = mx + __logf(tot);
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    for (int i0 = 0; i0 < splits; i0 += 32) {
        // weight of split i0 + lane (0 for an empty split or past the end)
        const float li =
            (i0 + lane < splits) ? __ldcg(lse_part + (i0 + lane) * lse_stride + lse_idx) : -INFINITY;
        const float wl = (li == -INFINITY) ? 0.f : fast_exp2((li - L) * kLog2e);
        const int n = min(32, splits - i0);
#pragma unroll 8
        for (int j = 0; j < n; ++j) {
            const float w = __shfl_sync(0xffffffffu, wl, j);
#pragma unroll
            for (int e = 0; e < PER; ++e)
                acc[e] = fmaf(w, __ldcg(src + (i0 + j) * o_stride + 32 * e), acc[e]);
        }
    }
    return L;
}

// The reduce of one output row (batch, query row, head) by one warp. The
// partials are read through L2 only (other CTAs wrote them).
template <int D, bool BF16>
__device__ __forceinline__ void combine_row(const float *__restrict__ o_part,
                                            const float *__restrict__ lse_part, void *o, float *lse,
                                            int b, int sq, int h, int splits, int batch, int qrow,
                                            int head, int lane) {
    constexpr int PER = D >= 32 ? D / 32 : 1;
    const int64_t rows = static_cast<int64_t>(b) * sq * h;
    const int64_t r = (static_cast<int64_t>(batch) * sq + qrow) * h + head;
    const int64_t lse_idx = (static_cast<int64_t>(batch) * h + head) * sq + qrow;
    const int64_t lse_stride = static_cast<int64_t>(b) * h * sq;
    const int64_t o_stride = rows * D;
    constexpr float kLog2e = 1.4426950408889634f;

    const bool active = D >= 32 || lane < D;
    const float *src = o_part + r * D + (active ? lane : 0);
    float acc[PER];
    float L;
    constexpr int kFew = 16;
    if (splits <= kFew) {
        // Few splits: lane i holds LSE_i, and every partial of the row is
        // requested at once, so the reduce waits for one memory latency.
        const float li = lane < splits ? __ldcg(lse_part + lane * lse_stride + lse_idx) : -INFINITY;
        float ov[kFew][PER];
#pragma unroll
        for (int i = 0; i < kFew; ++i)
#pragma unroll
            for (int e = 0; e < PER; ++e) ov[i][e] = i < splits ? __ldcg(src + i * o_stride + 32 * e) : 0.f;
        float mx = li;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        float tot = (li == -INFINITY) ? 0.f : fast_exp2((li - mx) * kLog2e);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
        L = mx + __logf(tot);
        const float wl = (li == -INFINITY) ? 0.f : fast_exp2((li - L) * kLog2e);
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[e] = 0.f;
#pragma unroll
        for (int i = 0; i < kFew; ++i) {
            const float w = __shfl_sync(0xffffffffu, wl, i);  // 0 past the last split
#pragma unroll
            for (int e = 0; e < PER; ++e) acc[e] = fmaf(w, ov[i][e], acc[e]);
        }
    } else {
        L = combine_many<D>(lse_part, src, lse_idx, lse_stride, o_stride, splits, lane, acc);
    }
    if (active) {
        uint16_t *dst = reinterpret_cast<uint16_t *>(o) + r * D;
#pragma unroll
        for (int e = 0; e < PER; ++e) dst[lane + 32 * e] = to_elem<BF16>(acc[e]);
    }
    if (lane == 0) lse[lse_idx] = L;
}

template <int D, int ST, int QR, bool BF16, bool PAGED>
__global__ void __launch_bounds__(DecGeom<D, ST>::THREADS)
    decode_split_kernel(const __grid_constant__ CUtensorMap tk,
                        const __grid_constant__ CUtensorMap tv, const DecodeArgs a) {
    using G = DecGeom<D, ST>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 127u) & ~127u;
    uint8_t *smem = smem_raw + (sbase - raw);
    auto full = [&](int s) { return sbase + G::OFF_BAR + 8u * s; };
    auto empty = [&](int s) { return sbase + G::OFF_BAR + 8u * (G::STAGES + s); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int split = blockIdx.x, head = blockIdx.y;
    const int nqb = (a.sq + QR - 1) / QR;
    const int batch = blockIdx.z / nqb;
    const int q0 = (blockIdx.z % nqb) * QR;
    const int nq = min(QR, a.sq - q0);
    // keys of this sequence: sk, or its own length with a paged cache
    int sk_b = a.sk;
    if constexpr (PAGED) sk_b = min(max(a.seqlens[batch], 0), a.sk);
    const int nblocks = (sk_b + G::BN - 1) / G::BN;
    const int blk0 = split * a.blocks_per_split;
    const int blk1 = min(nblocks, blk0 + a.blocks_per_split);
    const int row_end = min(sk_b, blk1 * G::BN);

    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + G::OFF_MISC);
    if (threadIdx.x == 0) {
        for (int s = 0; s < G::STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), G::NCW);
        }
        *abort_flag = 0u;
        fence_mbar_init();
    }
    __syncthreads();
    const WaitGuard g{abort_flag, a.status, kKernDecode};

    if (warp == G::NCW) {
        // ---------------------------------------------------- producer
        if (PAGED && !(a.flags & kFlagSkipLoads)) {
            // A paged cache's blocks are gathered as boxes of at most a page
            // (box_rows, a power of two dividing page_size, so none crosses a
            // page), one box per lane: the block-table lookups and TMA issues
            // of a block run side by side (a 64-key block of 16-key pages is
            // four boxes per tensor). Lane 0 waits for the stage and arms it.
            // Rows past the sequence's end are masked by the consumers; their
            // page index is only kept in range.
            if (lane == 0) {
                tma_prefetch_desc(&tk);
                tma_prefetch_desc(&tv);
            }
            const uint64_t stream_once = policy_evict_first();
            const int boxes = G::BN / a.box_rows;  // at most 32
            int issued = 0;
            for (int blk = blk0; blk < blk1; ++blk, ++issued) {
                const int s = issued % G::STAGES;
                const uint32_t ph = (issued / G::STAGES) & 1;
                int r = blk * G::BN + lane * a.box_rows;
                int outer = 0;
                if (static_cast<int>(lane) < boxes) {
                    const int lp = min(r / a.page_size, a.max_pages - 1);
                    const int pg = __ldg(a.block_table + static_cast<int64_t>(batch) * a.max_pages + lp);
                    outer = min(max(pg, 0), a.num_pages - 1);
                    r -= lp * a.page_size;
                }
                bool got = true;
                if (lane == 0) {
                    got = mbar_wait(empty(s), ph ^ 1, g, 1);
                    if (got) mbar_arrive_expect_tx(full(s), G::STAGE_BYTES);
                }
                if (!__shfl_sync(0xffffffffu, got, 0)) break;
                if (static_cast<int>(lane) < boxes) {
                    const uint32_t dst = sbase + s * G::STAGE_BYTES + lane * a.box_rows * D * 2;
                    tma_load_4d_hint(dst, &tk, full(s), 0, head, r, outer, stream_once);
                    tma_load_4d_hint(dst + G::BLOCK_BYTES, &tv, full(s), 0, head, r, outer,
                                     stream_once);
                }
                __syncwarp();
            }
            if (lane == 0) {
                WaitGuard drain = g;
                uint32_t no_abort = 0;
                drain.abort = &no_abort;
                for (int i = (issued > G::STAGES ? issued - G::STAGES : 0); i < issued; ++i)
                    mbar_wait(full(i % G::STAGES), (i / G::STAGES) & 1, drain, 2);
            }
        } else if (!PAGED && lane == 0 && !(a.flags & kFlagSkipLoads)) {
            tma_prefetch_desc(&tk);
            tma_prefetch_desc(&tv);
            const uint64_t stream_once = policy_evict_first();
            int issued = 0;
            for (int blk = blk0; blk < blk1; ++blk, ++issued) {
                const int s = issued % G::STAGES;
                const uint32_t ph = (issued / G::STAGES) & 1;
                if (!mbar_wait(empty(s), ph ^ 1, g, 1)) break;
                mbar_arrive_expect_tx(full(s), G::STAGE_BYTES);
                const uint32_t dst = sbase + s * G::STAGE_BYTES;
#pragma unroll
                for (int x = 0; x < G::BOXES; ++x) {
                    const int r = blk * G::BN + x * G::BOX_ROWS;
                    tma_load_4d_hint(dst + x * G::BOX_ROWS * D * 2, &tk, full(s), 0, head, r, batch,
                                     stream_once);
                    tma_load_4d_hint(dst + G::BLOCK_BYTES + x * G::BOX_ROWS * D * 2, &tv, full(s), 0,
                                     head, r, batch, stream_once);
                }
            }
            WaitGuard drain = g;
            uint32_t no_abort = 0;
            drain.abort = &no_abort;
            for (int i = (issued > G::STAGES ? issued - G::STAGES : 0); i < issued; ++i)
                mbar_wait(full(i % G::STAGES), (i / G::STAGES) & 1, drain, 2);
        }
    } else {
        decode_consume<D, ST, QR, BF16, PAGED>(smem, full, empty, warp, lane, split, head, batch, q0,
                                               nq, blk0, blk1, row_end, a, g);
    }
    __syncthreads();

    // ---------------------------------------- reduce by the last split
    // Every CTA counts its arrival once its partials are written (also after
    // an abort, so that the counter still comes back to zero). The fence
    // orders the CTA's partial stores, which thread 0 has observed through
    // the barrier, before the count; the last arriver fences again before it
    // reads the others' partials.
    if (a.splits > 1 && a.arrivals != nullptr) {
        volatile uint32_t *is_last = reinterpret_cast<volatile uint32_t *>(smem + G::OFF_MISC + 8);
        if (threadIdx.x == 0) {
            __threadfence();
            uint32_t *cnt = a.arrivals + static_cast<int64_t>(blockIdx.z) * a.h + head;
            const bool last = atomicAdd(cnt, 1u) == static_cast<uint32_t>(a.splits - 1);
            if (last) {
                atomicExch(cnt, 0u);  // every split has counted: ready for the next call
                __threadfence();
            }
            *is_last = last ? 1u : 0u;
        }
        __syncthreads();
        if (*is_last && warp < nq)
            combine_row<D, BF16>(a.o_part, a.lse_part, a.o, a.lse, a.b, a.sq, a.h, a.splits, batch,
                                 q0 + warp, head, lane);
    }
}

// One warp per output row (batch, query row, head).
template <int D, bool BF16>
__global__ void __launch_bounds__(128)
    combine_kernel(const float *__restrict__ o_part, const float *__restrict__ lse_part, void *o,
                   float *lse, int b, int sq, int h, int splits) {
    const int lane = threadIdx.x & 31;
    const int64_t rows = static_cast<int64_t>(b) * sq * h;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
    if (r >= rows) return;
    const int head = static_cast<int>(r % h);
    const int qrow = static_cast<int>((r / h) % sq);
    const int batch = static_cast<int>(r / (static_cast<int64_t>(h) * sq));
    // The partials come from the split kernel, which may still be draining
    // when this grid starts (programmatic dependent launch).
    griddep_wait();
    combine_row<D, BF16>(o_part, lse_part, o, lse, b, sq, h, splits, batch, qrow, head, lane);
}

template <int D, int ST, int QR, bool BF16, bool PAGED>
cudaError_t launch_decode_t(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeArgs &a,
                            cudaStream_t stream) {
    using G = DecGeom<D, ST>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_set[dev]) {
        e = cudaFuncSetAttribute(decode_split_kernel<D, ST, QR, BF16, PAGED>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const int nqb = (a.sq + QR - 1) / QR;
    dim3 grid(a.splits, a.h, a.b * nqb);
    decode_split_kernel<D, ST, QR, BF16, PAGED><<<grid, G::THREADS, G::SMEM_BYTES, stream>>>(tk, tv, a);
    return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_decode_d(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeArgs &a,
                            cudaStream_t stream) {
    const bool deep = a.splits == 1;
    if (a.block_table)  // sq == 1
        return deep ? launch_decode_t<D, 4, 1, BF16, true>(tk, tv, a, stream)
                    : launch_decode_t<D, 3, 1, BF16, true>(tk, tv, a, stream);
    // Several query rows run on the tensor-core forward kernel instead.
    if (a.sq != 1) return cudaErrorNotSupported;
    return deep ? launch_decode_t<D, 4, 1, BF16, false>(tk, tv, a, stream)
                : launch_decode_t<D, 3, 1, BF16, false>(tk, tv, a, stream);
}

template <int D, bool BF16>
cudaError_t launch_combine_t(const float *o_part, const float *lse_part, void *o, float *lse, int b,
                             int sq, int h, int splits, cudaStream_t stream) {
    const int64_t rows = static_cast<int64_t>(b) * sq * h;
    // Programmatic dependent launch: this grid is set up while the split
    // grid drains; griddep_wait() inside orders the memory accesses.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((rows + 3) / 4));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel<D, BF16>, o_part, lse_part, o, lse, b, sq, h,
                              splits);
}

}  // namespace

cudaError_t launch_decode(int d, bool bf16, const CUtensorMap &tk, const CUtensorMap &tv,
                          const DecodeArgs &a, cudaStream_t stream) {
#define EXATTN_DEC_CASE(DD)                                           \
    case DD:                                                          \
        return bf16 ? launch_decode_d<DD, true>(tk, tv, a, stream)    \
                    : launch_decode_d<DD, false>(tk, tv, a, stream);
    switch (d) {
        EXATTN_DEC_CASE(16)
        EXATTN_DEC_CASE(32)
        EXATTN_DEC_CASE(64)
        EXATTN_DEC_CASE(128)
        default:
            return cudaErrorInvalidValue;
    }
#undef EXATTN_DEC_CASE
}

cudaError_t launch_combine(int d, bool bf16, const float *o_part, const float *lse_part, void *o,
                           float *lse, int b, int sq, int h, int splits, cudaStream_t stream) {
#define EXATTN_CMB_CASE(DD)                                                                  \
    case DD:                                                                                 \
        return bf16 ? launch_combine_t<DD, true>(o_part, lse_part, o, lse, b, sq, h, splits, \
                                                 stream)                                     \
                    : launch_combine_t<DD, false>(o_part, lse_part, o, lse, b, sq, h, splits, \
                                                  stream);
    switch (d) {
        EXATTN_CMB_CASE(16)
        EXATTN_CMB_CASE(32)
        EXATTN_CMB_CASE(64)
        EXATTN_CMB_CASE(128)
        default:
            return cudaErrorInvalidValue;
    }
#undef EXATTN_CMB_CASE
}

}  // namespace exattn
