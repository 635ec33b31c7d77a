// C-ABI layer of exattn: argument validation, the split heuristic, TMA
// tensor-map encoding, the decode workspace and the device status word.
// Declared in include/exattn.h.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "exattn.h"
#include "internal.h"

using namespace exattn;

namespace exattn {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_encode_mu;
unsigned int g_flags = 0;
}  // namespace

bool load_tensor_map_encoder() {
    std::lock_guard<std::mutex> lock(g_encode_mu);
    if (g_encode != nullptr) return true;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return false;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return true;
}

unsigned int debug_flags() { return g_flags; }

static bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

attn_status_t validate_args(const void *q, const void *k, const void *v, const void *o,
                            const float *lse, int b, int sq, int sk, int h, int d, float scale,
                            int dtype) {
    if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
        return ATTN_ERR_INVALID_ARG;
    if (b < 1 || sq < 1 || sk < 1 || h < 1) return ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (dtype != ATTN_FP16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
    if (d != 16 && d != 32 && d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (b > 65535 || h > 65535) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

// (d, h, s, b) view of a contiguous [b, s, h, d] tensor; box (box0, 1, box2, 1).
bool encode_4d(CUtensorMap *map, const void *base, bool bf16, int d, int h, int s, int b,
               int box0, int box2, CUtensorMapSwizzle swizzle) {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(h),
                                static_cast<cuuint64_t>(s), static_cast<cuuint64_t>(b)};
    const cuuint64_t row = static_cast<cuuint64_t>(d) * 2;
    const cuuint64_t strides[3] = {row, row * h, row * h * static_cast<cuuint64_t>(s)};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(box0), 1u, static_cast<cuuint32_t>(box2), 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    const CUresult r = g_encode(
        map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
        const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace exattn

namespace {

constexpr int kMaxDevices = 64;
constexpr float kLog2e = 1.4426950408889634f;

struct DeviceState {
    bool ready = false;
    uint32_t *status = nullptr;  // device word written by kernels that give up a wait
    int num_sms = 0;
    // copy streams of the host-buffer forward, made on first use
    cudaStream_t s_h2d = nullptr, s_d2h = nullptr;
    // the backward's second compute stream (its query-tile kernel runs there
    // beside the key-tile kernel), made on first use
    cudaStream_t s_side = nullptr;
    // The split decode's workspace, one per stream: arrival counters of the
    // in-kernel reduce (all zero whenever a call starts) and the per-split
    // partials. Calls on one stream are ordered, so each call may reuse them.
    struct StreamWs {
        cudaStream_t stream;
        uint32_t *counters;
        int64_t n_counters;
        void *part;
        size_t part_bytes;
    };
    std::vector<StreamWs> stream_ws;
};

DeviceState g_dev[kMaxDevices];
std::mutex g_mu;
unsigned int g_last_site = 0;

}  // namespace

void exattn::record_timeout_site(unsigned int word) { g_last_site = word; }

namespace {

attn_status_t device_state(DeviceState **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &st = g_dev[dev];
    if (!st.ready) {
        if (!load_tensor_map_encoder()) return ATTN_ERR_CUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return ATTN_ERR_CUDA;
        uint32_t *status = nullptr;
        if (cudaMalloc(&status, 16) != cudaSuccess) return ATTN_ERR_NO_MEMORY;
        if (cudaMemset(status, 0, 16) != cudaSuccess) {
            cudaFree(status);
            return ATTN_ERR_CUDA;
        }
        // Keep decode workspace that was handed back cached in the pool
        // instead of returning it to the system at every synchronisation.
        cudaMemPool_t pool;
        if (cudaDeviceGetDefaultMemPool(&pool, dev) == cudaSuccess) {
            uint64_t keep = UINT64_MAX;
            cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        }
        st.status = status;
        st.num_sms = sms;
        st.ready = true;
    }
    *out = &st;
    return ATTN_OK;
}

// The two copy streams of the host-buffer forward (non-blocking, kept for the
// life of the process).
attn_status_t copy_streams(DeviceState *ds) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!ds->s_h2d && cudaStreamCreateWithFlags(&ds->s_h2d, cudaStreamNonBlocking) != cudaSuccess) {
        ds->s_h2d = nullptr;
        return ATTN_ERR_CUDA;
    }
    if (!ds->s_d2h && cudaStreamCreateWithFlags(&ds->s_d2h, cudaStreamNonBlocking) != cudaSuccess) {
        ds->s_d2h = nullptr;
        return ATTN_ERR_CUDA;
    }
    return ATTN_OK;
}

// The backward's side stream (non-blocking, kept for the life of the
// process); nullptr when `stream` is being captured into a graph or the
// stream cannot be made, and the tile kernels then run one after the other.
cudaStream_t side_stream(DeviceState *ds, cudaStream_t stream) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (cs != cudaStreamCaptureStatusNone) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!ds->s_side && cudaStreamCreateWithFlags(&ds->s_side, cudaStreamNonBlocking) != cudaSuccess) {
        cudaGetLastError();
        ds->s_side = nullptr;
    }
    return ds->s_side;
}

// The split decode's per-stream workspace: at least n zeroed arrival
// counters and part_bytes of partials, grown stream-ordered on `stream`
// (what is replaced is freed after the work already queued there). False
// while the stream is being captured into a graph, whose replays could run
// concurrently: the caller then takes a workspace per call and the separate
// reduce kernel.
bool stream_workspace(DeviceState *ds, cudaStream_t stream, int64_t n, size_t part_bytes,
                      uint32_t **counters, void **part) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (cs != cudaStreamCaptureStatusNone) return false;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState::StreamWs *e = nullptr;
    for (auto &x : ds->stream_ws)
        if (x.stream == stream) e = &x;
    if (e == nullptr) {
        ds->stream_ws.push_back(DeviceState::StreamWs{stream, nullptr, 0, nullptr, 0});
        e = &ds->stream_ws.back();
    }
    if (e->n_counters < n) {
        const int64_t cap = n < 1024 ? 1024 : n;
        uint32_t *p = nullptr;
        if (cudaMallocAsync(reinterpret_cast<void **>(&p), cap * sizeof(uint32_t), stream) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        if (cudaMemsetAsync(p, 0, cap * sizeof(uint32_t), stream) != cudaSuccess) {
            cudaFreeAsync(p, stream);
            cudaGetLastError();
            return false;
        }
        if (e->counters != nullptr) cudaFreeAsync(e->counters, stream);
        e->counters = p;
        e->n_counters = cap;
    }
    if (e->part_bytes < part_bytes) {
        const size_t cap = part_bytes < (1u << 20) ? (1u << 20) : part_bytes;
        void *p = nullptr;
        if (cudaMallocAsync(&p, cap, stream) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        if (e->part != nullptr) cudaFreeAsync(e->part, stream);
        e->part = p;
        e->part_bytes = cap;
    }
    *counters = e->counters;
    *part = e->part;
    return true;
}

CUtensorMapSwizzle fwd_swizzle(int d) {
    switch (fwd_row_bytes(d)) {
        case 128: return CU_TENSOR_MAP_SWIZZLE_128B;
        case 64: return CU_TENSOR_MAP_SWIZZLE_64B;
        default: return CU_TENSOR_MAP_SWIZZLE_32B;
    }
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Per-split partials O_i [splits, b, sq, h, d] then LSE_i [splits, b, h, sq]
// (fp32), taken stream-ordered from the device's default memory pool.
attn_status_t alloc_partials(int64_t splits, int b, int sq, int h, int d, cudaStream_t stream,
                             void **ws, float **o_part, float **lse_part) {
    const int64_t rows = static_cast<int64_t>(b) * sq * h;
    const size_t o_bytes = static_cast<size_t>(splits * rows * d) * sizeof(float);
    const size_t l_bytes = static_cast<size_t>(splits * rows) * sizeof(float);
    if (cudaMallocAsync(ws, o_bytes + l_bytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_NO_MEMORY;
    }
    *o_part = static_cast<float *>(*ws);
    *lse_part = reinterpret_cast<float *>(static_cast<char *>(*ws) + o_bytes);
    return ATTN_OK;
}

// Partials of the tensor-core kernel over key ranges: the stream's own
// workspace (kept per stream: no allocation per call), or, while the stream
// is being captured into a graph, a workspace of the call's own, returned in
// *owned for the caller to free after the reduce.
attn_status_t range_partials(DeviceState *ds, int64_t splits, int b, int sq, int h, int d,
                             cudaStream_t stream, void **owned, float **o_part, float **lse_part) {
    const int64_t rows = static_cast<int64_t>(b) * sq * h;
    const size_t o_bytes = static_cast<size_t>(splits * rows * d) * sizeof(float);
    const size_t l_bytes = static_cast<size_t>(splits * rows) * sizeof(float);
    uint32_t *counters = nullptr;
    void *part = nullptr;
    *owned = nullptr;
    if (stream_workspace(ds, stream, 1, o_bytes + l_bytes, &counters, &part)) {
        *o_part = static_cast<float *>(part);
        *lse_part = reinterpret_cast<float *>(static_cast<char *>(part) + o_bytes);
        return ATTN_OK;
    }
    return alloc_partials(splits, b, sq, h, d, stream, owned, o_part, lse_part);
}

// The CUDA-core split decode with splits > 1 (a.o, a.lse, sizes and splits
// set): the stream's own workspace and the in-kernel reduce, or, while the
// stream is being captured, a workspace of its own and the reduce kernel.
attn_status_t run_split_decode(DeviceState *ds, int d, bool bf16, const CUtensorMap &tk,
                               const CUtensorMap &tv, DecodeArgs &a, cudaStream_t stream) {
    const int64_t rows = static_cast<int64_t>(a.b) * a.sq * a.h;
    const size_t o_bytes = static_cast<size_t>(a.splits * rows * d) * sizeof(float);
    const size_t l_bytes = static_cast<size_t>(a.splits * rows) * sizeof(float);
    uint32_t *counters = nullptr;
    void *part = nullptr;
    if (stream_workspace(ds, stream, static_cast<int64_t>(a.b) * cdiv(a.sq, dec_rows_per_cta(a.sq)) * a.h,
                         o_bytes + l_bytes, &counters, &part)) {
        a.arrivals = counters;
        a.o_part = static_cast<float *>(part);
        a.lse_part = reinterpret_cast<float *>(static_cast<char *>(part) + o_bytes);
        return launch_decode(d, bf16, tk, tv, a, stream) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
    }
    void *ws = nullptr;
    attn_status_t st = alloc_partials(a.splits, a.b, a.sq, a.h, d, stream, &ws, &a.o_part, &a.lse_part);
    if (st != ATTN_OK) return st;
    a.arrivals = nullptr;
    cudaError_t e = launch_decode(d, bf16, tk, tv, a, stream);
    if (e == cudaSuccess)
        e = launch_combine(d, bf16, a.o_part, a.lse_part, static_cast<void *>(a.o), a.lse, a.b, a.sq, a.h,
                           a.splits, stream);
    const cudaError_t ef = cudaFreeAsync(ws, stream);
    return (e == cudaSuccess && ef == cudaSuccess) ? ATTN_OK : ATTN_ERR_CUDA;
}

// The tensor-core forward kernel, over all keys (splits = 1) or over key
// ranges of whole 128-key tiles whose fp32 partials the combine kernel
// reduces. A split count above the tile count is clamped, and it is lowered
// so that no split is empty.
attn_status_t run_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int b,
                      int sq, int sk, int h, int d, float scale, bool bf16, int64_t splits,
                      bool causal, DeviceState *ds, cudaStream_t stream) {
    const int64_t nkv = cdiv(sk, FWD_BN);
    if (splits > nkv) splits = nkv;
    if (splits > DEC_MAX_SPLITS) splits = DEC_MAX_SPLITS;
    if (splits < 1) splits = 1;
    const int64_t tps = cdiv(nkv, splits);
    splits = cdiv(nkv, tps);
    // work units (256 query rows of one batch, head and key range) must fit an int
    const int64_t units = cdiv(sq, FWD_BM * FWD_QTILES) * splits * h * b;
    if (units > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    const int box0 = fwd_row_bytes(d) / 2;
    CUtensorMap tq, tk, tv;
    // Short key sequences with small heads (every key of a head in one tile,
    // several tiles in flight per SM): the short forward.
    // Grouped items (head dim 16, heads in fours) once there are more
    // one-head tiles than SMs: with fewer, each tile has an SM to itself and
    // the grouped item's extra step (the block-diagonal copy, four QK^T MMAs)
    // only lengthens the one chain per SM (b2 s50 h16: 10.2 against 8.2 us).
    ShortArgs sa;
    const bool grouped_ok = cdiv(sq, SHORT_BM) * h * b > ds->num_sms;
    if (splits == 1 && !causal && !(debug_flags() & kFlagGeneralFwd) &&
        short_plan(sq, sk, h, d, grouped_ok, &sa)) {
        sa.sq = sq;
        const int64_t su = short_units(sa, b, h);
        // the CTA-local item counts (grouped: pairs times query blocks) fit an int
        if (su * (sa.grouped ? sa.nblk : 1) > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
        // grouped items read four heads at a time: the same memory viewed as
        // [b, s, h / 4, 64], 128-byte rows (one 32-row query block per box)
        const bool ok =
            sa.grouped
                ? encode_4d(&tq, q, bf16, 64, h / 4, sq, b, 64, 32, fwd_swizzle(64)) &&
                      encode_4d(&tk, k, bf16, 64, h / 4, sk, b, 64, sa.n_keys, fwd_swizzle(64)) &&
                      encode_4d(&tv, v, bf16, 64, h / 4, sk, b, 64, sa.n_keys, fwd_swizzle(64))
                : encode_4d(&tq, q, bf16, d, h, sq, b, d, SHORT_BM, fwd_swizzle(d)) &&
                      encode_4d(&tk, k, bf16, d, h, sk, b, d, sa.n_keys, fwd_swizzle(d)) &&
                      encode_4d(&tv, v, bf16, d, h, sk, b, d, sa.n_keys, fwd_swizzle(d));
        if (!ok) return ATTN_ERR_CUDA;
        sa.o = o;
        sa.lse = lse;
        sa.b = b;
        sa.sk = sk;
        sa.h = h;
        sa.scale_log2 = scale * kLog2e;
        sa.status = ds->status;
        sa.flags = debug_flags();
        // CTA c takes units c, c + grid, c + 2 grid, ...; a grid that shares
        // no factor with the tiles per head deals every CTA each tile index
        // in turn (with 2 tiles per head and 152 CTAs, half of the CTAs would
        // get only full first tiles and the other half only short last ones;
        // grouped units are all alike)
        const int64_t ntile = sa.grouped ? 1 : cdiv(sq, SHORT_BM);
        int64_t grid = su < ds->num_sms ? su : ds->num_sms;
        auto gcd = [](int64_t x, int64_t y) {
            while (y) {
                const int64_t t = x % y;
                x = y;
                y = t;
            }
            return x;
        };
        while (grid > 1 && su > grid && gcd(grid, ntile) != 1) --grid;
        return launch_fwd_short(d, bf16, tq, tk, tv, sa, static_cast<int>(grid), stream) ==
                       cudaSuccess
                   ? ATTN_OK
                   : ATTN_ERR_CUDA;
    }
    if (!encode_4d(&tq, q, bf16, d, h, sq, b, box0, FWD_BM, fwd_swizzle(d)) ||
        !encode_4d(&tk, k, bf16, d, h, sk, b, box0, FWD_BN, fwd_swizzle(d)) ||
        !encode_4d(&tv, v, bf16, d, h, sk, b, box0, FWD_BN, fwd_swizzle(d)))
        return ATTN_ERR_CUDA;
    FwdArgs a;
    a.o = o;
    a.lse = lse;
    a.b = b;
    a.sq = sq;
    a.sk = sk;
    a.h = h;
    a.scale_log2 = scale * kLog2e;
    a.status = ds->status;
    a.flags = debug_flags();
    a.num_sms = ds->num_sms;
    a.splits = static_cast<int>(splits);
    a.tiles_per_split = static_cast<int>(tps);
    a.o_part = nullptr;
    a.lse_part = nullptr;
    a.causal = causal ? 1 : 0;
    a.longest_first = causal ? 1 : 0;
    if (splits == 1)
        return launch_fwd(d, bf16, tq, tk, tv, a, stream) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
    void *ws = nullptr;
    attn_status_t st = range_partials(ds, splits, b, sq, h, d, stream, &ws, &a.o_part, &a.lse_part);
    if (st != ATTN_OK) return st;
    cudaError_t e = launch_fwd(d, bf16, tq, tk, tv, a, stream);
    if (e == cudaSuccess)
        e = launch_combine(d, bf16, a.o_part, a.lse_part, o, lse, b, sq, h, a.splits, stream);
    const cudaError_t ef = ws != nullptr ? cudaFreeAsync(ws, stream) : cudaSuccess;
    return (e == cudaSuccess && ef == cudaSuccess) ? ATTN_OK : ATTN_ERR_CUDA;
}

// Several new query rows per sequence from a paged cache: the tensor-core
// forward kernel over key ranges of whole 128-key tiles, its K/V tiles
// gathered through the block table in boxes of at most a page, with fp32
// partials reduced by the combine kernel when there is more than one split.
// Splits are chosen for the longest sequence the table allows (the lengths
// live on the device); splits past a sequence's end are empty.
attn_status_t run_fwd_paged(const void *q, const void *k_pages, const void *v_pages,
                            const int32_t *block_table, const int32_t *seqlens, void *o,
                            float *lse, int b, int sq, int h, int d, int num_pages, int page_size,
                            int max_pages, float scale, int num_splits, bool causal, bool bf16,
                            DeviceState *ds, cudaStream_t stream) {
    const int64_t sk_max = static_cast<int64_t>(max_pages) * page_size;
    const int64_t nkv = cdiv(sk_max, FWD_BN);
    int64_t splits =
        num_splits == 0
            ? attn_decode_num_splits_for_sms(b, sq, static_cast<int>(sk_max), h, d, ds->num_sms)
            : num_splits;
    if (splits > nkv) splits = nkv;
    if (splits > DEC_MAX_SPLITS) splits = DEC_MAX_SPLITS;
    if (splits < 1) splits = 1;
    const int64_t tps = cdiv(nkv, splits);
    splits = cdiv(nkv, tps);
    if (cdiv(sq, FWD_BM * FWD_QTILES) * splits * h * b > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    // boxes: the largest power of two that divides the page and the tile
    int box_rows = FWD_BN;
    while (page_size % box_rows != 0) box_rows /= 2;
    const int box0 = fwd_row_bytes(d) / 2;
    CUtensorMap tq, tk, tv;
    if (!encode_4d(&tq, q, bf16, d, h, sq, b, box0, FWD_BM, fwd_swizzle(d)) ||
        !encode_4d(&tk, k_pages, bf16, d, h, page_size, num_pages, box0, box_rows,
                   fwd_swizzle(d)) ||
        !encode_4d(&tv, v_pages, bf16, d, h, page_size, num_pages, box0, box_rows, fwd_swizzle(d)))
        return ATTN_ERR_CUDA;
    FwdArgs a;
    a.o = o;
    a.lse = lse;
    a.b = b;
    a.sq = sq;
    a.sk = static_cast<int>(sk_max);
    a.h = h;
    a.scale_log2 = scale * kLog2e;
    a.status = ds->status;
    a.flags = debug_flags();
    a.num_sms = ds->num_sms;
    a.splits = static_cast<int>(splits);
    a.tiles_per_split = static_cast<int>(tps);
    a.o_part = nullptr;
    a.lse_part = nullptr;
    a.causal = causal ? 1 : 0;
    a.longest_first = causal ? 1 : 0;
    a.block_table = block_table;
    a.seqlens = seqlens;
    a.page_size = page_size;
    a.max_pages = max_pages;
    a.num_pages = num_pages;
    a.box_rows = box_rows;
    if (splits == 1)
        return launch_fwd(d, bf16, tq, tk, tv, a, stream) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
    void *ws = nullptr;
    attn_status_t st = range_partials(ds, splits, b, sq, h, d, stream, &ws, &a.o_part, &a.lse_part);
    if (st != ATTN_OK) return st;
    cudaError_t e = launch_fwd(d, bf16, tq, tk, tv, a, stream);
    if (e == cudaSuccess)
        e = launch_combine(d, bf16, a.o_part, a.lse_part, o, lse, b, sq, h, a.splits, stream);
    const cudaError_t ef = ws != nullptr ? cudaFreeAsync(ws, stream) : cudaSuccess;
    return (e == cudaSuccess && ef == cudaSuccess) ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

namespace exattn {

int dec_num_splits(int b, int sq, int sk, int h, int d, int num_sms) {
    if (b < 1 || sq < 1 || sk < 1 || h < 1 || num_sms < 1) return 0;
    if (d != 16 && d != 32 && d != 64 && d != 128) return 0;
    const int64_t units = static_cast<int64_t>(b) * h * cdiv(sq, dec_rows_per_cta(sq));
    const int64_t nblocks = cdiv(sk, dec_block_rows(d));
    if (units >= num_sms) return 1;  // every SM already has work: no reason to split
    // Otherwise give each SM one CTA: one CTA keeps three 32 KB K/V blocks
    // requested ahead, which is enough bytes in flight per SM, and more CTAs
    // than SMs would leave a second, partial wave on some SMs. Splits are
    // never smaller than one key block.
    int64_t s = static_cast<int64_t>(num_sms) / units;
    if (s > nblocks) s = nblocks;
    if (s > 128) s = 128;
    return s < 1 ? 1 : static_cast<int>(s);
}

}  // namespace exattn

extern "C" {

int attn_version(void) { return 101; }

const char *attn_status_string(attn_status_t s) {
    switch (s) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_INVALID_ARG: return "invalid argument";
        case ATTN_ERR_UNSUPPORTED: return "unsupported size or head dim";
        case ATTN_ERR_CUDA: return "CUDA error";
        case ATTN_ERR_NO_MEMORY: return "out of device memory";
        case ATTN_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait";
    }
    return "unknown status";
}

void attn_debug_set_flags(unsigned int flags) {
    g_flags = flags & (ATTN_DEBUG_SKIP_LOADS | ATTN_DEBUG_GENERAL_FWD | ATTN_DEBUG_GENERAL_BWD);
}

unsigned int attn_last_timeout_site(void) { return g_last_site; }

attn_status_t attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int b,
                       int sq, int sk, int h, int d, float scale, attn_dtype_t dtype,
                       cudaStream_t stream) {
    attn_status_t st = validate_args(q, k, v, o, lse, b, sq, sk, h, d, scale, dtype);
    if (st != ATTN_OK) return st;
    DeviceState *ds = nullptr;
    if ((st = device_state(&ds)) != ATTN_OK) return st;
    return run_fwd(q, k, v, o, lse, b, sq, sk, h, d, scale, dtype == ATTN_BF16, 1, false, ds,
                   stream);
}

attn_status_t attn_fwd_causal(const void *q, const void *k, const void *v, void *o, float *lse,
                              int b, int sq, int sk, int h, int d, float scale, attn_dtype_t dtype,
                              cudaStream_t stream) {
    attn_status_t st = validate_args(q, k, v, o, lse, b, sq, sk, h, d, scale, dtype);
    if (st != ATTN_OK) return st;
    DeviceState *ds = nullptr;
    if ((st = device_state(&ds)) != ATTN_OK) return st;
    return run_fwd(q, k, v, o, lse, b, sq, sk, h, d, scale, dtype == ATTN_BF16, 1, true, ds,
                   stream);
}

namespace {

constexpr int kHostChunks = 8;  // most batch chunks of the host-buffer forward
constexpr int kHostRowChunks = 4;

struct HostChunk {
    int b0, nb;  // batches
    int r0, nr;  // query rows (all of them unless one batch is cut by rows)
};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

attn_status_t attn_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse,
                            int b, int sq, int sk, int h, int d, float scale, attn_dtype_t dtype,
                            int causal, cudaStream_t stream) {
    attn_status_t st = validate_args(q, k, v, o, lse, b, sq, sk, h, d, scale, dtype);
    if (st != ATTN_OK) return st;
    // The pipeline runs on the library's copy streams, joined to `stream` by
    // events: not something to record into a graph.
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    if (cs != cudaStreamCaptureStatusNone) return ATTN_ERR_UNSUPPORTED;
    DeviceState *ds = nullptr;
    if ((st = device_state(&ds)) != ATTN_OK) return st;
    if ((st = copy_streams(ds)) != ATTN_OK) return st;
    const bool bf16 = dtype == ATTN_BF16;
    const size_t row = static_cast<size_t>(h) * d * 2;  // bytes of one sequence position
    const size_t qbat = row * sq, kbat = row * sk, lbat = static_cast<size_t>(h) * sq * sizeof(float);

    // The plan (at most 8 chunks): whole batches per chunk; one batch
    // without the mask is cut into ranges of query rows (multiples of the
    // kernel's 256-row block, so every row sees the same tiles as in one
    // call), its K and V going up with the first range. (Cutting several
    // batches into row ranges as well made b4 s512 slower: 2 MB copies and
    // twice the events and launches cost more than the shorter tail gains.)
    HostChunk plan[kHostChunks];
    int n = 0;
    bool by_rows = false;
    const int blk = FWD_BM * FWD_QTILES;
    int ranges = 1;  // row ranges per batch
    if (!causal && b == 1 && sq >= 2 * blk)
        ranges = static_cast<int>(cdiv(sq, blk) < kHostRowChunks ? cdiv(sq, blk) : kHostRowChunks);
    if (ranges > 1) {
        const int per = static_cast<int>(cdiv(cdiv(sq, ranges), blk) * blk);
        for (int bb = 0; bb < b; ++bb)
            for (int r0 = 0; r0 < sq; r0 += per)
                plan[n++] = HostChunk{bb, 1, r0, sq - r0 < per ? sq - r0 : per};
        by_rows = true;
    } else if (b >= 2) {
        const int nc = b < kHostChunks ? b : kHostChunks;
        for (int i = 0; i < nc; ++i) {
            const int b0 = static_cast<int>(static_cast<int64_t>(b) * i / nc);
            const int b1 = static_cast<int>(static_cast<int64_t>(b) * (i + 1) / nc);
            plan[n++] = HostChunk{b0, b1 - b0, 0, sq};
        }
    } else {
        plan[n++] = HostChunk{0, b, 0, sq};
    }

    // Device workspace Q, K, V, O, LSE (+ with row ranges, LSE [h, rows] of
    // each chunk at [batch, h * row0]), one stream-ordered allocation on
    // `stream`.
    const size_t oq = 0, ok_ = round_up(oq + qbat * b, 256), ov = round_up(ok_ + kbat * b, 256),
                 oo = round_up(ov + kbat * b, 256), ol = round_up(oo + qbat * b, 256),
                 ot = round_up(ol + lbat * b, 256), total = ot + (by_rows ? lbat * b : 0);
    char *ws = nullptr;
    if (cudaMallocAsync(reinterpret_cast<void **>(&ws), total, stream) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_NO_MEMORY;
    }
    cudaEvent_t ev[2 * kHostChunks + 2] = {};
    const int nev = 2 * n + 2;
    bool good = true;
    for (int i = 0; i < nev && good; ++i)
        good = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) == cudaSuccess;
    cudaEvent_t ev_start = ev[2 * n], ev_end = ev[2 * n + 1];
    const char *hq = static_cast<const char *>(q), *hk = static_cast<const char *>(k),
               *hv = static_cast<const char *>(v);
    char *ho = static_cast<char *>(o);
    auto h2d = [&](size_t off_dev, const char *src, size_t bytes) {
        if (good) good = cudaMemcpyAsync(ws + off_dev, src, bytes, cudaMemcpyHostToDevice, ds->s_h2d) == cudaSuccess;
    };
    // the copy streams start after the allocation and whatever precedes the call
    if (good) good = cudaEventRecord(ev_start, stream) == cudaSuccess;
    if (good) good = cudaStreamWaitEvent(ds->s_h2d, ev_start, 0) == cudaSuccess;
    if (good) good = cudaStreamWaitEvent(ds->s_d2h, ev_start, 0) == cudaSuccess;
    for (int c = 0; c < n && good; ++c) {
        const HostChunk &x = plan[c];
        // in: K and V of the chunk's batches (with its first row range), then its Q rows
        if (x.r0 == 0) {
            h2d(ok_ + kbat * x.b0, hk + kbat * x.b0, kbat * x.nb);
            h2d(ov + kbat * x.b0, hv + kbat * x.b0, kbat * x.nb);
        }
        const size_t qoff = qbat * x.b0 + row * x.r0, qbytes = by_rows ? row * x.nr : qbat * x.nb;
        h2d(oq + qoff, hq + qoff, qbytes);
        if (good) good = cudaEventRecord(ev[2 * c], ds->s_h2d) == cudaSuccess;
        // compute on the caller's stream
        if (good) good = cudaStreamWaitEvent(stream, ev[2 * c], 0) == cudaSuccess;
        float *lse_dev = by_rows ? reinterpret_cast<float *>(ws + ot) + static_cast<size_t>(h) * sq * x.b0 +
                                       static_cast<size_t>(h) * x.r0
                                 : reinterpret_cast<float *>(ws + ol) + static_cast<size_t>(h) * sq * x.b0;
        if (good)
            good = run_fwd(ws + oq + qoff, ws + ok_ + kbat * x.b0, ws + ov + kbat * x.b0, ws + oo + qoff,
                           lse_dev, x.nb, x.nr, sk, h, d, scale, bf16, 1, causal != 0, ds,
                           stream) == ATTN_OK;
        if (good) good = cudaEventRecord(ev[2 * c + 1], stream) == cudaSuccess;
        // out: O rows and LSE on the second copy stream
        if (good) good = cudaStreamWaitEvent(ds->s_d2h, ev[2 * c + 1], 0) == cudaSuccess;
        if (good)
            good = cudaMemcpyAsync(ho + qoff, ws + oo + qoff, qbytes, cudaMemcpyDeviceToHost,
                                   ds->s_d2h) == cudaSuccess;
        if (good) {
            if (by_rows)  // LSE [h, rows] into the rows' columns of the batch's [h, sq]
                good = cudaMemcpy2DAsync(lse + static_cast<size_t>(h) * sq * x.b0 + x.r0,
                                         static_cast<size_t>(sq) * sizeof(float), lse_dev,
                                         static_cast<size_t>(x.nr) * sizeof(float),
                                         static_cast<size_t>(x.nr) * sizeof(float), h,
                                         cudaMemcpyDeviceToHost, ds->s_d2h) == cudaSuccess;
            else
                good = cudaMemcpyAsync(lse + static_cast<size_t>(h) * sq * x.b0, lse_dev, lbat * x.nb,
                                       cudaMemcpyDeviceToHost, ds->s_d2h) == cudaSuccess;
        }
    }
    // Join: the caller's stream waits for both copy streams (also after an
    // error, so that the workspace is freed only when nothing uses it).
    bool joined = ev_end != nullptr;
    if (joined) joined = cudaEventRecord(ev_end, ds->s_h2d) == cudaSuccess;
    if (joined) joined = cudaStreamWaitEvent(stream, ev_end, 0) == cudaSuccess;
    if (joined) joined = cudaEventRecord(ev_end, ds->s_d2h) == cudaSuccess;
    if (joined) joined = cudaStreamWaitEvent(stream, ev_end, 0) == cudaSuccess;
    if (!joined) {
        // without the join the copy streams may still use the workspace
        cudaStreamSynchronize(ds->s_h2d);
        cudaStreamSynchronize(ds->s_d2h);
    }
    const bool freed = cudaFreeAsync(ws, stream) == cudaSuccess;
    for (int i = 0; i < nev; ++i)
        if (ev[i]) cudaEventDestroy(ev[i]);
    return (good && joined && freed) ? ATTN_OK : ATTN_ERR_CUDA;
}

static attn_status_t run_bwd(const void *q, const void *k, const void *v, const void *o,
                             const float *lse, const void *dout, void *dq, void *dk, void *dv,
                             int b, int sq, int sk, int h, int d, float scale, attn_dtype_t dtype,
                             bool causal, cudaStream_t stream) {
    attn_status_t st = validate_args(q, k, v, o, lse, b, sq, sk, h, d, scale, dtype);
    if (st != ATTN_OK) return st;
    if (!dout || !dq || !dk || !dv || !aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) ||
        !aligned(dv, 16))
        return ATTN_ERR_INVALID_ARG;
    if (cdiv(sq, 128) * h * b > 0x7fffffffLL || cdiv(sk, 128) * h * b > 0x7fffffffLL)
        return ATTN_ERR_UNSUPPORTED;
    DeviceState *ds = nullptr;
    if ((st = device_state(&ds)) != ATTN_OK) return st;
    const bool bf16 = dtype == ATTN_BF16;
    // short problems: one kernel finishes each (batch, head); its Q / dO boxes
    // hold every query row (one or two 128-row tiles), its K / V boxes every
    // key. With fewer (batch, head) items than half the SMs it leaves most of
    // them idle, and the tile kernels, which spread one problem over several
    // CTAs, win unless the problem is a single tile on each side (b2 s150 h16
    // d16: 19.5 against 15.7 us; b2 s50: 13.7 against 15.0 us).
    const bool short_bwd = !(debug_flags() & kFlagGeneralBwd) &&
                           bwd_short_plan(sq, sk, d, causal) &&
                           (static_cast<int64_t>(b) * h * 2 >= ds->num_sms || (sq <= 128 && sk <= 128));
    const int box0 = fwd_row_bytes(d) / 2;
    const int qrows = short_bwd ? static_cast<int>(cdiv(sq, 128) * 128) : 128;
    const int krows = short_bwd ? static_cast<int>(cdiv(sk, 32) * 32) : 128;
    CUtensorMap tq, tk, tv, tdo;
    if (!encode_4d(&tq, q, bf16, d, h, sq, b, box0, qrows, fwd_swizzle(d)) ||
        !encode_4d(&tk, k, bf16, d, h, sk, b, box0, krows, fwd_swizzle(d)) ||
        !encode_4d(&tv, v, bf16, d, h, sk, b, box0, krows, fwd_swizzle(d)) ||
        !encode_4d(&tdo, dout, bf16, d, h, sq, b, box0, qrows, fwd_swizzle(d)))
        return ATTN_ERR_CUDA;
    BwdArgs a;
    a.o = o;
    a.dout = dout;
    a.lse = lse;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.b = b;
    a.sq = sq;
    a.sk = sk;
    a.h = h;
    a.scale = scale;
    a.scale_log2 = scale * kLog2e;
    a.status = ds->status;
    a.flags = debug_flags();
    a.num_sms = ds->num_sms;
    a.causal = causal ? 1 : 0;
    // D = rowsum(dO * O), fp32 [b, h, sq], from the stream-ordered pool
    void *ws = nullptr;
    if (cudaMallocAsync(&ws, static_cast<size_t>(b) * h * sq * sizeof(float), stream) !=
        cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_NO_MEMORY;
    }
    a.dvec = static_cast<float *>(ws);
    const cudaError_t e = short_bwd
                              ? launch_bwd_short(d, bf16, tq, tk, tv, tdo, a, stream)
                              : launch_bwd(d, bf16, tq, tk, tv, tdo, a, stream, side_stream(ds, stream));
    const cudaError_t ef = cudaFreeAsync(ws, stream);
    return (e == cudaSuccess && ef == cudaSuccess) ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t attn_bwd(const void *q, const void *k, const void *v, const void *o,
                       const float *lse, const void *dout, void *dq, void *dk, void *dv, int b,
                       int sq, int sk, int h, int d, float scale, attn_dtype_t dtype,
                       cudaStream_t stream) {
    return run_bwd(q, k, v, o, lse, dout, dq, dk, dv, b, sq, sk, h, d, scale, dtype, false,
                   stream);
}

attn_status_t attn_bwd_causal(const void *q, const void *k, const void *v, const void *o,
                              const float *lse, const void *dout, void *dq, void *dk, void *dv,
                              int b, int sq, int sk, int h, int d, float scale,
                              attn_dtype_t dtype, cudaStream_t stream) {
    return run_bwd(q, k, v, o, lse, dout, dq, dk, dv, b, sq, sk, h, d, scale, dtype, true,
                   stream);
}

int attn_decode_num_splits_for_sms(int b, int sq, int sk, int h, int d, int num_sms) {
    if (sq == 1) return dec_num_splits(b, sq, sk, h, d, num_sms);
    if (b < 1 || sq < 1 || sk < 1 || h < 1 || num_sms < 1) return 0;
    if (d != 16 && d != 32 && d != 64 && d != 128) return 0;
    // Several query rows: the tensor-core kernel, whose work unit is 256 query
    // rows of one (batch, head) over a range of 128-key tiles; the same rule,
    // one CTA per SM.
    const int64_t units = static_cast<int64_t>(b) * h * cdiv(sq, FWD_BM * FWD_QTILES);
    const int64_t ntiles = cdiv(sk, FWD_BN);
    if (units >= num_sms) return 1;
    int64_t s = static_cast<int64_t>(num_sms) / units;
    if (s > ntiles) s = ntiles;
    if (s > 128) s = 128;
    return s < 1 ? 1 : static_cast<int>(s);
}

int attn_decode_num_splits(int b, int sq, int sk, int h, int d) {
    DeviceState *ds = nullptr;
    if (device_state(&ds) != ATTN_OK) return 0;
    return attn_decode_num_splits_for_sms(b, sq, sk, h, d, ds->num_sms);
}

attn_status_t attn_decode_splitkv_ex(const void *q, const void *k, const void *v, void *o,
                                     float *lse, int b, int sq, int sk, int h, int d, float scale,
                                     int num_splits, attn_dtype_t dtype, cudaStream_t stream) {
    attn_status_t st = validate_args(q, k, v, o, lse, b, sq, sk, h, d, scale, dtype);
    if (st != ATTN_OK) return st;
    if (num_splits < 0) return ATTN_ERR_INVALID_ARG;
    DeviceState *ds = nullptr;
    if ((st = device_state(&ds)) != ATTN_OK) return st;
    const bool bf16 = dtype == ATTN_BF16;
    if (sq > 1) {
        // Several query rows share every K/V read in the tensor-core kernel,
        // split along the keys.
        const int64_t s = num_splits == 0
                              ? attn_decode_num_splits_for_sms(b, sq, sk, h, d, ds->num_sms)
                              : num_splits;
        return run_fwd(q, k, v, o, lse, b, sq, sk, h, d, scale, bf16, s, false, ds, stream);
    }
    const int64_t nblocks = cdiv(sk, dec_block_rows(d));
    int64_t splits = num_splits == 0
                         ? attn_decode_num_splits_for_sms(b, sq, sk, h, d, ds->num_sms)
                         : num_splits;
    if (splits > nblocks) splits = nblocks;
    if (splits > DEC_MAX_SPLITS) splits = DEC_MAX_SPLITS;
    if (splits < 1) splits = 1;

    CUtensorMap tk, tv;
    if (!encode_4d(&tk, k, bf16, d, h, sk, b, d, dec_box_rows(d), CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_4d(&tv, v, bf16, d, h, sk, b, d, dec_box_rows(d), CU_TENSOR_MAP_SWIZZLE_NONE))
        return ATTN_ERR_CUDA;

    DecodeArgs a;
    a.q = q;
    a.o = o;
    a.lse = lse;
    a.o_part = nullptr;
    a.lse_part = nullptr;
    a.b = b;
    a.sq = sq;
    a.sk = sk;
    a.h = h;
    a.splits = static_cast<int>(splits);
    a.blocks_per_split = static_cast<int>(cdiv(nblocks, splits));
    a.scale_log2 = scale * kLog2e;
    a.status = ds->status;
    a.flags = debug_flags();

    if (splits == 1)
        return launch_decode(d, bf16, tk, tv, a, stream) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;

    return run_split_decode(ds, d, bf16, tk, tv, a, stream);
}

attn_status_t attn_decode_splitkv_causal(const void *q, const void *k, const void *v, void *o,
                                         float *lse, int b, int sq, int sk, int h, int d,
                                         float scale, int num_splits, attn_dtype_t dtype,
                                         cudaStream_t stream) {
    // One query row sees every key under the bottom-right-aligned mask.
    if (sq == 1)
        return attn_decode_splitkv_ex(q, k, v, o, lse, b, sq, sk, h, d, scale, num_splits, dtype,
                                      stream);
    attn_status_t st = validate_args(q, k, v, o, lse, b, sq, sk, h, d, scale, dtype);
    if (st != ATTN_OK) return st;
    if (num_splits < 0) return ATTN_ERR_INVALID_ARG;
    DeviceState *ds = nullptr;
    if ((st = device_state(&ds)) != ATTN_OK) return st;
    const int64_t s = num_splits == 0
                          ? attn_decode_num_splits_for_sms(b, sq, sk, h, d, ds->num_sms)
                          : num_splits;
    return run_fwd(q, k, v, o, lse, b, sq, sk, h, d, scale, dtype == ATTN_BF16, s, true, ds,
                   stream);
}

attn_status_t attn_decode_paged_ex(const void *q, const void *k_pages, const void *v_pages,
                                   const int32_t *block_table, const int32_t *seqlens_k, void *o,
                                   float *lse, int b, int sq, int h, int d, int num_pages,
                                   int page_size, int max_pages_per_seq, float scale,
                                   int num_splits, int causal, attn_dtype_t dtype,
                                   cudaStream_t stream) {
    if (!block_table || !seqlens_k || !aligned(block_table, 4) || !aligned(seqlens_k, 4))
        return ATTN_ERR_INVALID_ARG;
    if (num_pages < 1 || page_size < 1 || max_pages_per_seq < 1 || num_splits < 0)
        return ATTN_ERR_INVALID_ARG;
    // TMA boxes of at most a page: page sizes are multiples of 16 keys
    if (page_size % 16 != 0) return ATTN_ERR_UNSUPPORTED;
    const int64_t sk_max = static_cast<int64_t>(max_pages_per_seq) * page_size;
    if (sk_max > 0x7fffffffLL || static_cast<int64_t>(b) * max_pages_per_seq > 0x7fffffffLL)
        return ATTN_ERR_UNSUPPORTED;
    // q [b, sq, h, d]; the pools stand in for k and v in the common checks
    attn_status_t st = validate_args(q, k_pages, v_pages, o, lse, b, sq, static_cast<int>(sk_max),
                                     h, d, scale, dtype);
    if (st != ATTN_OK) return st;
    DeviceState *ds = nullptr;
    if ((st = device_state(&ds)) != ATTN_OK) return st;
    const bool bf16 = dtype == ATTN_BF16;
    if (sq > 1) return run_fwd_paged(q, k_pages, v_pages, block_table, seqlens_k, o, lse, b, sq, h,
                                     d, num_pages, page_size, max_pages_per_seq, scale, num_splits,
                                     causal != 0, bf16, ds, stream);
    // One new row per sequence (which sees every key under the causal mask):
    // the CUDA-core split kernel. The lengths live on the device, so splits
    // are chosen for the longest sequence the table allows; splits past a
    // sequence's end are empty.
    const int64_t nblocks = cdiv(sk_max, dec_block_rows(d));
    int64_t splits = num_splits == 0
                         ? dec_num_splits(b, 1, static_cast<int>(sk_max), h, d, ds->num_sms)
                         : num_splits;
    if (splits > nblocks) splits = nblocks;
    if (splits > DEC_MAX_SPLITS) splits = DEC_MAX_SPLITS;
    if (splits < 1) splits = 1;

    // the largest power of two that divides the page and fits the kernel's box
    int box_rows = dec_box_rows(d);
    while (page_size % box_rows != 0) box_rows /= 2;
    CUtensorMap tk, tv;
    if (!encode_4d(&tk, k_pages, bf16, d, h, page_size, num_pages, d, box_rows,
                   CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_4d(&tv, v_pages, bf16, d, h, page_size, num_pages, d, box_rows,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
        return ATTN_ERR_CUDA;
    DecodeArgs a;
    a.q = q;
    a.o = o;
    a.lse = lse;
    a.o_part = nullptr;
    a.lse_part = nullptr;
    a.b = b;
    a.sq = 1;
    a.sk = static_cast<int>(sk_max);
    a.h = h;
    a.splits = static_cast<int>(splits);
    a.blocks_per_split = static_cast<int>(cdiv(nblocks, splits));
    a.scale_log2 = scale * kLog2e;
    a.status = ds->status;
    a.flags = debug_flags();
    a.block_table = block_table;
    a.seqlens = seqlens_k;
    a.page_size = page_size;
    a.max_pages = max_pages_per_seq;
    a.num_pages = num_pages;
    a.box_rows = box_rows;
    if (splits == 1)
        return launch_decode(d, bf16, tk, tv, a, stream) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
    return run_split_decode(ds, d, bf16, tk, tv, a, stream);
}

attn_status_t attn_decode_paged(const void *q, const void *k_pages, const void *v_pages,
                                const int32_t *block_table, const int32_t *seqlens_k, void *o,
                                float *lse, int b, int h, int d, int num_pages, int page_size,
                                int max_pages_per_seq, float scale, int num_splits,
                                attn_dtype_t dtype, cudaStream_t stream) {
    return attn_decode_paged_ex(q, k_pages, v_pages, block_table, seqlens_k, o, lse, b, 1, h, d,
                                num_pages, page_size, max_pages_per_seq, scale, num_splits, 0,
                                dtype, stream);
}

attn_status_t attn_decode_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                                  int b, int sq, int sk, int h, int d, float scale, int num_splits,
                                  cudaStream_t stream) {
    return attn_decode_splitkv_ex(q, k, v, o, lse, b, sq, sk, h, d, scale, num_splits, ATTN_BF16,
                                  stream);
}

attn_status_t attn_get_device_status(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
    DeviceState *ds = nullptr;
    if (device_state(&ds) != ATTN_OK) return ATTN_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, ds->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (word != 0) {
        record_timeout_site(word);
        if (cudaMemset(ds->status, 0, sizeof(word)) != cudaSuccess) return ATTN_ERR_CUDA;
        return ATTN_ERR_DEVICE_TIMEOUT;
    }
    return ATTN_OK;
}

void attn_release_workspace(void) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return;
    cudaDeviceSynchronize();
    if (dev < kMaxDevices) {
        std::lock_guard<std::mutex> lock(g_mu);
        for (auto &x : g_dev[dev].stream_ws) {
            if (x.counters) cudaFree(x.counters);
            if (x.part) cudaFree(x.part);
        }
        g_dev[dev].stream_ws.clear();
    }
    cudaMemPool_t pool;
    if (cudaDeviceGetDefaultMemPool(&pool, dev) == cudaSuccess) cudaMemPoolTrimTo(pool, 0);
}

}  // extern "C"
