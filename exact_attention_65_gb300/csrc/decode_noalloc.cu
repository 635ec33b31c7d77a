// Split-KV decode for callers that cannot allocate device memory.
//
// attn_decode_splitkv_ex takes its per-split partials (O_i, LSE_i) from the
// device's memory pool. Some callers must not allocate at all once they are
// running: an application whose device memory is entirely owned by its own
// allocator or pool, code under a hard memory budget, or real-time code that
// forbids allocation after start-up. This entry point serves them: the
// partials live in one fixed array compiled into the library, and nothing
// here calls cudaMalloc, cudaMallocAsync, cudaFree or any allocating routine.
// The kernels are the ones the allocating entry point launches: the CUDA-core
// split kernel for one query row, the tensor-core forward kernel split along
// the keys for several, each followed by the combine kernel.
#include <cstdint>
#include <mutex>

#include "exattn.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = ATTN_NOALLOC_SCRATCH_BYTES;
constexpr size_t kAlign = 256;
constexpr int kMaxDevices = 64;
constexpr float kLog2e = 1.4426950408889634f;

// Every GPU that loads the library holds these until the process exits.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];
// Bounded-wait status word of this entry point's kernels. Zero when the
// module loads; attn_get_noalloc_status() clears it after each report.
static __device__ __align__(16) uint32_t g_status[4];

struct Slot {
    bool ready = false;
    unsigned char *scratch = nullptr;  // device address of g_scratch on this device
    uint32_t *status = nullptr;        // device address of g_status on this device
    int num_sms = 0;
};

Slot g_slots[kMaxDevices];
std::mutex g_mu;

// Once per device, with that device current: look up the device addresses of
// the arrays (the host-side names are only stand-ins, not device addresses).
attn_status_t setup(Slot **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    Slot &s = g_slots[dev];
    if (!s.ready) {
        void *scratch = nullptr;
        void *status = nullptr;
        if (cudaGetSymbolAddress(&scratch, g_scratch) != cudaSuccess) return ATTN_ERR_CUDA;
        if (cudaGetSymbolAddress(&status, g_status) != cudaSuccess) return ATTN_ERR_CUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return ATTN_ERR_CUDA;
        if (!exattn::load_tensor_map_encoder()) return ATTN_ERR_CUDA;
        s.scratch = static_cast<unsigned char *>(scratch);
        s.status = static_cast<uint32_t *>(status);
        s.num_sms = sms;
        s.ready = true;
    }
    *out = &s;
    return ATTN_OK;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Partials O_i [splits, b, sq, h, d] then LSE_i [splits, b, h, sq], fp32,
// each part starting on a 256-byte boundary of the array; false if they do
// not fit.
bool carve(const Slot &slot, int64_t splits, int b, int sq, int h, int d, float **o_part,
           float **lse_part) {
    const int64_t rows = static_cast<int64_t>(b) * sq * h;
    const size_t o_bytes = round_up(static_cast<size_t>(splits * rows * d) * sizeof(float));
    const size_t l_bytes = round_up(static_cast<size_t>(splits * rows) * sizeof(float));
    if (o_bytes + l_bytes > kScratchBytes) return false;
    *o_part = reinterpret_cast<float *>(slot.scratch);
    *lse_part = reinterpret_cast<float *>(slot.scratch + o_bytes);
    return true;
}

CUtensorMapSwizzle fwd_swizzle(int d) {
    switch (exattn::fwd_row_bytes(d)) {
        case 128: return CU_TENSOR_MAP_SWIZZLE_128B;
        case 64: return CU_TENSOR_MAP_SWIZZLE_64B;
        default: return CU_TENSOR_MAP_SWIZZLE_32B;
    }
}

// sq > 1: the tensor-core forward kernel over ranges of whole 128-key tiles
// (every query row of a head shares each K/V read), partials in the array,
// then the combine kernel. The split count follows the allocating entry
// point: clamped to the tile count and lowered so that no split is empty.
attn_status_t run_rows(const Slot &slot, const void *q, const void *k, const void *v, void *o,
                       float *lse, int b, int sq, int sk, int h, int d, float scale,
                       int num_splits, bool bf16, cudaStream_t stream) {
    using namespace exattn;
    const int64_t nkv = cdiv(sk, FWD_BN);
    int64_t splits = num_splits == 0
                         ? attn_decode_num_splits_for_sms(b, sq, sk, h, d, slot.num_sms)
                         : num_splits;
    if (splits > nkv) splits = nkv;
    if (splits > DEC_MAX_SPLITS) splits = DEC_MAX_SPLITS;
    if (splits < 1) splits = 1;
    const int64_t tps = cdiv(nkv, splits);
    splits = cdiv(nkv, tps);
    if (cdiv(sq, FWD_BM * FWD_QTILES) * splits * h * b > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    FwdArgs a;
    a.o = o;
    a.lse = lse;
    a.o_part = nullptr;
    a.lse_part = nullptr;
    if (splits > 1 && !carve(slot, splits, b, sq, h, d, &a.o_part, &a.lse_part))
        return ATTN_ERR_UNSUPPORTED;
    const int box0 = fwd_row_bytes(d) / 2;
    CUtensorMap tq, tk, tv;
    if (!encode_4d(&tq, q, bf16, d, h, sq, b, box0, FWD_BM, fwd_swizzle(d)) ||
        !encode_4d(&tk, k, bf16, d, h, sk, b, box0, FWD_BN, fwd_swizzle(d)) ||
        !encode_4d(&tv, v, bf16, d, h, sk, b, box0, FWD_BN, fwd_swizzle(d)))
        return ATTN_ERR_CUDA;
    a.b = b;
    a.sq = sq;
    a.sk = sk;
    a.h = h;
    a.scale_log2 = scale * kLog2e;
    a.status = slot.status;
    a.flags = debug_flags();
    a.num_sms = slot.num_sms;
    a.splits = static_cast<int>(splits);
    a.tiles_per_split = static_cast<int>(tps);
    a.causal = 0;
    a.longest_first = 0;
    // Every split writes all of its O_i and LSE_i, so nothing left in the
    // array by an earlier call is read.
    cudaError_t e = launch_fwd(d, bf16, tq, tk, tv, a, stream);
    if (e == cudaSuccess && splits > 1)
        e = launch_combine(d, bf16, a.o_part, a.lse_part, o, lse, b, sq, h, a.splits, stream);
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// sq == 1: the CUDA-core split kernel (key blocks of 16 KB per tensor), its
// partials in the array, then the combine kernel.
attn_status_t run_one_row(const Slot &slot, const void *q, const void *k, const void *v, void *o,
                          float *lse, int b, int sk, int h, int d, float scale, int num_splits,
                          bool bf16, cudaStream_t stream) {
    using namespace exattn;
    const int64_t nblocks = cdiv(sk, dec_block_rows(d));
    int64_t splits = num_splits == 0 ? dec_num_splits(b, 1, sk, h, d, slot.num_sms) : num_splits;
    if (splits > nblocks) splits = nblocks;
    if (splits > DEC_MAX_SPLITS) splits = DEC_MAX_SPLITS;
    if (splits < 1) splits = 1;
    DecodeArgs a;
    a.o_part = nullptr;
    a.lse_part = nullptr;
    if (splits > 1 && !carve(slot, splits, b, 1, h, d, &a.o_part, &a.lse_part))
        return ATTN_ERR_UNSUPPORTED;
    CUtensorMap tk, tv;
    if (!encode_4d(&tk, k, bf16, d, h, sk, b, d, dec_box_rows(d), CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_4d(&tv, v, bf16, d, h, sk, b, d, dec_box_rows(d), CU_TENSOR_MAP_SWIZZLE_NONE))
        return ATTN_ERR_CUDA;
    a.q = q;
    a.o = o;
    a.lse = lse;
    a.b = b;
    a.sq = 1;
    a.sk = sk;
    a.h = h;
    a.splits = static_cast<int>(splits);
    a.blocks_per_split = static_cast<int>(cdiv(nblocks, splits));
    a.scale_log2 = scale * kLog2e;
    a.status = slot.status;
    a.flags = debug_flags();
    // Every split writes all of its O_i and LSE_i (an empty split writes 0
    // and -inf), so nothing left in the array by an earlier call is read.
    cudaError_t e = launch_decode(d, bf16, tk, tv, a, stream);
    if (e == cudaSuccess && splits > 1)
        e = launch_combine(d, bf16, a.o_part, a.lse_part, o, lse, b, 1, h, a.splits, stream);
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

extern "C" attn_status_t attn_decode_splitkv_noalloc(const void *q, const void *k, const void *v,
                                                     void *o, float *lse, int b, int sq, int sk,
                                                     int h, int d, float scale, int num_splits,
                                                     attn_dtype_t dtype, cudaStream_t stream) {
    using namespace exattn;
    attn_status_t st = validate_args(q, k, v, o, lse, b, sq, sk, h, d, scale, dtype);
    if (st != ATTN_OK) return st;
    if (num_splits < 0) return ATTN_ERR_INVALID_ARG;
    Slot *slot = nullptr;
    if ((st = setup(&slot)) != ATTN_OK) return st;
    const bool bf16 = dtype == ATTN_BF16;
    if (sq > 1)
        return run_rows(*slot, q, k, v, o, lse, b, sq, sk, h, d, scale, num_splits, bf16, stream);
    return run_one_row(*slot, q, k, v, o, lse, b, sk, h, d, scale, num_splits, bf16, stream);
}

extern "C" attn_status_t attn_get_noalloc_status(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    uint32_t *status = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_slots[dev].ready) return ATTN_OK;  // nothing has run here
        status = g_slots[dev].status;
    }
    uint32_t word = 0;
    if (cudaMemcpy(&word, status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (word == 0) return ATTN_OK;
    exattn::record_timeout_site(word);
    const uint32_t zero = 0;
    if (cudaMemcpy(status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_ERR_DEVICE_TIMEOUT;
}
