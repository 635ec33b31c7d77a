// Internal interface between the C-ABI layer (api.cu) and the kernel
// translation units. Not installed; not part of the ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "exattn.h"

namespace exattn {

// ------------------------------------------------------------ forward
// One CTA owns FWD_QTILES query tiles of FWD_BM rows of one (batch, head)
// and streams the keys in tiles of FWD_BN rows.
constexpr int FWD_BM = 128;
constexpr int FWD_BN = 128;
constexpr int FWD_QTILES = 2;
constexpr int FWD_THREADS = 384;

// Bytes of one swizzled smem row of a tile (the TMA box's inner extent):
// d*2 for d <= 64 (32/64/128-byte swizzle), 128 for d = 128 (two panels).
constexpr int fwd_row_bytes(int d) { return d * 2 < 128 ? d * 2 : 128; }

struct FwdArgs {
    void *o;
    float *lse;
    int b, sq, sk, h;
    float scale_log2;  // scale * log2(e)
    uint32_t *status;
    uint32_t flags;
    int num_sms;  // persistent grid: at most one CTA per SM
    // Split along the keys: split i covers key tiles [i * tiles_per_split,
    // (i + 1) * tiles_per_split) and writes its normalised O_i and LSE_i to
    // o_part [splits, b, sq, h, d] and lse_part [splits, b, h, sq] (fp32).
    // splits == 1 writes the final o and lse.
    int splits;
    int tiles_per_split;
    float *o_part;
    float *lse_part;
    // Causal mask, bottom-right aligned: query row i sees key j only if
    // j <= i + sk - sq; rows that see no key get O = 0 and LSE = -inf.
    int causal;
    // Causal units in longest-first order across all (batch, head) pairs,
    // instead of alternating the query-block order per (batch, head).
    int longest_first;
    // Paged K/V (block_table != nullptr; key-split instantiation only): the
    // K/V maps cover page pools [num_pages, page_size, h, d]; key row r of
    // sequence bb is row r % page_size of pool page
    // block_table[bb * max_pages + r / page_size], and the sequence has
    // seqlens[bb] keys (sk is then max_pages * page_size, the most it may
    // have; the causal mask is aligned to each sequence's own count). K/V
    // tiles are loaded as boxes of box_rows rows, a power of two dividing
    // both page_size and the 128-key tile.
    const int32_t *block_table = nullptr;
    const int32_t *seqlens = nullptr;
    int page_size = 0;
    int max_pages = 0;
    int num_pages = 0;
    int box_rows = 0;
};

cudaError_t launch_fwd(int d, bool bf16, const CUtensorMap &tq, const CUtensorMap &tk,
                       const CUtensorMap &tv, const FwdArgs &a, cudaStream_t stream);

// ------------------------------------------------------------ short forward
// Forward for sk <= SHORT_MAX_KEYS and d <= 64 (fwd_short.cu): one work item
// is a 128-row query tile of one (batch, head) against all of its keys, and
// up to SHORT_MAX_SLOTS items are in flight per SM, one per TMEM slot.
constexpr int SHORT_BM = 128;
constexpr int SHORT_MAX_KEYS = 256;
constexpr int SHORT_MAX_SLOTS = 3;
constexpr int SHORT_MAX_STAGES = 8;
constexpr int SHORT_SMEM_BYTES = 220 * 1024;

struct ShortArgs {
    void *o;
    float *lse;
    int b, sq, sk, h;
    float scale_log2;  // scale * log2(e)
    uint32_t *status;
    uint32_t flags;
    // the plan (short_plan): key columns N of S (sk rounded up to 32), the
    // O accumulator's column in a slot, slot width, slots in use, bytes of
    // one K or V tile (N rows), bytes of one stage (Q + K + V), stages
    int n_keys, o_off, slot_cols, nslot, kv_bytes, stage_bytes, nstage;
    // Grouped items (head dim 16, h a multiple of 4; fwd_short.cu): a work
    // item is one 32-row query block of a group of four consecutive heads;
    // the group's K and V tiles (kv_bytes each, 128-byte rows) sit in a ring
    // of nkv_stage stages of kv_stage_bytes after the item stages. nblk:
    // query blocks per head. q_bytes: the query part of an item stage.
    int grouped, nblk, kv_stage_bytes, nkv_stage, q_bytes;
};

// Fills the plan fields of `a` for sq query rows, sk keys, h heads and
// head dim d (grouped items only if grouped_ok); false if the short
// forward does not take this shape.
bool short_plan(int sq, int sk, int h, int d, bool grouped_ok, ShortArgs *a);

// What the persistent grid deals out over b batches and h heads: plain
// items, or (batch, group of four heads) pairs when grouped.
int64_t short_units(const ShortArgs &a, int64_t b, int64_t h);

cudaError_t launch_fwd_short(int d, bool bf16, const CUtensorMap &tq, const CUtensorMap &tk,
                             const CUtensorMap &tv, const ShortArgs &a, int grid,
                             cudaStream_t stream);

// ------------------------------------------------------------ backward
struct BwdArgs {
    const void *o;      // forward output [b, sq, h, d]
    const void *dout;   // upstream gradient [b, sq, h, d]
    const float *lse;   // forward LSE [b, h, sq] (natural log)
    float *dvec;        // workspace: D = rowsum(dO * O) [b, h, sq]
    void *dq, *dk, *dv;
    int b, sq, sk, h;
    float scale;
    float scale_log2;  // scale * log2(e)
    uint32_t *status;
    uint32_t flags;
    int num_sms;
    int causal;  // the forward's bottom-right-aligned causal mask
};

// Backward for short sequences (bwd_short.cu): one (batch, head) per work
// item, all of its keys in one row of S, dQ, dK and dV finished in the CTA.
// Head dims 16 and 32, at most 256 query rows, and keys while TMEM holds S,
// dP, dQ, dK and dV (sk <= 160); not causal.
constexpr int SBWD_MAX_Q = 256;   // query rows (two 128-row tiles)
constexpr int SBWD_MAX_K = 256;   // key rows a K / V box can hold
bool bwd_short_plan(int sq, int sk, int d, bool causal);
// D = rowsum(dO * O) into a.dvec (the first kernel of every backward).
cudaError_t launch_bwd_dot(int d, bool bf16, const BwdArgs &a, cudaStream_t stream);
// The short backward proper; Q and dO maps with boxes of 128 * ceil(sq /
// 128) rows, K and V maps with boxes of sk rounded up to 32 rows.
cudaError_t launch_bwd_short(int d, bool bf16, const CUtensorMap &tq, const CUtensorMap &tk,
                             const CUtensorMap &tv, const CUtensorMap &tdo, const BwdArgs &a,
                             cudaStream_t stream);

// D, then the key-tile (dK, dV) and query-tile (dQ) kernels. With a side
// stream the two tile kernels run at the same time, on SM shares in
// proportion to their work (they are independent once D is made); without
// one they run one after the other on `stream`, each on every SM.
cudaError_t launch_bwd(int d, bool bf16, const CUtensorMap &tq, const CUtensorMap &tk,
                       const CUtensorMap &tv, const CUtensorMap &tdo, const BwdArgs &a,
                       cudaStream_t stream, cudaStream_t side);

// ------------------------------------------------------------ decode
// Keys are streamed in blocks of 16 KB per tensor (dec_block_rows(d) rows).
constexpr int DEC_BLOCK_BYTES = 16384;
constexpr int DEC_MAX_SPLITS = 1024;
constexpr int dec_block_rows(int d) { return DEC_BLOCK_BYTES / (d * 2); }
constexpr int dec_box_rows(int d) { return dec_block_rows(d) < 256 ? dec_block_rows(d) : 256; }
// Query rows handled by one CTA of the CUDA-core kernel (which runs sq == 1
// only; several rows go to the tensor-core forward kernel).
inline int dec_rows_per_cta(int sq) { return sq == 1 ? 1 : 4; }

// Split count of the CUDA-core decode kernel for num_splits = 0: 1 when the
// b * h * ceil(sq / rows per CTA) work units cover the SMs, else one CTA per
// SM (capped by the key blocks and 128). api.cu.
int dec_num_splits(int b, int sq, int sk, int h, int d, int num_sms);

struct DecodeArgs {
    const void *q;
    void *o;          // final output when splits == 1
    float *lse;       // final LSE when splits == 1
    float *o_part;    // [splits, b, sq, h, d] when splits > 1
    float *lse_part;  // [splits, b, h, sq] when splits > 1
    int b, sq, sk, h;
    int splits;
    int blocks_per_split;
    float scale_log2;
    uint32_t *status;
    uint32_t flags;
    // Paged K/V (block_table != nullptr): the K/V maps cover page pools
    // [num_pages, page_size, h, d]; key row r of sequence bb lives in page
    // block_table[bb * max_pages + r / page_size] at row r % page_size, and
    // the sequence has seqlens[bb] keys (sk above is then max_pages *
    // page_size, the most it may have).
    const int32_t *block_table = nullptr;
    const int32_t *seqlens = nullptr;
    int page_size = 0;
    int max_pages = 0;
    int num_pages = 0;
    int box_rows = 0;  // rows of one TMA box: a power of two dividing page_size
    // splits > 1: one arrival counter per (batch, query block, head), zero
    // between calls; the split that arrives last reduces the partials of its
    // rows and sets the counter back to zero. nullptr: the combine kernel
    // reduces instead.
    uint32_t *arrivals = nullptr;
};

cudaError_t launch_decode(int d, bool bf16, const CUtensorMap &tk, const CUtensorMap &tv,
                          const DecodeArgs &a, cudaStream_t stream);

cudaError_t launch_combine(int d, bool bf16, const float *o_part, const float *lse_part, void *o,
                           float *lse, int b, int sq, int h, int splits, cudaStream_t stream);

constexpr uint32_t kFlagSkipLoads = 1u;
constexpr uint32_t kFlagGeneralFwd = 2u;  // test hook: short problems take the general forward
constexpr uint32_t kFlagGeneralBwd = 4u;  // test hook: short problems take the tile backward

// ------------------------------------------------------------ host helpers (api.cu)
// None of these allocates device memory.
bool load_tensor_map_encoder();
unsigned int debug_flags();
// Remembers a status word's (kernel, site) for attn_last_timeout_site().
void record_timeout_site(unsigned int word);
attn_status_t validate_args(const void *q, const void *k, const void *v, const void *o,
                            const float *lse, int b, int sq, int sk, int h, int d, float scale,
                            int dtype);
bool encode_4d(CUtensorMap *map, const void *base, bool bf16, int d, int h, int s, int b,
               int box0, int box2, CUtensorMapSwizzle swizzle);

}  // namespace exattn
