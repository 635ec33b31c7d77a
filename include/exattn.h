/*
 * exattn -- exact scaled-dot-product attention on one GB300 (sm_103a).
 *
 * C ABI. Every entry point takes plain pointers and sizes; no C++ or
 * framework types cross it and no exception leaves it.
 *
 * Common conventions
 *   Layout   q, o: [b, sq, h, d]; k, v: [b, sk, h, d]; contiguous, d
 *            innermost (the (b, s, h, d) layout "Why FlashAttention is
 *            fast" section 2 item 2 says flash_attn_func consumes directly,
 *            so no transposes are needed). lse: [b, h, sq], fp32.
 *   Memory   q, k, v, o, lse are DEVICE pointers on the current CUDA device
 *            (attn_fwd_host alone takes host pointers), owned by the caller;
 *            the library never frees or keeps them. q, k, v, o must be
 *            16-byte aligned, lse 4-byte aligned.
 *   Streams  every compute call is asynchronous on `stream` (0 = legacy
 *            default stream). Argument errors are returned before anything
 *            is enqueued. A wait inside a kernel that exceeds its bound
 *            (about two seconds) ends the kernel early and records a device
 *            status word; attn_get_device_status() reports it.
 *   Math     O = softmax(scale * Q K^T) V row by row, with fp32 accumulation
 *            and an online (running max / running sum) softmax, so the
 *            score matrix never reaches global memory ("Why FlashAttention
 *            is fast", sections 3.1-3.3). LSE[b, h, i] = ln sum_j
 *            exp(scale * q_i . k_j), natural log, of the scaled scores.
 *            O is rounded to nearest even into the input dtype.
 *   Sizes    b, sq, sk, h >= 1; d in {16, 32, 64, 128}; scale finite
 *            (0 and negative values are accepted). b and h at most 65535.
 */
#ifndef EXATTN_H
#define EXATTN_H

#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { ATTN_FP16 = 0, ATTN_BF16 = 1 } attn_dtype_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, size < 1, non-finite scale, bad dtype */
    ATTN_ERR_UNSUPPORTED = 2,    /* d outside {16, 32, 64, 128}, or a size beyond the grid limits */
    ATTN_ERR_CUDA = 3,           /* a CUDA runtime/driver call failed (launch, tensor-map encode, ...) */
    ATTN_ERR_NO_MEMORY = 4,      /* a workspace (decode partials, backward, host forward) could not be allocated */
    ATTN_ERR_DEVICE_TIMEOUT = 5  /* a kernel gave up on a bounded wait (see attn_get_device_status) */
} attn_status_t;

/*
 * Forward attention: O and LSE for every query row.
 * Defined by "Why FlashAttention is fast" section 2 item 4 (S = Q K^T * scale,
 * softmax, times V; the call flash_attn_func(q, k, v) of item 5), computed
 * tile by tile with the online softmax of section 3.3. Non-causal, no
 * dropout. dtype selects fp16 or bf16 for q, k, v and o.
 * Inputs are taken to be finite: at d = 16 with h a multiple of 4, heads
 * are computed four at a time in one tile, and a key holding an infinity
 * or a NaN also turns the rows of the other three heads of its group to
 * NaN.
 * Returns ATTN_OK once the kernel is enqueued on `stream`.
 */
attn_status_t attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                       int b, int sq, int sk, int h, int d, float scale,
                       attn_dtype_t dtype, cudaStream_t stream);

/*
 * attn_fwd with a causal mask. Causal masking is not on the pages; the mask
 * is the bottom-right-aligned one: query row i (of sq) sees key j (of sk)
 * only if j <= i + sk - sq, so with sq == sk row i sees keys 0..i, and with
 * sq < sk the last query row sees every key (new tokens appended to a
 * cache). Rows that see no key (i < sq - sk) get O = 0 and LSE = -inf.
 * Key tiles wholly past a query tile's last visible key are skipped.
 * Arguments, layouts and errors are those of attn_fwd.
 */
attn_status_t attn_fwd_causal(const void *q, const void *k, const void *v, void *o, float *lse,
                              int b, int sq, int sk, int h, int d, float scale,
                              attn_dtype_t dtype, cudaStream_t stream);

/*
 * attn_fwd (causal != 0: attn_fwd_causal) on HOST buffers: q, k, v, o, lse
 * as in attn_fwd but in host memory, 16-byte aligned; pinned memory
 * (cudaHostAlloc, cudaHostRegister) lets the copies overlap, pageable
 * memory works but its copies serialise with the host. The call runs a
 * copy / compute / copy-back pipeline: the problem is cut into chunks of
 * whole batches (at most 8), or, for one non-causal batch of at least 512
 * query rows, into at most 4 ranges of query rows that are multiples of 256
 * (K and V go first); the chunk's inputs go up on a library copy stream,
 * its forward runs on `stream`, and its O and LSE come back on a second
 * copy stream while the next chunk goes up. Results are bit-identical to
 * attn_fwd on device copies of the same inputs. Device workspace for all
 * five tensors is taken stream-ordered from the device's default memory
 * pool on `stream` and returned. The call is stream-ordered on `stream`:
 * it starts after the work already queued there, and work queued there
 * afterwards starts once every copy-back is done, so o and lse may be read
 * after `stream` is synchronised (the host buffers must stay valid until
 * then). Errors as attn_fwd; ATTN_ERR_NO_MEMORY if the workspace cannot be
 * had; ATTN_ERR_UNSUPPORTED while `stream` is being captured into a graph
 * (the pipeline runs on the library's own copy streams).
 */
attn_status_t attn_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse,
                            int b, int sq, int sk, int h, int d, float scale, attn_dtype_t dtype,
                            int causal, cudaStream_t stream);

/*
 * Backward pass of attn_fwd (non-causal): dq, dk, dv from q, k, v, the
 * forward's o and lse, and the upstream gradient dout. The flash-attn timing
 * issue times a backward pass; none of the pages writes one out, so it is
 * the chain rule of the forward's definition: with P = exp(scale Q K^T - LSE),
 *     dV = P^T dO,  dP = dO V^T,  D = rowsum(dO * O),  dS = P * (dP - D),
 *     dQ = scale dS K,  dK = scale dS^T Q.
 *   q, o, dout, dq   [b, sq, h, d]; k, v, dk, dv [b, sk, h, d]; lse fp32
 *                    [b, h, sq] as written by attn_fwd; all in `dtype`
 *                    except lse, device pointers, 16-byte aligned.
 * Every output element is written. A workspace of 4 * b * h * sq bytes is
 * taken stream-ordered from the device's default memory pool and returned.
 * The key-tile (dK, dV) and query-tile (dQ) kernels run at the same time,
 * the second on a library stream forked from and joined back to `stream` by
 * events (one after the other on `stream` while it is being captured into a
 * graph); the call stays stream-ordered on `stream`. Short problems (d 16
 * or 32, sq <= 256, sk <= 160, not causal, with b * h at least half the SM
 * count or sq, sk <= 128) run one kernel instead, which finishes each
 * (batch, head) in one CTA (all of its keys in one row of S).
 * Errors as attn_fwd; ATTN_ERR_NO_MEMORY if the workspace cannot be had.
 */
attn_status_t attn_bwd(const void *q, const void *k, const void *v, const void *o,
                       const float *lse, const void *dout, void *dq, void *dk, void *dv,
                       int b, int sq, int sk, int h, int d, float scale, attn_dtype_t dtype,
                       cudaStream_t stream);

/*
 * Backward pass of attn_fwd_causal: the same chain rule with P = 0 wherever
 * the forward's bottom-right-aligned mask hides a key (key j of row i is
 * hidden when j > i + sk - sq). lse must be the one attn_fwd_causal wrote
 * (-inf for rows that see no key; those rows get dq = 0, and keys that no
 * row sees get dk = dv = 0). Tiles that the mask hides wholly are skipped.
 * Arguments, layouts, workspace and errors are those of attn_bwd.
 */
attn_status_t attn_bwd_causal(const void *q, const void *k, const void *v, const void *o,
                              const float *lse, const void *dout, void *dq, void *dk, void *dv,
                              int b, int sq, int sk, int h, int d, float scale,
                              attn_dtype_t dtype, cudaStream_t stream);

/*
 * Split-KV decode, bf16 q/k/v/o ("where is flash decoding second stage
 * (reduce) code?" issue). seqlen_k is cut into num_splits ranges of whole
 * key blocks; split i writes its own O_i and LSE_i (fp32, library
 * workspace), and the reduce forms, with the max LSE taken out first,
 *     LSE = log(sum_i exp(LSE_i)),   O = sum_i exp(LSE_i - LSE) * O_i.
 * With sq == 1 the reduce runs inside the split kernel: the split of a
 * (batch, head) that finishes last reduces it, found through arrival
 * counters (zero between calls) that the library keeps per stream together
 * with the partials (calls on a stream are ordered, so each reuses them;
 * grown stream-ordered on demand, freed by attn_release_workspace). With
 * sq > 1 the partials come from the same per-stream workspace and a second
 * kernel reduces them. While the stream is being captured into a graph, the
 * partials are taken per call as below and the second kernel reduces.
 * num_splits = 0 lets attn_decode_num_splits() choose; a positive value is
 * clamped to the number of key blocks. With one split the first kernel
 * writes O and LSE directly and no workspace is used. Any sq >= 1 is
 * accepted (non-causal). With sq == 1 the splits run on a CUDA-core kernel
 * (key blocks of 16 KB per tensor). With sq > 1 they run on the tensor-core
 * forward kernel, so each K/V byte is read once for all query rows of a
 * head (the issue's case of 1 to 10 new tokens); its key blocks are tiles of
 * 128 keys and a requested count is lowered so that no split is empty.
 * Under graph capture the per-call workspace is taken stream-ordered from
 * the device's default memory pool and returned after the reduce; it is
 * kept cached in the pool until attn_release_workspace().
 */
attn_status_t attn_decode_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                                  int b, int sq, int sk, int h, int d, float scale,
                                  int num_splits, cudaStream_t stream);

/* attn_decode_splitkv with an explicit dtype (fp16 or bf16). */
attn_status_t attn_decode_splitkv_ex(const void *q, const void *k, const void *v, void *o, float *lse,
                                     int b, int sq, int sk, int h, int d, float scale,
                                     int num_splits, attn_dtype_t dtype, cudaStream_t stream);

/*
 * attn_decode_splitkv_ex with the causal mask of attn_fwd_causal (bottom-right
 * aligned: the sq new query rows are the last sq positions of the sk keys).
 * With sq == 1 it is attn_decode_splitkv_ex. Splits wholly past a query
 * row's last visible key contribute nothing to it (LSE_i = -inf).
 */
attn_status_t attn_decode_splitkv_causal(const void *q, const void *k, const void *v, void *o,
                                         float *lse, int b, int sq, int sk, int h, int d,
                                         float scale, int num_splits, attn_dtype_t dtype,
                                         cudaStream_t stream);

/*
 * Split-KV decode of new query rows from a paged KV cache. Paged caches are
 * not on the pages beyond a mention ("Why FlashAttention is fast", section
 * 5, item 2: FlashAttention with a paged KV cache is the standard for long
 * contexts); the layout read here is the common one.
 *   q            [b, sq, h, d] (device, 16-byte aligned): the sq new rows of
 *                each sequence (the flash-decoding issue's 1 to 10 new tokens)
 *   k_pages,
 *   v_pages      page pools [num_pages, page_size, h, d] (device, 16-byte
 *                aligned); page_size must be a multiple of 16
 *                (ATTN_ERR_UNSUPPORTED otherwise)
 *   block_table  int32 [b, max_pages_per_seq] (device): logical page p of
 *                sequence i is pool page block_table[i * max_pages_per_seq + p]
 *   seqlens_k    int32 [b] (device): keys of sequence i, 0 <= seqlens_k[i]
 *                <= max_pages_per_seq * page_size (values outside are
 *                clamped; entries of the table past a sequence's last page
 *                are not used)
 *   o, lse       [b, sq, h, d] and fp32 [b, h, sq]
 *   causal       non-zero: the bottom-right-aligned mask of attn_fwd_causal,
 *                aligned to each sequence's own key count (row r of sequence
 *                i sees key j only if j <= r + seqlens_k[i] - sq); rows that
 *                see no key get O = 0 and LSE = -inf
 * With sq == 1 the splits run on the CUDA-core kernel (pages read in boxes of
 * at most a page); with sq > 1 on the tensor-core forward kernel, whose
 * 128-key tiles are gathered from the pages and whose rows past a
 * sequence's end are zero-filled or zeroed in shared memory, so stale page
 * data (even NaN) never reaches O. The split count (num_splits = 0: the
 * heuristic of attn_decode_num_splits) is chosen for the longest allowed
 * sequence, since the lengths are only known on the device; splits past a
 * sequence's end are empty. A sequence with no key gets O = 0 and
 * LSE = -inf. The reduce, the workspace and the errors are those of
 * attn_decode_splitkv_ex.
 */
attn_status_t attn_decode_paged_ex(const void *q, const void *k_pages, const void *v_pages,
                                   const int32_t *block_table, const int32_t *seqlens_k, void *o,
                                   float *lse, int b, int sq, int h, int d, int num_pages,
                                   int page_size, int max_pages_per_seq, float scale,
                                   int num_splits, int causal, attn_dtype_t dtype,
                                   cudaStream_t stream);

/* attn_decode_paged_ex with one new row per sequence (sq = 1, q [b, 1, h, d]). */
attn_status_t attn_decode_paged(const void *q, const void *k_pages, const void *v_pages,
                                const int32_t *block_table, const int32_t *seqlens_k, void *o,
                                float *lse, int b, int h, int d, int num_pages, int page_size,
                                int max_pages_per_seq, float scale, int num_splits,
                                attn_dtype_t dtype, cudaStream_t stream);

/*
 * Split-KV decode that allocates no device memory. The pages have no
 * counterpart: this is a library convenience, not part of the method.
 *
 * For callers that cannot call cudaMalloc once they are running: an
 * application whose device memory is all owned by its own allocator or pool,
 * code under a fixed memory budget, or real-time code that forbids
 * allocation after start-up. attn_decode_splitkv_ex takes its per-split
 * partials from the device's memory pool; this entry point keeps them in
 * one fixed scratch array of ATTN_NOALLOC_SCRATCH_BYTES compiled into the
 * library instead, and calls no cudaMalloc, cudaFree or other allocating
 * routine. Every GPU that loads the library holds that array until the
 * process exits.
 *
 * Arguments, layouts and results are those of attn_decode_splitkv_ex; the
 * caller still passes all inputs and outputs. The kernels are the same:
 * with sq == 1 the CUDA-core split kernel, with sq > 1 the tensor-core
 * forward kernel split along the keys (tiles of 128 keys, a requested count
 * lowered so that no split is empty), each followed by the combine kernel;
 * num_splits = 0 picks the count attn_decode_num_splits() reports. With more
 * than one split the partials need 4 * splits * b * sq * h * (d + 1) bytes
 * (each part rounded up to 256); a request that needs more than the array
 * holds returns ATTN_ERR_UNSUPPORTED before anything is enqueued.
 *
 * The first call on a device does a one-time set-up (it looks up the
 * array's device address; nothing is written); make that first call before
 * any stream capture. All calls share the one array, which keeps the last
 * call's contents (every split rewrites all of its partials, so none is
 * read stale): calls that overlap on the GPU, from different streams or
 * host threads, race on it and must be serialised by the caller. A
 * bounded-wait timeout in this entry point's kernels is recorded in a
 * status word of its own, read by attn_get_noalloc_status(), not by
 * attn_get_device_status() (whose first use allocates its word).
 */
#define ATTN_NOALLOC_SCRATCH_BYTES (8u << 20)
attn_status_t attn_decode_splitkv_noalloc(const void *q, const void *k, const void *v, void *o,
                                          float *lse, int b, int sq, int sk, int h, int d,
                                          float scale, int num_splits, attn_dtype_t dtype,
                                          cudaStream_t stream);

/*
 * Status reader of attn_decode_splitkv_noalloc, allocating nothing either.
 * Synchronises `stream`, then reports and clears that entry point's status
 * word on the current device: ATTN_ERR_DEVICE_TIMEOUT if one of its kernels
 * abandoned a bounded wait since the last call (attn_last_timeout_site()
 * then names the kernel and wait), ATTN_ERR_CUDA if the stream reported an
 * error, ATTN_OK otherwise (also before the entry point's first call).
 */
attn_status_t attn_get_noalloc_status(cudaStream_t stream);

/*
 * The split heuristic for num_splits = 0 on the current device (same issue:
 * split only when the work units leave SMs idle; then one CTA per SM, at
 * most one split per key block and 128 splits). A work unit is one query
 * row of a (batch, head) when sq == 1, and 256 query rows of a (batch,
 * head) when sq > 1. Returns the split count (>= 1), or 0 on invalid sizes
 * or when no device can be queried.
 */
int attn_decode_num_splits(int b, int sq, int sk, int h, int d);

/* The same heuristic for an explicit SM count; pure host arithmetic. */
int attn_decode_num_splits_for_sms(int b, int sq, int sk, int h, int d, int num_sms);

/*
 * Synchronises `stream`, then reports and clears the current device's
 * status word: ATTN_ERR_DEVICE_TIMEOUT if a kernel abandoned a bounded wait
 * since the last call, ATTN_ERR_CUDA if the stream reported an error,
 * ATTN_OK otherwise.
 */
attn_status_t attn_get_device_status(cudaStream_t stream);

/* Where the last recorded timeout happened (kernel and wait site code), 0 if none. */
unsigned int attn_last_timeout_site(void);

/* Static, human-readable name of a status code. */
const char *attn_status_string(attn_status_t status);

/*
 * Waits for the current device to finish its work, frees the split
 * decode's per-stream workspaces (counters and partials; the next split
 * decode on a stream makes them again) and returns the memory the device's
 * default pool keeps cached to the system. No other call of this library
 * may run on the device meanwhile (from another host thread).
 */
void attn_release_workspace(void);

/*
 * Test hooks, host-side only and never needed in production; 0 restores
 * normal operation. ATTN_DEBUG_SKIP_LOADS makes the next launched kernels
 * issue no loads at all, so their first wait runs out and they return with
 * a timeout status instead of hanging. ATTN_DEBUG_GENERAL_FWD makes forward
 * calls with at most 256 keys and d <= 64, which normally run the short
 * forward kernel (all keys of a head in one tile), run the general
 * key-tile-loop kernel instead, so that both can be checked on one shape.
 * ATTN_DEBUG_GENERAL_BWD does the same for the short backward kernel: those
 * backward calls run the key-tile and query-tile kernels.
 */
#define ATTN_DEBUG_SKIP_LOADS 1u
#define ATTN_DEBUG_GENERAL_FWD 2u
#define ATTN_DEBUG_GENERAL_BWD 4u
void attn_debug_set_flags(unsigned int flags);

/*
 * Test hook, host-side only (launches nothing, needs no GPU): the plan the
 * short forward kernel (all keys of a head in one tile) would run a forward
 * of sq query rows, sk keys, h heads and head dim d with. grouped_ok != 0
 * allows heads in groups of four (attn_fwd allows it when the one-head tiles
 * outnumber the SMs). Returns 1 and writes 12 ints to out (caller-owned):
 *   out[0] key columns N of S (sk rounded up to 32)
 *   out[1] TMEM column of the O accumulator within a slot
 *   out[2] TMEM columns of one slot       out[3] slots (items in flight)
 *   out[4] bytes of one K or V tile       out[5] bytes of one stage
 *   out[6] stages                         out[7] 1 if heads are grouped
 *   out[8] 32-row query blocks per head (grouped; else 0)
 *   out[9] K/V stages (grouped; else 0)
 *   out[10] shared-memory bytes the tiles take
 *   out[11] shared-memory bytes available to them
 * Returns 0 and leaves out untouched when the short kernel does not take
 * the shape (sq, sk or h below 1, sk > 256, d not 16, 32 or 64) or out is
 * NULL.
 */
int attn_debug_short_plan(int sq, int sk, int h, int d, int grouped_ok, int *out);

/* Library ABI version (major * 100 + minor): 101. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EXATTN_H */
