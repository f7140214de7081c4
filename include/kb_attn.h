/*
 * kb_attn.h -- C ABI of libkb_attn.so: bitwise-aligned causal grouped-query
 * attention forward for NVIDIA GB300 (sm_103a).
 *
 * The operation (KernelBraid README, sections "Features" and "Usage / Use a
 * selected kernel"): BF16 causal attention over contiguous
 * [batch, heads, sequence, head_dim] tensors, 32 query heads sharing 8 KV
 * heads (query head h reads KV head h / 4), head_dim 128, scale 1/sqrt(128).
 * For a query row at absolute position p the output is
 *     o = sum_{j<=p} softmax_j(q . k_j / sqrt(128)) v_j.
 *
 * The three entry points follow one numerical contract (README "Method":
 * the contract connects full-sequence prefill, partitioned forward execution
 * and one-token decode; "Advantages": prefill and incremental decode give
 * bitwise-identical outputs).  A row at position p computed by
 * kb_attn_prefill, by kb_attn_chunk (any split of the sequence) and by
 * kb_attn_decode (ctx_len = p + 1) has the same bf16 bits.
 *
 * Contract version 3 (kb_contract_version): key tiles of 128 keys visited in
 * ascending order; one tcgen05 MMA shape and k-order; one per-row online
 * softmax (fp32 max and sum, one exp2 path, scale 1/sqrt(128)); one final
 * normalisation; and a fixed, length-determined split of every row's keys
 * into segments of 1024 keys (8 tiles) anchored at key 0, each segment run
 * from the fresh softmax state and the segments folded left to right by one
 * fold function.  The split lets a small-batch decode of a long context run
 * its segments on several SMs at once while prefill folds the same segments
 * in order, so both stay bit-identical.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers on the current CUDA device,
 *    bf16, contiguous, 16-byte aligned, owned by the caller.  The library
 *    never allocates, frees or keeps them.
 *  - Hq must equal 4 * Hkv (the GQA group size of the contract); head_dim is
 *    fixed at 128.  Other shapes return KB_ERR_UNSUPPORTED.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and do not synchronise the host.  Argument errors are
 *    reported before anything is enqueued.  A device-side wait that gave up
 *    (never expected) is reported by kb_attn_check_device_status.
 *  - Outputs are valid only once kb_attn_check_device_status has returned
 *    KB_OK after the call.  KB_OK from an entry point means only that the
 *    arguments passed the host checks and the kernels were enqueued.  When a
 *    kernel gives up on a wait or finds a device-resident argument out of
 *    range (a page index, a per-sequence length) it records that in the
 *    library's per-device error word; until kb_attn_check_device_status reads
 *    and clears that word, every later kernel on the device skips its work
 *    and leaves its output unwritten, although its entry point returns KB_OK.
 *  - The sizes are all the library sees of the buffers: it cannot check that
 *    a buffer is as large as its shape says.  A caller that passes sizes
 *    larger than its allocations makes the kernels read or write past them.
 *  - Rows of the KV cache beyond the visible context are never used, so they
 *    may hold anything (including NaN bit patterns).
 */
#ifndef KB_ATTN_H
#define KB_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kb_status {
    KB_OK = 0,
    KB_ERR_INVALID_ARG = 1,   /* null or misaligned pointer, non-positive size, not device memory */
    KB_ERR_UNSUPPORTED = 2,   /* shape outside the contract (Hq != 4*Hkv, sizes too large) */
    KB_ERR_CUDA = 3,          /* a CUDA runtime or driver call failed */
    KB_ERR_TIMEOUT = 4        /* a bounded device-side wait gave up (see kb_attn_check_device_status) */
} kb_status;

/*
 * Full-sequence causal prefill (README "Usage": unified_prefill(q, k, v, H_Q, H_KV)).
 *   q, o : [B, Hq, S, 128]   query rows are positions 0..S-1; o has q's shape
 *   k, v : [B, Hkv, S, 128]
 * Identical to kb_attn_chunk(q, k, v, o, B, Hq, Hkv, S, 0, S, stream).
 */
kb_status kb_attn_prefill(const void* q, const void* k, const void* v, void* o,
                          int B, int Hq, int Hkv, int S, void* stream);

/*
 * Partitioned (chunked) forward against a KV cache (README "Method":
 * partitioned forward execution; "Usage": prompt/answer splits).
 *   q, o : [B, Hq, L, 128]       query row i is absolute position start + i
 *   k, v : [B, Hkv, kv_cap, 128] rows 0..start+L-1 must already hold the keys
 *                                and values of every position up to the chunk's
 *                                last row (the caller appends the chunk's own
 *                                K/V before the call)
 * Requires L >= 1, start >= 0, start + L <= kv_cap.
 */
kb_status kb_attn_chunk(const void* q, const void* k, const void* v, void* o,
                        int B, int Hq, int Hkv, int L, int start, int kv_cap, void* stream);

/*
 * One-token decode (README "Usage": unified_decode(q[:, :, -1:], k, v, H_Q, H_KV)).
 *   q, o : [B, Hq, 1, 128]       the query sits at position ctx_len - 1
 *   k, v : [B, Hkv, kv_cap, 128] rows 0..ctx_len-1 are the visible context
 * Requires 1 <= ctx_len <= kv_cap.
 */
kb_status kb_attn_decode(const void* q, const void* k, const void* v, void* o,
                         int B, int Hq, int Hkv, int ctx_len, int kv_cap, void* stream);

/*
 * Partitioned (chunked) forward against a paged KV cache: as kb_attn_chunk,
 * with the keys and values of every sequence in pages of a shared pool (the
 * page table is this library's addition; the pages show only a contiguous
 * cache).
 *   q, o         : [B, Hq, L, 128]; query row i is absolute position start + i
 *   k_pages,
 *   v_pages      : pools [num_pages, Hkv, page_size, 128] bf16; positions
 *                  0..start+L-1 of every sequence must be written
 *   block_table  : device int32 [B, pages_per_seq]; key position p of batch b
 *                  lives in page block_table[b, p / page_size], row p % page_size
 * page_size must be a positive multiple of 128; start + L <= pages_per_seq *
 * page_size.  Bits equal kb_attn_chunk on the same data laid out contiguously.
 * An out-of-range page index is found on the device and reported by the next
 * kb_attn_check_device_status as KB_ERR_INVALID_ARG.
 */
kb_status kb_attn_chunk_paged(const void* q, const void* k_pages, const void* v_pages, void* o,
                              int B, int Hq, int Hkv, int L, int start, const int* block_table,
                              int pages_per_seq, int page_size, int num_pages, void* stream);

/*
 * Ragged batch: chunked forward where every sequence has its own start
 * position and row count (device int32 arrays), against a contiguous cache
 * (block_table == NULL) or a paged pool.  A full prefill of sequences of
 * different lengths is starts[b] = 0, lens[b] = S_b.  (The per-sequence
 * lengths are this library's addition; the pages' workloads are uniform.)
 *   q, o     : [B, Hq, L_max, 128]; row i < lens[b] of batch b is position
 *              starts[b] + i; rows lens[b]..L_max-1 are neither read for any
 *              other row nor written
 *   k, v     : block_table == NULL: [B, Hkv, kv_cap, 128]
 *              else pools [num_pages, Hkv, page_size, 128] addressed as in
 *              kb_attn_chunk_paged (kv_cap is then pages_per_seq * page_size)
 *   starts,
 *   lens     : device int32 [B]; 0 <= lens[b] <= L_max, starts[b] >= 0,
 *              starts[b] + lens[b] <= kv_cap; keys 0..starts[b]+lens[b]-1 of
 *              every sequence must be written, later cache rows may hold anything
 * Bits equal kb_attn_chunk on each sequence alone.  Out-of-range starts, lens
 * or page indices are found on the device: those sequences are not written and
 * the next kb_attn_check_device_status returns KB_ERR_INVALID_ARG.
 */
kb_status kb_attn_chunk_varlen(const void* q, const void* k, const void* v, void* o,
                               int B, int Hq, int Hkv, int L_max, const int* starts, const int* lens,
                               int kv_cap, const int* block_table, int pages_per_seq, int page_size,
                               int num_pages, void* stream);

/*
 * One-token decode over a paged KV cache, one context length per sequence
 * (README "Usage": unified_decode; the page table is this library's
 * addition, the pages show only a contiguous cache).
 *   q, o         : [B, Hq, 1, 128]; the query of batch b sits at position ctx_lens[b] - 1
 *   k_pages,
 *   v_pages      : pools [num_pages, Hkv, page_size, 128] bf16
 *   block_table  : device int32 [B, pages_per_seq]; key position p of batch b lives in
 *                  page block_table[b, p / page_size] at row p % page_size
 *   ctx_lens     : device int32 [B], each in 1 .. pages_per_seq * page_size
 * page_size must be a positive multiple of 128.  Page rows past a sequence's
 * context may hold anything.  Bits equal kb_attn_decode on the same keys and
 * values laid out contiguously.  Out-of-range ctx_lens or page indices are
 * found on the device: the affected rows are not written and the next
 * kb_attn_check_device_status returns KB_ERR_INVALID_ARG.
 */
kb_status kb_attn_decode_paged(const void* q, const void* k_pages, const void* v_pages, void* o,
                               int B, int Hq, int Hkv, const int* block_table, int pages_per_seq,
                               int page_size, int num_pages, const int* ctx_lens, void* stream);

/*
 * Synchronises `stream`, then reads and clears the library's device-side
 * error word on the current device.  Returns KB_ERR_TIMEOUT if any kernel
 * since the last check gave up on a bounded wait (its output is then
 * undefined), KB_ERR_INVALID_ARG if a kernel found a device-resident argument
 * out of range, KB_ERR_CUDA if the synchronisation failed, else KB_OK.
 */
kb_status kb_attn_check_device_status(void* stream);

/*
 * Test hook for the failure path: enqueues a one-CTA kernel that waits on a
 * barrier nothing will signal, giving up after `limit_us` microseconds
 * (1..1000000).  A following kb_attn_check_device_status returns
 * KB_ERR_TIMEOUT.  Faults and hangs nothing.
 */
kb_status kb_attn_debug_wait_timeout(int limit_us, void* stream);

/*
 * Explicit segment length (contract C5 with seg_tiles instead of 8): a row's
 * key tiles are cut into segments of seg_tiles 128-key tiles anchored at key
 * 0; each segment runs the tile steps from the fresh state and the segments
 * are folded left to right by the contract's fold function, then normalised.
 * Every entry point below gives the same bits for a row at position p when
 * called with the same seg_tiles (>= 1).  seg_tiles = 8 gives the default
 * entry points' bits; a seg_tiles of at least the row's tile count is the
 * unsplit online softmax (contract version 2's default).  These calls run a
 * different fold path from the default entry points (short chunks write
 * per-segment partials to a workspace that a second kernel folds), so with
 * seg_tiles = 8 they also cross-check the default path's bits.
 *
 * kb_attn_prefill_seg: as kb_attn_prefill (no workspace).
 * kb_attn_chunk_seg:   as kb_attn_chunk.  Chunks of at most 32 rows (and
 *   decode) run one CTA per (segment, batch, KV head) and need a device
 *   workspace of kb_attn_seg_workspace_bytes(B, Hq, L, start, seg_tiles)
 *   bytes (16-byte aligned, caller-owned, contents scratch); longer chunks
 *   fold in the kernel and ignore it.  Too small a workspace returns
 *   KB_ERR_INVALID_ARG.
 * kb_attn_decode_seg:  as kb_attn_decode (a chunk of one row at ctx_len-1).
 * Paged and ragged caches are not offered in this mode (KB_ERR_UNSUPPORTED).
 */
kb_status kb_attn_prefill_seg(const void* q, const void* k, const void* v, void* o,
                              int B, int Hq, int Hkv, int S, int seg_tiles, void* stream);
kb_status kb_attn_chunk_seg(const void* q, const void* k, const void* v, void* o,
                            int B, int Hq, int Hkv, int L, int start, int kv_cap, int seg_tiles,
                            void* workspace, size_t workspace_bytes, void* stream);
kb_status kb_attn_decode_seg(const void* q, const void* k, const void* v, void* o,
                             int B, int Hq, int Hkv, int ctx_len, int kv_cap, int seg_tiles,
                             void* workspace, size_t workspace_bytes, void* stream);
/*
 * kb_attn_decode_seg without a caller workspace: the partials go to a 4 MiB
 * scratch array the library owns (one per device, part of the loaded module),
 * so the call allocates nothing and takes nothing but the decode's tensors.
 * It serves callers that cannot allocate device memory at the point of the
 * call: a serving loop whose memory pool is already handed out, or code that
 * must not enter the CUDA allocator (which may synchronise the device) in its
 * decode step.  No paper counterpart: it is a deployment variant of
 * kb_attn_decode_seg.
 * Requests needing more than 4 MiB of partials (B * Hq * segments * 528 bytes)
 * return KB_ERR_UNSUPPORTED before anything is enqueued.  The scratch is
 * shared and keeps the last call's contents (every call overwrites the part
 * it reads): calls of this entry point on one device that overlap on the GPU
 * race, so issue them on one stream.  The first call of any entry point on a
 * device looks up the scratch's device address (cudaGetSymbolAddress); make
 * that first call before any stream capture.  Bits equal kb_attn_decode_seg's.
 */
kb_status kb_attn_decode_seg_static(const void* q, const void* k, const void* v, void* o,
                                    int B, int Hq, int Hkv, int ctx_len, int kv_cap, int seg_tiles,
                                    void* stream);
/* Workspace bytes kb_attn_chunk_seg / kb_attn_decode_seg need for a chunk of
 * L <= 32 rows at positions start..start+L-1 (0 for bad arguments or L > 32). */
size_t kb_attn_seg_workspace_bytes(int B, int Hq, int L, int start, int seg_tiles);

/*
 * Training forward: kb_attn_prefill plus each row's log-sum-exp, which the
 * backward needs (README "Motivation": the RL policy update differentiates
 * the same attention).
 *   q, o, k, v : as kb_attn_prefill; o gets the same bits as kb_attn_prefill
 *   lse        : [B, Hq, S] fp32, device, 4-byte aligned, caller-owned;
 *                lse[b,h,i] = ln sum_{j<=i} exp(q_i . k_j / sqrt(128))
 * Always runs the default tile kernel (CTA shape 3), whose bits every other
 * shape reproduces.
 */
kb_status kb_attn_prefill_lse(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int Hq, int Hkv, int S, void* stream);

/*
 * Backward of the whole-sequence causal prefill (query row i at position i):
 * the gradients of q, k and v for a given gradient dout of the output.
 *   q, dout, o : [B, Hq, S, 128] bf16; o and lse from kb_attn_prefill_lse
 *   k, v       : [B, Hkv, S, 128] bf16
 *   lse        : [B, Hq, S] fp32 (input)
 *   delta      : [B, Hq, S] fp32 (output): delta[b,h,i] = dout_i . o_i
 *   dq         : [B, Hq, S, 128] bf16 (output)
 *   dk, dv     : [B, Hkv, S, 128] bf16 (output); each sums the four query
 *                heads of its group
 * With P the softmax rows recomputed from lse, dP_ij = dout_i . v_j and
 * dS_ij = P_ij (dP_ij - delta_i):
 *   dq_i = sum_j dS_ij k_j / sqrt(128),  dk_j = sum_{h,i} dS_ij q_i / sqrt(128),
 *   dv_j = sum_{h,i} P_ij dout_i   (P and dS rounded to bf16 for the products,
 *   fp32 accumulation, bf16 outputs).
 * No atomics: every output element is summed by one CTA in a fixed order, so
 * repeated calls give identical bits.  All pointers are device memory,
 * caller-owned; errors as for the forward entry points.
 */
kb_status kb_attn_backward(const void* q, const void* k, const void* v, const void* o, const void* dout,
                           const float* lse, float* delta, void* dq, void* dk, void* dv,
                           int B, int Hq, int Hkv, int S, void* stream);

/*
 * Prefill/chunk with an explicit kernel shape, for tests of the contract:
 * q_tiles_per_cta = 3 runs the tile kernel (one 128-row query tile per CTA,
 * one CTA per SM, three score buffers, so Q K^T of later key tiles overlaps
 * the softmax of the current one), launched persistent (CTAs walk balanced
 * pairs of query tiles, or single tiles longest first dealt to the CTAs
 * back and forth) or one CTA per tile as the sizes suit; 4 is 3 with the
 * persistent launch on pairs forced, 5 with the back-and-forth deal forced;
 * 0 runs the packed kernel (the 4 heads of a
 * GQA group times the chunk's rows in one MMA tile; L <= 32).  Other values
 * return KB_ERR_INVALID_ARG.  kb_attn_chunk, kb_attn_prefill and
 * kb_attn_decode pick packed for L <= 32 and 3 otherwise.  Every shape gives
 * the same bits.
 */
kb_status kb_attn_chunk_cta_shape(const void* q, const void* k, const void* v, void* o,
                                  int B, int Hq, int Hkv, int L, int start, int kv_cap,
                                  int q_tiles_per_cta, void* stream);

/* The cudaError_t code (as int) and its description for the most recent
 * KB_ERR_CUDA returned on the calling host thread; 0 / "no error" if none. */
int kb_attn_last_cuda_error(void);
const char* kb_attn_last_cuda_error_string(void);

/* Static description of a status code (never NULL). */
const char* kb_status_string(kb_status s);

/* Version of the numerical contract; outputs are bit-identical across builds
 * with the same contract version on the same GPU architecture. */
int kb_contract_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KB_ATTN_H */
