/*
 * attn.h -- C ABI of the GB300 (sm_103a) exact-attention library.
 *
 * Exact scaled dot-product attention computed without materialising the score
 * matrix S = QK^T: every query row carries an online-softmax state (running
 * max m, normaliser l referenced to m, unnormalised accumulator O~), rescaled
 * by exp(m_old - m_new) whenever the max rises, and disjoint key sets combine
 * through the associative merge of two states.
 *
 * Sources (page title, then section):
 *   [NA]  "Naive attention and the online softmax" -- opening section (shapes,
 *         GQA broadcast), (3) "The online recurrence", "Extending the
 *         recurrence to the output", "The state that gets passed around is the
 *         log-sum-exp", "The base case is a NaN factory".
 *   [OSR] "The Online Softmax Recurrence" -- "The recurrence", "Where it breaks".
 *   [DEC] "Decode attention: FlashDecoding, split-K, paged kernels" -- "The
 *         grid", "Segment length, and the early exit", "What the merge costs",
 *         "Where GQA enters", paged addressing, "CUDA graphs need the split
 *         count pinned".
 *   [MRG] "Merge normalized attention without averaging tile outputs".
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers (cudaMalloc / PyTorch CUDA
 *     memory) unless a parameter says otherwise; the caller owns every buffer.
 *     The library never allocates memory, frees or synchronises: each call
 *     only enqueues work on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and returns. The one exception is attn_prefill_host called
 *     without a pipe of the caller's: its first call on a device creates two
 *     copy streams and five events that it keeps (no memory allocation).
 *   - Tensors are dense, row-major, with the shapes given below. Tensor base
 *     pointers must be 16-byte aligned (TMA and 128-bit vector loads);
 *     `workspace` must be 256-byte aligned.
 *   - bf16 is IEEE-style bfloat16 (1-8-7); fp32 is IEEE binary32.
 *   - LSE is the natural-log log-sum-exp m + ln(l) of the scaled logits, fp32.
 *   - A query row with no allowed key yields output 0 and LSE = -inf ([MRG],
 *     last paragraph: zero output is the extension chosen for empty rows).
 *   - Signatures. The three core calls keep their minimal argument lists,
 *     with these additions, each where the minimal form could not serve:
 *       attn_prefill       workspace, workspace_bytes (after dtype): scratch
 *                          for the fp16 copy of V with which P V runs as one
 *                          fp16 tensor-core product per key tile instead of
 *                          two bf16 ones (1.13x on the causal T = 8192
 *                          layer); NULL keeps the no-scratch form.
 *       attn_decode_paged  num_blocks (after page_size): the cache's page
 *                          count, which the TMA tensor map over the cache
 *                          needs, and against which table entries are
 *                          checked (an entry outside the cache reads zeros
 *                          and sets an error bit instead of reading past it).
 *       attn_merge_states  none.
 *     attn_decode_workspace_bytes and attn_recommended_splits keep theirs;
 *     the ragged-batch split rule, which needs the batch's total length, is
 *     attn_recommended_splits_ragged. Every other call is an addition.
 *   - Errors: arguments are validated on the host before anything is
 *     launched; an invalid call returns ATTN_ERR_INVALID_ARG (or
 *     ATTN_ERR_UNSUPPORTED for a well-formed but unbuilt shape) and enqueues
 *     nothing. ATTN_ERR_CUDA reports a failed launch (cudaGetLastError).
 *     Kernels never trap: a bounded wait that gives up, or a page index
 *     outside the cache, sets a device error word that
 *     attn_get_device_error() reads.
 */
#ifndef ONLINE_SOFTMAX_ATTN_GB300_ATTN_H_
#define ONLINE_SOFTMAX_ATTN_GB300_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,
  ATTN_ERR_UNSUPPORTED = 2,
  ATTN_ERR_CUDA = 3,
  ATTN_ERR_DEVICE = 4,        /* a device error bit other than a wait timeout */
  ATTN_ERR_DEVICE_TIMEOUT = 5 /* a kernel's bounded wait gave up               */
} attn_status_t;

typedef enum { ATTN_DTYPE_F32 = 0, ATTN_DTYPE_BF16 = 1 } attn_dtype_t;

/* Device error bits reported by attn_get_device_error(). */
#define ATTN_DEVERR_WAIT_TIMEOUT 0x1u /* a bounded mbarrier wait gave up      */
#define ATTN_DEVERR_BAD_PAGE 0x2u     /* block_table entry outside the cache */
#define ATTN_DEVERR_TMEM 0x4u         /* tensor-memory allocation failed     */
#define ATTN_DEVERR_BAD_SEQ_LEN 0x8u  /* seq_len < 0 or beyond the table row  */
/* Builds compiled with -DATTN_DEBUG only: an index or offset check failed;
 * the access it guarded was skipped (release builds carry no such checks). */
#define ATTN_DEVERR_DEBUG_INDEX 0x10u

/* Human-readable name of a status code; never NULL. */
const char* attn_status_string(attn_status_t status);

/* Library ABI version (major * 100 + minor): 301. */
int attn_version(void);

/*
 * attn_prefill_workspace_bytes -- scratch attn_prefill can use for the given
 * shape: an fp16 copy of V ([h_kv, T, d_h]), one int per (KV head, 128-key
 * tile) saying whether that tile fits fp16, and 256 bytes holding the
 * counter from which the attention kernel's CTAs claim work. Host-only, pure. 0 for
 * ATTN_DTYPE_F32 (the SIMT path needs none) and for T == 0; (size_t)-1 on
 * invalid arguments (T < 0, h_kv < 1, d_h not 64 or 128, unknown dtype).
 */
size_t attn_prefill_workspace_bytes(int T, int h_kv, int d_h, attn_dtype_t dtype);

/*
 * attn_prefill -- exact attention of T queries over the same T keys, per head.
 * Follows [NA] opening section (Q [h,T,d_h], K/V [h_kv,T,d_h] broadcast to
 * g = h/h_kv query heads: query head hq reads KV head hq / g) and [NA] (3) /
 * "Extending the recurrence to the output" (one pass over key tiles, divide
 * once at the end).
 *
 *   q     [h, T, d_h]     dtype                          (read)
 *   k, v  [h_kv, T, d_h]  dtype                          (read)
 *   o     [h, T, d_h]     dtype                          (written)
 *   lse   [h, T]          fp32, may be NULL               (written)
 *   causal: nonzero -> key j is allowed for query i iff j <= i.
 *   scale : multiplies q.k before the softmax (normally 1/sqrt(d_h)); must be
 *           finite and > 0.
 *   dtype : ATTN_DTYPE_BF16 -> tcgen05 tensor-core path (d_h = 128 or 64),
 *           fp32 accumulation and statistics;
 *           ATTN_DTYPE_F32  -> fp32 SIMT path (d_h = 64 or 128), fp32 throughout.
 *   workspace, workspace_bytes: caller-owned device scratch, 256-byte
 *           aligned, at least attn_prefill_workspace_bytes(T, h_kv, d_h,
 *           dtype) bytes; overwritten by the call (stream-ordered), so calls
 *           sharing one workspace must not overlap on the GPU. May be NULL
 *           (workspace_bytes ignored): the bf16 path then forms every P V
 *           product as P_hi V + P_lo V in bf16, exact but slower. With a
 *           workspace, V is first copied to fp16 (one extra kernel) and
 *           P V is a single fp16 product wherever V fits fp16.
 * Errors: INVALID_ARG for NULL q/k/v/o (T > 0), T < 0, h < 1, h > 65535,
 * h_kv < 1, h % h_kv != 0, misaligned pointers, scale not finite and > 0, a
 * non-NULL workspace that is misaligned or smaller than required;
 * UNSUPPORTED for other d_h, and for bf16 with more than 65535 query tiles
 * of 128 (T > 8388480). T == 0 is a no-op returning ATTN_OK.
 */
attn_status_t attn_prefill(const void* q, const void* k, const void* v, void* o, float* lse,
                           int T, int h, int h_kv, int d_h, int causal, float scale,
                           attn_dtype_t dtype, void* workspace, size_t workspace_bytes,
                           void* stream);

/*
 * attn_prefill_host -- attn_prefill with Q, K, V in host memory and O, LSE
 * written back to host memory, copies included in the call ([NA] (3), as
 * attn_prefill; heads are independent, so the layer is cut into groups of
 * KV heads with their query heads, and group c+1's inputs copy in while
 * group c computes and group c-1's outputs copy out).
 * Results are bitwise those of attn_prefill on the same inputs.
 *
 *   q, k, v, o, lse   host pointers, same shapes, dtypes and layouts as
 *                     attn_prefill; lse may be NULL. Page-locked memory
 *                     (cudaHostAlloc / cudaHostRegister) lets the copies run
 *                     asynchronously and overlap; pageable memory works but
 *                     copies through staging.
 *   n_chunks          > 0: that many equal groups, dividing h_kv (at most
 *                     64). 0: with h_kv >= 4, four groups in the proportions
 *                     3 : 2 : 2 : 1 (the compute and copy-out that nothing
 *                     overlaps stay short); with h_kv < 4, 2 equal groups
 *                     when h_kv is even, else 1
 *   scratch           device memory, 256-byte aligned, at least
 *                     attn_prefill_host_scratch_bytes(T, h, h_kv, d_h, dtype)
 *                     bytes: device copies of q, k, v, o, lse and the
 *                     prefill workspace
 *   stream            the caller's stream: the call is ordered after the work
 *                     already queued on it, runs the attention on it, and the
 *                     stream continues only after the last output copy; the
 *                     host buffers may be read after that work completes
 *                     (e.g. cudaStreamSynchronize). Returns once queued.
 *   pipe              NULL, or the caller's two copy streams and five events
 *                     (attn_host_pipe_t below): with them the call creates
 *                     nothing. With NULL the library creates such a pipe per
 *                     device on the first call without one (that first call
 *                     must therefore not be inside a stream capture) and
 *                     keeps it; calls on one device then hold a per-device
 *                     lock while they queue work.
 * Pageable host buffers work, but a copy from or to pageable memory blocks
 * the calling thread until it completes, so the groups do not overlap and
 * the call returns only after the last output copy (holding the device's
 * lock when pipe is NULL).
 * Errors: as attn_prefill, plus INVALID_ARG for n_chunks < 0, n_chunks > 64,
 * h_kv % n_chunks != 0, a NULL or misaligned scratch or one that is too
 * small, a pipe with a NULL member, with copy_in == copy_out or with either
 * equal to `stream`; UNSUPPORTED for more than 65535 query tiles of 128 on
 * the bf16 path (T > 8388480). All of these are found before anything is
 * queued. ATTN_ERR_CUDA if a copy, event or launch fails; the caller's
 * stream is then still joined to both copy streams, so nothing queued by the
 * call can touch the host buffers after the stream's later work starts.
 */
#define ATTN_HOST_PIPE_EVENTS 5
typedef struct attn_host_pipe {
  void* copy_in;   /* cudaStream_t for host-to-device copies                  */
  void* copy_out;  /* cudaStream_t for device-to-host copies                  */
  void* events[ATTN_HOST_PIPE_EVENTS]; /* cudaEvent_t each, e.g. created with
                                          cudaEventDisableTiming; re-recorded
                                          by every call (one call at a time
                                          per pipe)                          */
} attn_host_pipe_t;
size_t attn_prefill_host_scratch_bytes(int T, int h, int h_kv, int d_h, attn_dtype_t dtype);
attn_status_t attn_prefill_host(const void* q, const void* k, const void* v, void* o, float* lse,
                                int T, int h, int h_kv, int d_h, int causal, float scale,
                                attn_dtype_t dtype, int n_chunks, void* scratch,
                                size_t scratch_bytes, const attn_host_pipe_t* pipe,
                                void* stream);

/*
 * attn_prefill_paged -- exact attention for a batch of variable-length query
 * rows over a paged KV cache (chunked prefill, and mixed batches of prefill
 * and decode rows). Row b has the q_len_b = cu_seqlens_q[b+1] - cu_seqlens_q[b]
 * query tokens cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 of q, and keys
 * 0 .. seq_lens[b]-1 in the cache through block_table row b ([DEC] paged
 * addressing); its queries are its last q_len_b key positions, so with causal
 * query i sees keys up to seq_lens[b] - q_len_b + i (bottom-right alignment;
 * the pages leave unequal lengths open and this is the chunked-prefill
 * reading); without causal it sees all seq_lens[b] keys. Method as
 * attn_prefill ([NA] (3), "Extending the recurrence to the output"), on the
 * tcgen05 kernel with key tiles gathered page by page. P V runs in one of two
 * forms, as in attn_prefill: with the small workspace every V tile stays
 * bf16 and takes the exact two-term bf16 P; with the larger one
 * (attn_prefill_paged_v16_workspace_bytes) a pre-pass copies the pages each
 * row uses into an fp16 buffer in the workspace, row by row, and a 128-key
 * tile that converts exactly takes an fp16 P against it (one MMA instead of
 * two); a tile holding |v| >= 2^16, inf or NaN keeps the bf16 path (read
 * from the copy too, where it is stored as bf16).
 * Rows of one query (decode rows of a mixed batch): with decode_splits > 0
 * they get no query tile; after the prefill kernel the call runs the
 * split-KV decode of attn_decode_paged_adaptive over those rows alone
 * ([DEC] "Where GQA enters": one query in a 128-row tile leaves the rest of
 * the tile idle and the row's keys on one CTA), with at most decode_splits
 * splits per row planned on the device from their lengths, and writes their
 * outputs at token cu_seqlens_q[b]. With decode_splits == 0 they run as
 * 1-row query tiles.
 *
 *   q            [total_q, h, d_h] bf16, rows packed back to back    (read)
 *   k_cache,
 *   v_cache      [num_blocks, page_size, h_kv, d_h] bf16                (read)
 *   block_table  [B, max_blocks_per_seq] int32                          (read)
 *   cu_seqlens_q [B + 1] int32, cu_seqlens_q[0] = 0, non-decreasing,
 *                cu_seqlens_q[B] = total_q                              (read)
 *   seq_lens     [B] int32, q_len_b <= seq_lens[b] <= max_blocks_per_seq *
 *                page_size                                              (read)
 *   max_q_len    host bound on every q_len_b (sizes the grid)
 *   decode_splits 0, or the most splits a decode row may take
 *                (1 .. ATTN_MAX_SPLITS); see above
 *   workspace    256-byte aligned device memory, overwritten by the call:
 *                first attn_prefill_paged_decode_workspace_bytes(B, h,
 *                decode_splits, d_h) bytes (0 when decode_splits is 0) for the
 *                decode rows, then the prefill's own part: at least
 *                attn_prefill_paged_workspace_bytes(B) bytes (per-row tile
 *                offsets), or, for the fp16 V form, at least
 *                attn_prefill_paged_v16_workspace_bytes(B,
 *                max_blocks_per_seq, h_kv, d_h) bytes (when that is nonzero;
 *                the form is chosen by the size given)
 *   o            [total_q, h, d_h] bf16                                 (written)
 *   lse          [total_q, h] fp32, natural log, may be NULL             (written)
 * All tensor arguments are device pointers. Device-side problems set bits in
 * the error word instead of faulting: a block-table entry outside the cache
 * (ATTN_DEVERR_BAD_PAGE; that page reads as zeros), seq_lens outside
 * [q_len_b, max_blocks_per_seq * page_size] or q_len_b outside
 * [0, min(max_q_len, max_blocks_per_seq * page_size)]
 * (ATTN_DEVERR_BAD_SEQ_LEN; the length is clamped, or the row is skipped and
 * its outputs are not written).
 * Errors: INVALID_ARG for NULL or misaligned pointers (16 bytes for q, the
 * caches and o; 4 for the int32 arrays and lse), B < 0, total_q < 0,
 * max_q_len < 1 with total_q > 0, h < 1, h > 65535, h % h_kv != 0,
 * num_blocks < 1, max_blocks_per_seq < 1, scale not finite and > 0,
 * decode_splits outside [0, ATTN_MAX_SPLITS], a small workspace;
 * UNSUPPORTED for d_h other than 64 / 128, page_size != 16, g = h / h_kv
 * not in {1, 2, 4, 8} with decode_splits > 0, or more than 65535 query
 * tiles in the launch (min(ceil(total_q / 128) + B, B * ceil(max_q_len /
 * 128))). B == 0 or total_q == 0 is a no-op.
 */
size_t attn_prefill_paged_workspace_bytes(int B);
/*
 * attn_prefill_paged_v16_workspace_bytes -- workspace bytes for the fp16 V
 * form of attn_prefill_paged: the tile offsets (256-byte aligned), then
 * int32 V-format flags [B, h_kv, ceil(max_blocks_per_seq / 8)] (256-byte
 * aligned), then the fp16 copy [B, ceil(max_blocks_per_seq / 8) * 128,
 * h_kv, d_h] (row b's key t at token b * ceil(max_blocks_per_seq / 8) * 128
 * + t). Host-only, pure. Returns 0 for invalid arguments (B < 0,
 * max_blocks_per_seq outside [1, 2^26], h_kv outside [1, 65535], d_h other
 * than 64 / 128) and when B * ceil(max_blocks_per_seq / 8) * 128 >= 2^31 (the
 * copy's token index must fit int32); the small workspace then still works.
 */
size_t attn_prefill_paged_v16_workspace_bytes(int B, int max_blocks_per_seq, int h_kv, int d_h);
/*
 * attn_prefill_paged_decode_workspace_bytes -- bytes at the front of
 * attn_prefill_paged's workspace for its decode rows: split partials
 * (attn_decode_workspace_bytes(B, h, decode_splits, d_h)) and 256 bytes for
 * the device split plan. 0 when decode_splits is 0, and on invalid arguments.
 * Host-only, pure.
 */
size_t attn_prefill_paged_decode_workspace_bytes(int B, int h, int decode_splits, int d_h);
attn_status_t attn_prefill_paged(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* block_table, const int32_t* cu_seqlens_q,
                                 const int32_t* seq_lens, int B, int total_q, int h, int h_kv,
                                 int d_h, int page_size, int num_blocks, int max_blocks_per_seq,
                                 int max_q_len, int causal, float scale, int decode_splits,
                                 void* workspace, size_t workspace_bytes, void* o, float* lse,
                                 void* stream);

/*
 * attn_decode_split_plan -- how one row's keys are cut into splits.
 * Follows [DEC] "Segment length, and the early exit": a row of seq_len keys
 * has n_pages = ceil(seq_len / page_size) pages; with at most num_splits
 * splits each split covers pages_per_split = ceil(n_pages / num_splits)
 * consecutive pages and the number of splits that do work is
 * ceil(n_pages / pages_per_split) (0 for an empty row); surplus splits return
 * at once. The decode kernel and its reduce use this same function.
 * Host-only, pure. Returns the active split count; writes pages_per_split if
 * the pointer is non-NULL. Returns -1 on invalid arguments.
 */
int attn_decode_split_plan(int seq_len, int page_size, int num_splits, int* pages_per_split);

/*
 * attn_recommended_splits -- split count for a decode batch on `device`.
 * Follows [DEC] "The grid": fill the first wave, S* = ceil(N_SM / G_2D) with
 * G_2D = B * h_kv and N_SM the device's SM count; then each split of the
 * longest row keeps at least 32 pages (so a CTA's start-up is amortised).
 * Result in [1, ATTN_MAX_SPLITS]. Host-only (it queries the device's SM
 * count); -1 on invalid arguments or when the device cannot be queried.
 */
#define ATTN_MAX_SPLITS 1024
int attn_recommended_splits(int B, int h_kv, int max_seq_len, int device);

/*
 * attn_recommended_splits_ragged -- attn_recommended_splits for a ragged
 * batch, with the SM count given: when the longest row is more than 1.25x
 * the mean length (known from total_seq_len), the splits are raised until
 * the longest row's split is no larger than a quarter of the mean work per
 * CTA slot, before the 32-page floor. total_seq_len may be 0 when unknown
 * (the ragged rule is then skipped; the result is that of
 * attn_recommended_splits). Host-only, pure; -1 on invalid arguments.
 */
int attn_recommended_splits_ragged(int B, int h_kv, int max_seq_len, long long total_seq_len,
                                   int num_sms);

/*
 * attn_decode_workspace_bytes -- bytes of scratch that attn_decode_paged needs
 * for the split partial states ([DEC] "What the merge costs": one fp32
 * d_h-vector plus two fp32 scalars per (row, head, split)):
 *   O~ fp32 [B*h, num_splits, d_h], then m fp32 [B*h, num_splits], then
 *   l fp32 [B*h, num_splits], each region starting on a 256-byte boundary.
 * Host-only, pure; 0 on invalid arguments.
 */
size_t attn_decode_workspace_bytes(int B, int h, int num_splits, int d_h);

/*
 * attn_decode_paged -- split-KV (FlashDecoding) attention of one query token
 * per row over a paged KV cache, then the reduce of the split partials.
 * Follows [DEC] throughout: stage 1 gives each (row, KV head, split) its own
 * CTA, which runs the online recurrence over its pages for all g query heads
 * of the KV head ("Where GQA enters") and stores the unnormalised partial
 * (O~, m, l); stage 2 (the same kernel as attn_merge_states) takes the
 * overall max, rescales, sums and divides once. Page translation ([DEC],
 * paged addressing): key position p of row b is slot p % page_size of
 * physical page block_table[b * max_blocks_per_seq + p / page_size].
 *
 *   q           [B, h, d_h]                              bf16 (read)
 *   k_cache,
 *   v_cache     [num_blocks, page_size, h_kv, d_h]       bf16 (read)
 *   block_table [B, max_blocks_per_seq]                  int32 (read); entries
 *               for pages >= ceil(seq_len/page_size) are never read
 *   seq_lens    [B]                                      int32 (read), >= 0
 *   workspace   attn_decode_workspace_bytes(B,h,num_splits,d_h) bytes (scratch)
 *   o           [B, h, d_h]                              bf16 (written)
 *   lse         [B, h]                 fp32, may be NULL (written)
 * page_size must be 16; d_h must be 128 or 64; g = h / h_kv in {1,2,4,8};
 * 1 <= num_splits <= ATTN_MAX_SPLITS; B <= 65535; scale finite and > 0. The launch geometry depends only on
 * (B, h_kv, num_splits), never on the lengths, so the call can be captured
 * in a CUDA graph and replayed with new lengths ([DEC] "CUDA graphs need the
 * split count pinned"). A row with seq_len 0 gives o = 0, lse = -inf. A
 * table entry outside [0, num_blocks) is treated as a page of zeros and sets
 * ATTN_DEVERR_BAD_PAGE. A seq_len below 0 or above max_blocks_per_seq *
 * page_size is clamped into that range and sets ATTN_DEVERR_BAD_SEQ_LEN.
 * Errors: INVALID_ARG for NULL pointers (B > 0), bad sizes, misalignment or
 * workspace_bytes too small; UNSUPPORTED for other d_h / g / page_size.
 */
attn_status_t attn_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_table, const int32_t* seq_lens,
                                int B, int h, int h_kv, int d_h, int page_size, int num_blocks,
                                int max_blocks_per_seq, int num_splits, float scale,
                                void* workspace, size_t workspace_bytes,
                                void* o, float* lse, void* stream);

/*
 * attn_decode_paged_adaptive -- attn_decode_paged with the split count chosen
 * on the device, for CUDA-graph capture. Follows [DEC] "SGLang: a split count
 * computed per sequence, on device" and "CUDA graphs need the split count
 * pinned": the launch geometry is fixed by max_splits (a grid of
 * max_splits x h_kv x B; CTAs past a row's splits return at once), while a
 * one-CTA plan kernel reads the batch's seq_lens, applies the rule of
 * attn_recommended_splits (with the GPU's SM count) capped at max_splits, and
 * turns it into pages per split of the longest row. Every row is cut into
 * splits of that many pages; the split kernel and the merge read the same
 * device value, so they agree on each row's active splits. A graph captured
 * once stays valid for any seq_lens with the same B and max_blocks_per_seq.
 *
 * Arguments, layouts and errors are those of attn_decode_paged with
 * num_splits replaced by max_splits (1 .. ATTN_MAX_SPLITS), plus:
 *   workspace: attn_decode_adaptive_workspace_bytes(B, h, max_splits, d_h)
 *     bytes; its last 256 bytes begin with the plan (int32 pages per split)
 *     written by the call.
 */
size_t attn_decode_adaptive_workspace_bytes(int B, int h, int max_splits, int d_h);
attn_status_t attn_decode_paged_adaptive(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_table, const int32_t* seq_lens,
                                         int B, int h, int h_kv, int d_h, int page_size,
                                         int num_blocks, int max_blocks_per_seq, int max_splits,
                                         float scale, void* workspace, size_t workspace_bytes,
                                         void* o, float* lse, void* stream);

/*
 * attn_decode_paged_deterministic -- attn_decode_paged with splits of a fixed
 * length, so that a row's result depends on the row alone. Follows [DEC]
 * "Split-K breaks bitwise reproducibility" (the split count, and with it the
 * order of the fp32 merge, otherwise follows the batch) and its fixed-tile
 * remedy: every split of a row covers pages_per_split pages (the last one the
 * rest), a row of n pages uses ceil(n / pages_per_split) splits, and the
 * partials are merged in split order. The output of a row is then
 * bit-identical whatever the other rows, the batch size or num_splits are.
 * The trade: a short row uses few splits, so a small batch may leave SMs idle.
 *
 * Arguments, layouts, workspace (attn_decode_workspace_bytes for num_splits)
 * and errors are those of attn_decode_paged, plus:
 *   pages_per_split >= 1: pages (of page_size keys) per split;
 *   num_splits: the grid's split count; must satisfy
 *     num_splits * pages_per_split >= max_blocks_per_seq (INVALID_ARG
 *     otherwise), so that every row's splits fit.
 */
attn_status_t attn_decode_paged_deterministic(const void* q, const void* k_cache,
                                              const void* v_cache, const int32_t* block_table,
                                              const int32_t* seq_lens, int B, int h, int h_kv,
                                              int d_h, int page_size, int num_blocks,
                                              int max_blocks_per_seq, int num_splits,
                                              int pages_per_split, float scale, void* workspace,
                                              size_t workspace_bytes, void* o, float* lse,
                                              void* stream);

/*
 * attn_decode_paged_static -- attn_decode_paged without a workspace argument
 * and without any allocation. The pages have no counterpart of this entry
 * point; it exists for callers that cannot obtain device memory at the call
 * site: for example a plugin loaded into a host program that owns all device
 * memory and offers it no allocation hook, or a serving hot loop that must not
 * call cudaMalloc (which can synchronise the device and takes allocator locks).
 *
 * The split partials live in a fixed array inside the library's device image
 * (ATTN_DECODE_STATIC_SCRATCH_BYTES on every GPU that loads the library, held
 * until the process exits). Arguments, layouts, results and errors are those
 * of attn_decode_paged, plus:
 *   - the partials, attn_decode_workspace_bytes(B, h, num_splits, d_h) bytes,
 *     must fit in ATTN_DECODE_STATIC_SCRATCH_BYTES; a larger request returns
 *     ATTN_ERR_INVALID_ARG before anything is launched (use fewer splits, a
 *     smaller batch, or attn_decode_paged);
 *   - the first call on each device looks up the array's device address with
 *     cudaGetSymbolAddress (with that device current) and keeps it for that
 *     device's context; a later call in a new context (after
 *     cudaDeviceReset) looks it up again. Make the first call on a device
 *     (and the first after a reset) before any stream capture;
 *   - every call on a device shares the one array, which keeps the last
 *     call's partials. Nothing in it needs to start at zero. Calls whose
 *     kernels can overlap on the GPU (different streams with no ordering
 *     between them, or several host threads) race on it and give wrong
 *     results: order them, e.g. issue them on one stream;
 *   - it calls no cudaMalloc, cudaFree or other allocating routine.
 */
#define ATTN_DECODE_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)
attn_status_t attn_decode_paged_static(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_table, const int32_t* seq_lens,
                                       int B, int h, int h_kv, int d_h, int page_size,
                                       int num_blocks, int max_blocks_per_seq, int num_splits,
                                       float scale, void* o, float* lse, void* stream);

/*
 * attn_merge_states -- N-way merge of split partial states, one output row
 * per input row. Follows [DEC] stage 2 ("reduce_segments") and [MRG]: over
 * the row's active splits i < n_active[row], M = max m_i, w_i = exp(m_i - M),
 * L = sum w_i l_i, o = (sum w_i O~_i) / L, lse = M + ln L. A row with no
 * active split or with M = -inf takes a branch (no -inf - -inf) and yields
 * o = 0, lse = -inf ([NA] "The base case is a NaN factory").
 *
 *   o_part   [rows, num_splits, d_h]  fp32 unnormalised accumulators (read)
 *   m_part   [rows, num_splits]       fp32 running max, natural-log units (read)
 *   l_part   [rows, num_splits]       fp32 normaliser referenced to m (read)
 *   n_active [rows] int32, may be NULL (= all num_splits active); splits at
 *            or past n_active[row] are never read
 *   o        [rows, d_h]  out_dtype (bf16 or fp32)          (written)
 *   lse      [rows]       fp32, may be NULL                 (written)
 * d_h must be 64 or 128. rows == 0 is a no-op.
 */
attn_status_t attn_merge_states(const float* o_part, const float* m_part, const float* l_part,
                                const int32_t* n_active, int rows, int num_splits, int d_h,
                                void* o, float* lse, attn_dtype_t out_dtype, void* stream);

/*
 * attn_merge_lse_pair -- merge two normalised attention results over
 * disjoint key sets, row by row. Follows [NA] "The state that gets passed
 * around is the log-sum-exp" (the symmetric merge: M = max(lse_a, lse_b),
 * e_x = exp(lse_x - M), o = (e_a o_a + e_b o_b) / (e_a + e_b), lse =
 * M + ln(e_a + e_b); the weights are formed first, so o is a convex
 * combination of o_a and o_b) and its prefix / suffix use ([NA] cascade
 * trace). An empty side has lse = -inf and weight 0; when both are empty the
 * row takes a branch and yields o = 0, lse = -inf ([NA] "The base case is a
 * NaN factory"). NaN inputs propagate; +inf is not reinterpreted.
 *
 *   o_a, o_b     [rows, d_h]  in_dtype (bf16 or fp32), normalised outputs (read)
 *   lse_a, lse_b [rows]       fp32, natural log (read)
 *   o            [rows, d_h]  out_dtype (bf16 or fp32) (written); may be
 *                o_a or o_b itself when the dtypes match (each element is read
 *                before it is written, by the same thread)
 *   lse          [rows]       fp32, may be NULL (written); must not overlap
 *                lse_a or lse_b
 * d_h must be 64 or 128. rows == 0 is a no-op. Errors: INVALID_ARG for NULL
 * inputs (rows > 0), rows < 0, unknown dtypes, pointers not 16-byte (o_a,
 * o_b, o) or 4-byte (lse) aligned, lse overlapping lse_a or lse_b;
 * UNSUPPORTED for other d_h.
 */
attn_status_t attn_merge_lse_pair(const void* o_a, const float* lse_a, const void* o_b,
                                  const float* lse_b, int rows, int d_h, attn_dtype_t in_dtype,
                                  void* o, float* lse, attn_dtype_t out_dtype, void* stream);

/*
 * attn_get_device_error -- synchronise `stream`, then read and clear the
 * device error word of every kernel module (ATTN_DEVERR_* bits, 0 = none)
 * into *bits. Returns ATTN_ERR_CUDA if the synchronisation fails.
 */
attn_status_t attn_get_device_error(void* stream, unsigned int* bits);

/*
 * attn_get_last_device_error -- the same query as a status: synchronise
 * `stream`, read and clear the device error word, and return ATTN_OK when it
 * was 0, ATTN_ERR_DEVICE_TIMEOUT when ATTN_DEVERR_WAIT_TIMEOUT was set (a
 * bounded wait gave up; that kernel's outputs are undefined), ATTN_ERR_DEVICE
 * for any other bit (a page index outside the cache, a clamped seq_len, a
 * failed tensor-memory allocation), or ATTN_ERR_CUDA if the synchronisation
 * fails.
 */
attn_status_t attn_get_last_device_error(void* stream);

/*
 * attn_selftest_wait_timeout -- exercise the failure path of the kernels'
 * bounded waits without a fault: one thread of one CTA waits, with the same
 * routine the kernels use, on an mbarrier that nothing ever arrives on, with
 * a limit of limit_us microseconds. The wait gives up, raises
 * ATTN_DEVERR_WAIT_TIMEOUT in the device error word (read it with
 * attn_get_device_error) and the kernel returns; the context stays usable.
 * limit_us in [1, 1000000]. Errors: INVALID_ARG outside that range,
 * ATTN_ERR_CUDA if the launch fails.
 */
attn_status_t attn_selftest_wait_timeout(unsigned int limit_us, void* stream);

/*
 * attn_selftest_prefill_stall -- exercise the bf16 prefill's abort path
 * without a fault; builds compiled with -DATTN_DEBUG only. From the next
 * contiguous tensor-core prefill on, every CTA skips loading K for the
 * key_tile-th key tile it visits (counted over its work items; nothing is
 * requested for that tile), so the MMA warp's bounded wait for it gives up
 * after 2 s and raises ATTN_DEVERR_WAIT_TIMEOUT; every role of the CTA then
 * stops, drains the copies and MMAs it issued, frees tensor memory and
 * exits, and the call's outputs are undefined. key_tile < 0 turns it off.
 * Device-wide (the current device) until turned off; synchronous. Errors:
 * ATTN_ERR_UNSUPPORTED in release builds, ATTN_ERR_CUDA if the device write
 * fails.
 */
attn_status_t attn_selftest_prefill_stall(int key_tile);

/*
 * attn_selftest_delayed_copy -- test aid for the decode kernels' reads before
 * their dependency wait. The split-KV decode kernel reads seq_lens and the
 * block table before it waits for the previous kernel on its stream (to warm
 * L2 with its first pages), and again after the wait for the values it
 * uses. A stale early read only happens when the kernel before it lets it
 * start early and then writes those arrays; this call is such a kernel: one
 * CTA that lets the next kernel on `stream` start at once, waits delay_us
 * microseconds (a bounded spin), then copies n int32 from src to dst (device
 * pointers). n == 0 is a no-op. Errors: INVALID_ARG for n < 0, delay_us >
 * 1000, NULL or misaligned pointers with n > 0; ATTN_ERR_CUDA if the launch
 * fails.
 */
attn_status_t attn_selftest_delayed_copy(int32_t* dst, const int32_t* src, int n,
                                         unsigned int delay_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ONLINE_SOFTMAX_ATTN_GB300_ATTN_H_ */
