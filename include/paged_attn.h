/*
 * paged_attn.h -- C ABI of the GB300 (sm_103a) paged-KV GQA attention library.
 *
 * Operation.  For every sequence b, new-token row i in [0, q_len) and query head h:
 *   g   = h / (num_q_heads / num_kv_heads)            GQA: contiguous groups of query heads
 *                                                       share one K/V head (studybook
 *                                                       fde-roadmap ch.10 "production latency
 *                                                       and cost", section 10.1.2)
 *   L   = context_lens[b]                              tokens in the cache, new ones included
 *   n   = L - q_len + i + 1                            causal: row i sees itself and everything
 *                                                       before it (sirzzang "Speculative
 *                                                       Decoding", parallel verification and
 *                                                       its causal-mask figure)
 *   k_j = K[block_table[b][j / bs], g, j % bs, :]      paged gather through the block table
 *   v_j = V[block_table[b][j / bs], g, j % bs, :]      (section 10.4.2, figure 10.4.2; aegloslab
 *                                                       servingai 5.3.7)
 *   s_j = scale * <q[b, i, h, :], k_j>,  j < n
 *   out[b, i, h, :] = sum_j softmax(s)_j v_j           attention over the cached K/V
 *                                                       (section 10.3.1), computed tile by tile
 *                                                       with an online softmax (10.1.2)
 * fp8 caches hold OCP E4M3 bytes; the value of a byte is e4m3(byte) * k_scale[block, g] (or
 * v_scale) with one fp32 scale per (physical block, kv head) -- the symmetric scale
 * quantisation of section 10.8.2.
 *
 * Layouts (row-major, contiguous, element sizes in brackets):
 *   q            [num_seqs, q_len, num_q_heads, head_dim]        bf16 [2]
 *   k_cache,
 *   v_cache      [num_blocks, num_kv_heads, block_size, head_dim] bf16 [2] or E4M3 [1]
 *   k_scale,
 *   v_scale      [num_blocks, num_kv_heads]                      fp32 [4]; NULL for bf16
 *   block_table  [num_seqs, max_blocks_per_seq]                   int32; entries past
 *                                                                 ceil(L / block_size) are
 *                                                                 never read
 *   context_lens [num_seqs]                                       int32
 *   out          [num_seqs, q_len, num_q_heads, head_dim]        bf16 [2]
 *
 * Ownership.  Every pointer argument is a device pointer owned by the caller; the library
 * never frees or retains one after the call returns.  Calls are asynchronous on `stream`
 * (a cudaStream_t; NULL is the legacy default stream) and do not synchronise it.
 *
 * Scratch.  When a sequence's context is split into several partitions the library keeps
 * per-partition partial results in stream-ordered scratch memory that it allocates from a
 * memory pool of its own (one per device) on `stream` and frees on `stream` after the merge.
 *
 * Errors.  Every entry point returns a pa_status.  Argument checks run on the host before any
 * launch; a failed check launches nothing.  PA_OK from an attention call means the kernels were
 * launched.  Conditions only the device can see (a block id outside [0, num_blocks), a
 * sequence with fewer than q_len tokens, an asynchronous copy that did not complete within
 * its wait limit) never fault: the affected page is skipped or the affected rows are written
 * as zeros, and a per-device error word records it for paged_attn_check_device_errors.
 */
#ifndef PAGED_ATTN_H_
#define PAGED_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,   /* a null pointer, a negative size, Hq % Hkv != 0, ...            */
  PA_ERR_UNSUPPORTED = 2,   /* a valid shape the kernels are not built for                     */
  PA_ERR_CUDA = 3,          /* a CUDA runtime call or a launch failed                          */
  PA_ERR_NO_MEMORY = 4,     /* the split-KV scratch could not be allocated                     */
  PA_ERR_DEVICE_BOUNDS = 5, /* device-side: a block id was out of range or a context too short */
  PA_ERR_DEVICE_TIMEOUT = 6, /* device-side: an asynchronous copy wait hit its iteration limit */
  PA_ERR_SCRATCH_LIMIT = 7   /* the static-scratch decode needs more than its fixed array      */
} pa_status;

typedef enum { PA_KV_BF16 = 0, PA_KV_FP8_E4M3 = 1 } pa_kv_dtype;

/*
 * Single-token decode for a continuous batch with ragged context lengths (studybook section
 * 10.2.2: one new token per step reads the whole cache; aegloslab servingai 5.3.1).
 *   q_len must be 1.  head_dim in {64, 128}; block_size 16; num_q_heads / num_kv_heads at most
 *   64; kv_dtype a pa_kv_dtype (k_scale/v_scale required for fp8, ignored for bf16).  max_context_len is a host-known upper bound of context_lens (it sizes the grid
 *   without reading device memory); it must not exceed max_blocks_per_seq * block_size.
 *   `scale` multiplies q.k (1/sqrt(head_dim) for standard attention).
 * Kernel: split-KV partitions (paged_attn_plan) merged by log-sum-exp; within a partition both
 * products run on the warp-level tensor-core instruction (mma.sync m16n8k16, fp32 accumulation,
 * the G heads as the columns of an 8-wide tile): bf16 caches in bf16, with each softmax weight
 * carried as a bf16 high part plus its rounded remainder (~16 significant bits); E4M3 caches
 * converted exactly to f16 pairs in registers, weights in f16 with each page's V scale folded in,
 * and q re-encoded as f16 after a power of two per query head that brings its largest |q| just
 * below 2^15 (exact for every element within 2^28 of the largest; the scores are scaled back),
 * so any bf16 q is accepted.  That kernel serves groups of 1, 2, 4 and
 * 8 query heads; any other group (3, 5, 7, 16, ...) runs the tcgen05 kernel of paged_attn_verify
 * with q_len = 1 (its balanced persistent split).
 */
int paged_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_table, const int32_t* context_lens, int num_seqs,
                      int max_blocks_per_seq, int num_blocks, int max_context_len, int q_len,
                      int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                      float scale, int kv_dtype, const float* k_scale, const float* v_scale,
                      void* out, void* stream);

/*
 * (K+1)-query causal verify forward of speculative decoding: the target scores the q_len =
 * K+1 newest tokens (K drafts plus the bonus position) in one call, row i masked to the
 * tokens up to itself (sirzzang "Speculative Decoding", parallel verification; aegloslab
 * servingai 5.3.9).  The new tokens' K/V must already be in the cache and context_lens counts
 * them.  Same arguments and limits as paged_attn_decode, with 1 <= q_len <= 16 and
 * (num_q_heads / num_kv_heads) * q_len <= 128 (rows beyond 64 per kv head -- e.g. 8 drafts under
 * groups of 8 -- run the chunked-prefill kernel, split into partitions like decode and merged
 * the same way).  bf16 caches run the products in bf16; E4M3 caches are converted exactly to
 * f16 in shared memory and the products run in f16 (each Q row re-encoded as f16 after the power
 * of two that keeps it in range, as for decode; each page's scales are applied to its scores and
 * weights), fp32 accumulation in both.
 */
int paged_attn_verify(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_table, const int32_t* context_lens, int num_seqs,
                      int max_blocks_per_seq, int num_blocks, int max_context_len, int q_len,
                      int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                      float scale, int kv_dtype, const float* k_scale, const float* v_scale,
                      void* out, void* stream);

/*
 * Tree verification: paged_attn_verify with the causal mask over the q_len new tokens replaced
 * by an ancestor mask, so that one forward scores a tree of draft branches (tree attention,
 * aegloslab servingai 5.3.13; Medusa-style candidate trees, sirzzang "Speculative Decoding").
 *   tree_mask [num_seqs, q_len] uint32, device: bit t of tree_mask[b * q_len + i] set means new
 *   token i attends to new token t (normally t = i and i's ancestors); every context token
 *   before the q_len new ones is visible to every row.  The chain mask (bits 0..i) reproduces
 *   paged_attn_verify.  A row whose mask and prefix are both empty comes out as zeros.
 * Same arguments, limits and errors as paged_attn_verify; a NULL tree_mask is
 * PA_ERR_INVALID_ARG.
 */
int paged_attn_tree_verify(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_table, const int32_t* context_lens,
                           const uint32_t* tree_mask, int num_seqs, int max_blocks_per_seq,
                           int num_blocks, int max_context_len, int q_len, int num_q_heads,
                           int num_kv_heads, int head_dim, int block_size, float scale,
                           int kv_dtype, const float* k_scale, const float* v_scale, void* out,
                           void* stream);

/*
 * Paged attention over packed, variable-length query rows: chunked prefill (a prompt chunk
 * attends to everything cached before it and causally within itself; aegloslab servingai 5.3.15,
 * Sarathi-style chunking with piggybacked decode) and, in the same call, decode (1 row) or verify
 * (K + 1 rows) sequences.  FlashAttention tiling with an online softmax (studybook fde-roadmap
 * ch.10, section 10.1.2) on the tensor cores, 128-row tiles of (token, query head) per kv head.
 *   q                [total_q, num_q_heads, head_dim] bf16, device, 16-byte aligned: sequence b's
 *                    new rows are q[query_start_loc[b] .. query_start_loc[b+1]).
 *   query_start_loc  [num_seqs + 1] int32, device, non-decreasing, query_start_loc[num_seqs] <=
 *                    total_q; q_len_b = query_start_loc[b+1] - query_start_loc[b] <= max_q_len.
 *   context_lens     [num_seqs] int32, device: cached tokens including the q_len_b new ones (their
 *                    K/V are in the cache: paged_attn_append_kv); new row i sees
 *                    context_lens[b] - q_len_b + i + 1 tokens.
 *   out              [total_q, num_q_heads, head_dim] bf16, device: written for every packed row.
 *   max_q_len        host-side bound on q_len_b (sizes the grid); total_q the rows of q and out.
 * Other arguments as paged_attn_decode.  Limits: bf16 or E4M3 KV (E4M3: k_scale / v_scale
 * required; pages converted exactly to f16 in shared memory, products in f16 with Q rows
 * re-encoded as in paged_attn_verify), head_dim 64 or 128, block_size 16, num_q_heads /
 * num_kv_heads in {1, 2, 4, 8}.  Device-side: a sequence whose rows fall outside
 * [0, total_q) or exceed max_q_len is skipped and flagged; rows that see no token (context
 * shorter than the new rows) come out as zeros and are flagged (PA_ERR_DEVICE_BOUNDS from
 * paged_attn_check_device_errors).  Asynchronous on `stream`; its work list (4 bytes per
 * (sequence, tile) pair) comes from the library's stream-ordered pool.  Returns PA_OK (also for
 * num_seqs == 0 or total_q == 0), PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_NO_MEMORY or
 * PA_ERR_CUDA.
 */
int paged_attn_prefill(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_table, const int32_t* context_lens,
                       const int32_t* query_start_loc, int num_seqs, int total_q, int max_q_len,
                       int max_blocks_per_seq, int num_blocks, int max_context_len,
                       int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                       float scale, int kv_dtype, const float* k_scale, const float* v_scale,
                       void* out, void* stream);

/*
 * KV append: store the new tokens' K and V in the paged cache, the step that precedes the
 * attention call of each decode or verify step (studybook fde-roadmap ch.10, sections 10.2.2
 * and 10.3.2: the step's K/V join the cache; section 10.12.2 and aegloslab servingai 5.3.7:
 * position j lives in slot j % block_size of block block_table[b][j / block_size]).
 *   k_new, v_new [num_seqs, n_new, num_kv_heads, head_dim] bf16, device, 16-byte aligned.
 *   k_cache, v_cache, block_table, as in paged_attn_decode; written in place.
 *   context_lens [num_seqs] int32, device: lengths AFTER the append; sequence b's new tokens
 *     take positions [context_lens[b] - n_new, context_lens[b]).
 *   kv_dtype PA_KV_BF16: the rows are stored unchanged.
 *   kv_dtype PA_KV_FP8_E4M3: k_scale / v_scale [num_blocks, num_kv_heads] fp32, device, read
 *     and written.  Each touched (block, head) gets the scale amax / 448 over its valid tokens
 *     (1 if all are zero) -- symmetric per-block scale quantisation (studybook section 10.8.2);
 *     the older tokens of the block are re-encoded when the scale changes.  All arithmetic is
 *     fp32; E4M3 rounding is to nearest even, saturating at +-448.
 * Slots past each sequence's last token are not touched.  Blocks written must belong to their
 * sequence alone (copy a shared block before appending to it).  Sequences whose context is
 * shorter than n_new, and out-of-range block ids, are skipped and flagged in the error word
 * (PA_ERR_DEVICE_BOUNDS from paged_attn_check_device_errors).  Asynchronous on `stream`; never
 * allocates.  Returns PA_OK (also for num_seqs == 0 or n_new == 0: nothing is launched),
 * PA_ERR_INVALID_ARG (NULL pointer, negative size, misaligned row pointer, n_new above the
 * table's capacity), PA_ERR_UNSUPPORTED (block_size != 16, head_dim not 64 or 128) or
 * PA_ERR_CUDA.
 */
int paged_attn_append_kv(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                         const int32_t* block_table, const int32_t* context_lens, int num_seqs,
                         int n_new, int max_blocks_per_seq, int num_blocks, int num_kv_heads,
                         int head_dim, int block_size, int kv_dtype, float* k_scale,
                         float* v_scale, void* stream);

/*
 * Speculative acceptance, the step after paged_attn_verify: decide which of the K drafted tokens
 * a round keeps and draw the token that ends the round (speculative sampling: studybook
 * fde-roadmap ch.10, section 10.6.2; aegloslab servingai 5.3.10; sirzzang "Speculative
 * Decoding", verification).  Per sequence, left to right, draft i is accepted when
 * p_i(x_i) >= q_i(x_i), else when u_accept[i] < p_i(x_i) / q_i(x_i) (IEEE fp32 division); the
 * first rejection at i ends the round with a token drawn from norm(max(0, p_i - q_i)) (from p_i
 * if that residual has no mass); if all K are accepted a bonus token is drawn from p_K.  A draw
 * from weights r uses the sequence's 32-bit word: w(x) = floor(min(max(r, 0), 1) * 2^40),
 * Z = sum w, T = floor(Z * word / 2^32), token = smallest x whose inclusive prefix of w exceeds T
 * (integer sums: the result does not depend on the order of summation).
 *   p            [num_seqs, num_draft + 1, vocab_size] fp32, device: target probabilities at the
 *                K + 1 verified positions (softmax of the verify forward's logits).
 *   q            [num_seqs, num_draft, vocab_size] fp32, device: draft probabilities at the K
 *                drafted positions.  May be NULL when num_draft == 0.
 *   draft_tokens [num_seqs, num_draft] int32, device.
 *   u_accept     [num_seqs, num_draft] fp32 in [0, 1), device: one uniform per draft.
 *   u_sample     [num_seqs] uint32, device: one uniform word per round.
 *   out_tokens   [num_seqs, num_draft + 1] int32, device, written: the accepted drafts, then the
 *                replacement or bonus token, then -1.
 *   num_accepted [num_seqs] int32, device, written: accepted drafts (the round emits this + 1).
 * A draft token outside [0, vocab_size) makes that sequence emit nothing (num_accepted -1, all
 * tokens -1) and sets the error word (PA_ERR_DEVICE_BOUNDS from paged_attn_check_device_errors);
 * so does a draw whose weights are all zero (token -1).  Scratch (8 bytes per 4096 vocabulary
 * entries per sequence) comes from the library's stream-ordered pool.  Asynchronous on
 * `stream`.  Returns PA_OK (also for num_seqs == 0), PA_ERR_INVALID_ARG (NULL pointer, negative
 * size), PA_ERR_UNSUPPORTED (num_draft > 31, vocab_size > 2^21, num_seqs > 65535),
 * PA_ERR_NO_MEMORY or PA_ERR_CUDA.
 */
int paged_attn_spec_accept(const float* p, const float* q, const int32_t* draft_tokens,
                           const float* u_accept, const uint32_t* u_sample, int num_seqs,
                           int num_draft, int vocab_size, int32_t* out_tokens,
                           int32_t* num_accepted, void* stream);

/*
 * Synchronises `stream`, then reads and clears the current device's error word.  Returns
 * PA_OK, PA_ERR_DEVICE_BOUNDS or PA_ERR_DEVICE_TIMEOUT (bounds wins when both are set), or
 * PA_ERR_CUDA.  Not from the pages: a diagnostic of this library.
 */
int paged_attn_check_device_errors(void* stream);

/*
 * Failure-detection self-test (not from the pages: a diagnostic of this library).  Launches one
 * warp on `stream` whose first thread waits on a shared-memory mbarrier that nothing ever
 * arrives at, through the same bounded wait the kernels use, cut off after `polls` polls:
 * helper 0 = the decode kernels' wait, helper 1 = the tcgen05 kernels' wait (which also
 * raises the CTA's abort flag), both made of suspending mbarrier.try_wait polls; helper 2 = a
 * loop of non-suspending mbarrier.test_wait probes, the form of the tensor-core issuers' idle
 * loops.  The wait gives up, the error word records a timeout (PA_ERR_DEVICE_TIMEOUT from
 * paged_attn_check_device_errors) and the kernel returns normally, so the context stays usable.
 * The kernels cut suspending waits off after PA_WAIT_LIMIT polls and idle loops after
 * PA_SPIN_LIMIT iterations; elapsed_ns / polls gives the time of one poll, hence of a full wait.
 *   polls       in [1, PA_WAIT_LIMIT] for helpers 0 and 1, [1, PA_SPIN_LIMIT] for helper 2;
 *   elapsed_ns  one uint64, device, 8-byte aligned, written: wall time of the wait (globaltimer).
 * Returns PA_OK (launched), PA_ERR_INVALID_ARG (helper not 0, 1 or 2, polls out of range, NULL
 * or misaligned elapsed_ns) or PA_ERR_CUDA.
 */
#define PA_WAIT_LIMIT (1u << 18)
#define PA_SPIN_LIMIT (1u << 22)
int paged_attn_selftest_wait(int helper, unsigned int polls, unsigned long long* elapsed_ns,
                             void* stream);

/* Static description of a status code (never NULL). */
const char* paged_attn_status_string(int status);

/*
 * Split-KV planning of paged_attn_decode.  A sequence's pages are cut into partitions of
 * pages_per_partition pages; each (sequence, kv head, partition) is one CTA and a log-sum-exp
 * merge combines the partitions.  paged_attn_set_max_partitions(p > 0) forces at most p
 * partitions per sequence (p = 1 disables splitting); p = 0 restores the automatic choice.
 * Process-wide setting.  Returns PA_OK or PA_ERR_INVALID_ARG (p < 0 or p > 4096).
 * (paged_attn_verify balances its work on the device instead: the pages of all sequences and kv
 * heads are laid end to end and cut into equal ranges, one per resident CTA, with the pieces of a
 * sequence merged by the same log-sum-exp rule; this setting does not affect it.)
 */
int paged_attn_set_max_partitions(int p);

/*
 * The split the library would choose for paged_attn_decode, as a pure function of the shape (no
 * CUDA call): writes pages_per_partition and the partition count of the longest sequence.  The
 * automatic plan aims at 8 CTAs per SM for bf16 pages and 4 for E4M3 pages (half the bytes per
 * CTA), with partitions of at most 64 (bf16) or 256 (E4M3) pages where 64 partitions allow.  num_sms is the device's SM
 * count (152 on GB300).  Returns PA_OK or PA_ERR_INVALID_ARG.
 */
int paged_attn_plan(int num_sms, int num_seqs, int num_kv_heads, int max_context_len,
                    int block_size, int q_len, int kv_dtype, int* pages_per_partition,
                    int* max_partitions);

/*
 * Decode that allocates nothing (no counterpart on the pages: a service of this library).
 *
 * For callers that cannot allocate device memory while they serve -- a host framework whose
 * memory manager reserved the GPU's memory up front, or a real-time loop that forbids
 * allocation after start-up.  Same arguments and limits as paged_attn_decode except that the
 * group (num_q_heads / num_kv_heads) must be 1, 2, 4 or 8 (else PA_ERR_UNSUPPORTED), and the same
 * results within its tolerances (it runs the library's CUDA-core decode kernel, fp32 FMAs), but
 * the split-KV partials live in a fixed array in the library's device image
 * (paged_attn_static_scratch_bytes() bytes, 32 MiB, held on every GPU that loads the library
 * until the process exits) instead of stream-ordered pool memory.  The call makes no
 * cudaMalloc, cudaMallocAsync, cudaFree or other allocating call.
 *   - The first call on a device looks up the array's device address (with that device
 *     current); make that first call before capturing any stream.
 *   - Every call shares the one array: calls whose kernels overlap on the GPU (different
 *     streams, or several host threads) race on it.  Serialise them, e.g. on one stream.
 *   - A shape whose partials need more than the array returns PA_ERR_SCRATCH_LIMIT and
 *     launches nothing: partials take num_seqs * q_len * num_q_heads * P * (head_dim + 1) * 4
 *     bytes when the plan splits into P > 1 partitions (paged_attn_plan), none when P = 1.
 *   - On PA_ERR_CUDA the contents of `out` are undefined: a launch may have failed after an
 *     earlier one of the same call had already written some rows.
 */
int paged_attn_decode_static_scratch(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_table, const int32_t* context_lens,
                                     int num_seqs, int max_blocks_per_seq, int num_blocks,
                                     int max_context_len, int q_len, int num_q_heads,
                                     int num_kv_heads, int head_dim, int block_size, float scale,
                                     int kv_dtype, const float* k_scale, const float* v_scale,
                                     void* out, void* stream);

/* Size in bytes of the fixed array paged_attn_decode_static_scratch uses. */
size_t paged_attn_static_scratch_bytes(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int paged_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_ATTN_H_ */
