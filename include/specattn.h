/*
 * specattn.h -- C ABI of the GB300 paged-attention + greedy-verification library.
 *
 * One GPU (sm_103a), one CUDA stream per call. All buffers, all device memory
 * and the stream belong to the caller; the library allocates no device memory
 * inside any call below except sa_plan_create (whose buffer lives until
 * sa_plan_destroy). Calls are asynchronous on `stream` and never synchronise
 * (unless the environment variable SA_DEBUG=1 is set, in which case each call
 * synchronises the stream and folds the device error flag into its status).
 *
 * Common conventions
 *   - `stream` is a cudaStream_t passed as void*; NULL means the legacy default
 *     stream.
 *   - bf16 tensors are passed as uint16_t bit patterns.
 *   - Host-detectable argument errors are returned synchronously and nothing
 *     is launched.
 *   - Device-detectable errors (a block-table entry outside [0, num_pages), a
 *     candidate count outside [0, k_max], q_len above the declared maximum)
 *     are OR-ed into *err_flag (an int32 in device memory, bit (1 << status)),
 *     and the affected work unit is skipped; its outputs are unspecified. The
 *     caller clears the flag and reads it when it chooses. err_flag may be
 *     NULL, in which case such errors are dropped silently.
 *   - Workspaces are caller-owned device buffers of at least the size the
 *     matching *_workspace_size call returns, 256-byte aligned. Both the
 *     sa_paged_attn and the sa_spec_verify_greedy workspace must be
 *     ZERO-FILLED BEFORE THEIR FIRST USE (they hold counters), and every call
 *     that completes without a device error leaves those counters at zero
 *     again; after a call that set a device error flag, zero the workspace
 *     again. A workspace can be reused call after call on one stream, for any
 *     shapes it is large enough for; two calls in flight at once need two
 *     workspaces.
 */
#ifndef SPECATTN_H
#define SPECATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SA_API __attribute__((visibility("default")))
#else
#define SA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SA_OK = 0,
    SA_ERR_ARG = 1,          /* bad pointer, size or shape (host check) */
    SA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. head_dim != 128) */
    SA_ERR_PAGE_OOB = 3,     /* block-table entry outside [0, num_pages) (device flag) */
    SA_ERR_CUDA = 4,         /* a CUDA runtime call failed */
    SA_ERR_TIMEOUT = 5,      /* a bounded wait inside a kernel gave up (device flag) */
    SA_ERR_WORKSPACE = 6,    /* workspace missing or too small (host check) */
    SA_ERR_QLEN = 7          /* q_lens[b] > seq_lens[b] or > max_q_len, n_cand out of range (device flag) */
} sa_status;

/* Shapes of one batch. The paged K/V layout is [num_pages, num_kv_heads,
 * page_size, head_dim]: each (page, KV head) is one contiguous
 * page_size*head_dim block (64 KiB at 256 x 128 bf16), so a page is streamed
 * with whole-block bulk copies. */
typedef struct {
    int32_t num_seqs;          /* B */
    int32_t num_q_heads;       /* Hq, a multiple of num_kv_heads */
    int32_t num_kv_heads;      /* Hkv */
    int32_t head_dim;          /* must be 128 */
    int32_t page_size;         /* must be 256 */
    int32_t num_pages;         /* physical pages in the pool */
    int32_t max_pages_per_seq; /* row stride of block_table */
    int32_t total_q;           /* sum of q_lens: rows of q and out */
    int32_t max_q_len;         /* upper bound on every q_lens[b] (1 for decode, k+1 to verify, a prefill
                                  chunk's length), <= 512 (<= 16 with a plan) */
} sa_dims;

typedef struct sa_plan sa_plan;

/* Human-readable name of a status code (static storage). */
SA_API const char *sa_status_string(int status);

/* Number of SMs of the current device (0 without a usable device). */
SA_API int sa_device_sm_count(void);

/*
 * sa_selftest_bounded_wait -- the failure path of the kernels' waits.
 *
 * Every wait of the library's kernels (on an mbarrier that copies or other
 * warps complete) gives up after a bounded number of cycles (about a quarter
 * of a second), sets bit 1 << SA_ERR_TIMEOUT of the caller's device flag and
 * returns, so that the context stays usable. This call launches one CTA that
 * makes that same wait on an mbarrier nothing completes, with no copies in
 * flight: after the limit it sets the bit in err_flag (device int32) and
 * returns. For tests of the failure path; asynchronous on `stream`.
 * Returns SA_ERR_ARG when err_flag is NULL.
 */
SA_API int sa_selftest_bounded_wait(int32_t *err_flag, void *stream);

/*
 * sa_kv_append -- write the K/V rows of the new tokens into their pages.
 *
 * ExLlamaV2 "Dynamic Generator" page, section "Continuous batching": the
 * cache is a pool of fixed 256-token pages indexed through per-sequence block
 * tables, so a sequence grows by writing through its block table.
 *
 * New token i of sequence b (0 <= i < q_lens[b]) sits at absolute position
 * p = seq_lens[b] - q_lens[b] + i; its row for KV head g goes to
 * k_pages[block_table[b][p / 256]][g][p % 256][:] (and likewise V).
 *   k_new, v_new  device bf16 [total_q, num_kv_heads, head_dim], packed
 *                 sequence after sequence in q_lens order
 *   k_pages, v_pages  device bf16 [num_pages, num_kv_heads, 256, 128]
 *   block_table   device int32 [num_seqs, max_pages_per_seq]
 *   seq_lens, q_lens  device int32 [num_seqs]; seq_lens include the new tokens
 * Writing into a page that another sequence also indexes is the caller's
 * responsibility (copy-on-write is the scheduler's job); it is not checked.
 * The kernel allows the next kernel on the stream to start early
 * (programmatic dependent launch); sa_paged_attn uses that, see there.
 */
SA_API int sa_kv_append(const sa_dims *dims, const uint16_t *k_new, const uint16_t *v_new,
                 uint16_t *k_pages, uint16_t *v_pages, const int32_t *block_table,
                 const int32_t *seq_lens, const int32_t *q_lens, int32_t *err_flag,
                 void *stream);

/*
 * sa_plan_create -- find the page runs that several sequences share.
 *
 * ExLlamaV2 "Dynamic Generator" page, section "Deduplication": several
 * sequences may index the same pages (a common prefix stored once). From host
 * copies of the block tables and lengths, the plan groups sequences whose
 * tables start with the same physical pages; paged_attn then streams each such
 * page from HBM once for the whole group, as one dense contraction on the
 * tensor cores, and attends the rest of each sequence page by page.
 *   block_table_host  host int32 [num_seqs, max_pages_per_seq]
 *   seq_lens_host, q_lens_host  host int32 [num_seqs], the values the
 *                 device arrays will hold at the paged_attn calls that use
 *                 this plan
 * The plan allocates one device buffer (its work lists) with cudaMalloc and
 * frees it in sa_plan_destroy. Make a new plan whenever the block tables or
 * lengths change. A plan with no shared runs is valid and costs nothing.
 * Plans take max_q_len <= 16 (else SA_ERR_UNSUPPORTED).
 * On success *out receives the plan.
 */
SA_API int sa_plan_create(const sa_dims *dims, const int32_t *block_table_host,
                   const int32_t *seq_lens_host, const int32_t *q_lens_host, sa_plan **out);
SA_API void sa_plan_destroy(sa_plan *plan);
/* Host-only dry run of sa_plan_create for inspection and tests: no CUDA call.
 * Fills, per sequence, the number of leading pages the shared-prefix path
 * would cover (skip_pages_out) and the partial slots it would write
 * (run_slots_out), and the numbers of shared runs and tensor-core work items
 * for a device with sm_count SMs. Output pointers may be NULL. */
SA_API int sa_plan_analyze(const sa_dims *dims, const int32_t *block_table_host,
                    const int32_t *seq_lens_host, const int32_t *q_lens_host, int32_t sm_count,
                    int32_t *skip_pages_out, int32_t *run_slots_out, int32_t *num_runs,
                    int32_t *num_tiles);
/* Shared-run statistics of a plan: runs, member sequences summed over runs,
 * logical pages summed over runs. Any pointer may be NULL. */
SA_API int sa_plan_stats(const sa_plan *plan, int32_t *num_runs, int32_t *num_members,
                  int32_t *num_pages);

/* Bytes of workspace sa_paged_attn needs for these shapes (plan may be NULL). */
SA_API size_t sa_paged_attn_workspace_size(const sa_dims *dims, const sa_plan *plan);

/*
 * sa_paged_attn -- attention of the new query tokens over the paged cache.
 *
 * For every sequence b, new token i < q_lens[b] and query head h:
 *   out[row][h] = softmax_t(scale * q[row][h] . K_b[t]) V_b[t],
 *   t = 0 .. seq_lens[b] - q_lens[b] + i  (causal inside the new tokens),
 * where row = (sum of q_lens before b) + i, K_b[t] is the row of KV head
 * h / (Hq / Hkv) at k_pages[block_table[b][t / 256]][.][t % 256], and V_b
 * likewise. ExLlamaV2 "Dynamic Generator" page, sections "Continuous
 * batching" (block-table gather) and "Deduplication" (shared pages); Hugging
 * Face "Assisted Generation" page, section "How Assisted Generation works"
 * (one forward pass over k+1 tokens scores every position). q_lens[b] = 1 is
 * plain decode.
 *   q, out       device bf16 [total_q, num_q_heads, 128]
 *   k_pages, v_pages, block_table, seq_lens, q_lens  as in sa_kv_append
 *   scale        softmax scale (1/sqrt(128) for the usual attention)
 *   plan         NULL, or a plan built from these tables and lengths
 *   workspace    device, >= sa_paged_attn_workspace_size(dims, plan) bytes
 * Accumulation is fp32; out is rounded to bf16 (nearest even).
 * Requires 0 <= q_lens[b] <= min(seq_lens[b], max_q_len). Entries of
 * block_table past a sequence's last page are never read.
 * Ordering: the call's kernels are launched as programmatic dependents, so
 * when the previous kernel on the stream is sa_kv_append (which allows an
 * early start) they begin while it runs. Before waiting for it they read only
 * the lengths and the block tables (which sa_kv_append does not write); q and
 * the pages are read after it has completed. After any other kernel, which
 * does not allow an early start, the call starts when that kernel ends.
 */
SA_API int sa_paged_attn(const sa_dims *dims, const uint16_t *q, const uint16_t *k_pages,
                  const uint16_t *v_pages, const int32_t *block_table,
                  const int32_t *seq_lens, const int32_t *q_lens, float scale, uint16_t *out,
                  const sa_plan *plan, void *workspace, size_t workspace_bytes,
                  int32_t *err_flag, void *stream);

/*
 * int8 K/V pages -- sa_kv_append_q8 and sa_paged_attn_q8.
 *
 * The ExLlamaV2 "Dynamic Generator" page, in its setup of the model and the
 * cache, names quantised cache modes (Q4 now, a Q8 mode planned) but gives no
 * format. This library's int8 format: for every (page, KV head, token) row of
 * 128 values, 128 int8 codes and one fp32 scale, with
 *   scale = amax / 127,  code = round-half-even(x / scale)
 * both computed in fp32 (IEEE division); a row of zeros has scale 0 and codes
 * 0. A cached value is code * scale. Pools:
 *   k_codes, v_codes    device int8 [num_pages, num_kv_heads, 256, 128]
 *   k_scales, v_scales  device fp32 [num_pages, num_kv_heads, 256]
 * (code pools 16-byte aligned, scale pools 16-byte aligned for attention and
 * 4-byte aligned for the append).
 *
 * sa_kv_append_q8: sa_kv_append for int8 pages: every new (token, KV head)
 * row is quantised as above and written, codes and scale, where the block
 * table puts it. Same arguments and errors as sa_kv_append.
 *
 * sa_paged_attn_q8: sa_paged_attn over int8 pages (same definition with every
 * cached value code * scale; fp32 accumulation, bf16 output). No plan, and at
 * most 128 query rows per KV head (num_q_heads / num_kv_heads * max_q_len <=
 * 128: decode and verification blocks, not prefill chunks), else
 * SA_ERR_UNSUPPORTED. The dequantisation is fused into the CUDA-core kernel;
 * above 16 rows per KV head the rows go in blocks of 16, each of which
 * streams the pages. The workspace is that of
 * sa_paged_attn_workspace_size(dims, NULL).
 */
SA_API int sa_kv_append_q8(const sa_dims *dims, const uint16_t *k_new, const uint16_t *v_new,
                           int8_t *k_codes, int8_t *v_codes, float *k_scales, float *v_scales,
                           const int32_t *block_table, const int32_t *seq_lens,
                           const int32_t *q_lens, int32_t *err_flag, void *stream);
SA_API int sa_paged_attn_q8(const sa_dims *dims, const uint16_t *q, const int8_t *k_codes,
                            const int8_t *v_codes, const float *k_scales, const float *v_scales,
                            const int32_t *block_table, const int32_t *seq_lens,
                            const int32_t *q_lens, float scale, uint16_t *out, void *workspace,
                            size_t workspace_bytes, int32_t *err_flag, void *stream);

/*
 * int4 K/V pages -- sa_kv_append_q4 and sa_paged_attn_q4.
 *
 * The Q4 cache mode that the same page names (it is the quantised mode the
 * dynamic generator takes; the page gives no format). This library's int4
 * format: for every (page, KV head, token) row of 128 values, 64 bytes of
 * 4-bit codes and one fp32 scale, with
 *   scale = amax / 7,  code = round-half-even(x / scale) clamped to [-7, 7]
 * both computed in fp32 (IEEE division), stored as the nibble code + 8; byte
 * c of the row holds value 2c in its low nibble and value 2c + 1 in its high
 * nibble. A row of zeros has scale 0 and every nibble 8. A cached value is
 * (nibble - 8) * scale. Pools:
 *   k_codes, v_codes    device uint8 [num_pages, num_kv_heads, 256, 64]
 *   k_scales, v_scales  device fp32 [num_pages, num_kv_heads, 256]
 * (alignment as for int8 pages).
 *
 * sa_kv_append_q4 and sa_paged_attn_q4: as the int8 calls above, over int4
 * pages; same arguments, restrictions and errors. sa_defrag_apply_bytes
 * moves int4 pools too (code pages of num_kv_heads * 256 * 64 bytes).
 */
SA_API int sa_kv_append_q4(const sa_dims *dims, const uint16_t *k_new, const uint16_t *v_new,
                           uint8_t *k_codes, uint8_t *v_codes, float *k_scales, float *v_scales,
                           const int32_t *block_table, const int32_t *seq_lens,
                           const int32_t *q_lens, int32_t *err_flag, void *stream);
SA_API int sa_paged_attn_q4(const sa_dims *dims, const uint16_t *q, const uint8_t *k_codes,
                            const uint8_t *v_codes, const float *k_scales, const float *v_scales,
                            const int32_t *block_table, const int32_t *seq_lens,
                            const int32_t *q_lens, float scale, uint16_t *out, void *workspace,
                            size_t workspace_bytes, int32_t *err_flag, void *stream);

/* Number of kernels one sa_paged_attn call with these shapes launches
 * (diagnostics; the same decomposition the call itself uses). Needs a device. */
SA_API int sa_paged_attn_kernel_count(const sa_dims *dims, const sa_plan *plan);

/*
 * sa_paged_attn_noalloc -- sa_paged_attn for callers that cannot allocate.
 *
 * The reference pages have no counterpart to this call; it exists for callers
 * that cannot allocate device memory at all, such as a plugin inside a serving
 * process whose memory pool owns the whole GPU, or a decode loop that may not
 * call cudaMalloc because it synchronises the device. It computes exactly what
 * sa_paged_attn computes (same arguments, no plan), but its scratch is a fixed
 * 16 MiB array inside the library. The caller still passes inputs and outputs.
 *   - Shapes whose workspace (sa_paged_attn_workspace_size with no plan) is
 *     above 16 MiB are rejected with SA_ERR_WORKSPACE before any GPU work.
 *   - The first call on a device looks up the array's device address with that
 *     device current. That lookup makes the driver load the library's device
 *     code on the device, which commits the 16 MiB there until the process
 *     exits: make the first call on each device before a memory pool reserves
 *     the rest of the device, and before any stream capture. The address is
 *     kept per device and looked up again when the device's context changes
 *     (after cudaDeviceReset).
 *   - Every call reuses the same array (partial accumulators and counters,
 *     zero when the library is loaded and left at zero by every call that
 *     completes without a device error): two calls that overlap on the GPU
 *     (different streams, or different host threads on one device) race and
 *     give wrong results.
 *   - No cudaMalloc, cudaFree or other allocating routine is called.
 */
SA_API int sa_paged_attn_noalloc(const sa_dims *dims, const uint16_t *q, const uint16_t *k_pages,
                                 const uint16_t *v_pages, const int32_t *block_table,
                                 const int32_t *seq_lens, const int32_t *q_lens, float scale,
                                 uint16_t *out, int32_t *err_flag, void *stream);

/* Bytes of workspace sa_spec_verify_greedy needs. */
SA_API size_t sa_spec_verify_workspace_size(int32_t num_seqs, int32_t k_max, int32_t vocab);

/*
 * sa_spec_verify_greedy -- greedy acceptance of draft tokens.
 *
 * Hugging Face "Assisted Generation" page, section "Assisted Generation loop",
 * steps 3-5. Per sequence b with c = candidates[b], n = n_cand[b]:
 *   t_j = lowest index of the largest logits[b][j][:], j = 0..n
 *         (NaN never wins; an all-NaN row gives 0; -0.0 == +0.0)
 *   accepted[b] = largest a <= n with c_j == t_j for every j < a
 *   next_tok[b] = t_{accepted[b]}  (the correction, or the bonus token when
 *                 all n candidates matched)
 *   window[b]  <- window[b] + 2 if accepted[b] == n, else max(1, window[b] - 1)
 *   logits       device fp32 [num_seqs, k_max + 1, vocab]
 *   candidates   device int32 [num_seqs, k_max]
 *   n_cand       device int32 [num_seqs], each in 0..k_max
 *   accepted, next_tok  device int32 [num_seqs] (outputs)
 *   window       device int32 [num_seqs], updated in place; may be NULL
 *   workspace    device, >= sa_spec_verify_workspace_size(...) bytes
 * Results are exact (integer); k_max <= 15.
 */
SA_API int sa_spec_verify_greedy(const float *logits, const int32_t *candidates, const int32_t *n_cand,
                          int32_t num_seqs, int32_t k_max, int32_t vocab, int32_t *accepted,
                          int32_t *next_tok, int32_t *window, void *workspace,
                          size_t workspace_bytes, int32_t *err_flag, void *stream);

/*
 * sa_spec_verify_greedy_advance -- sa_spec_verify_greedy, then the shapes of
 * the next verify call, in the same launch.
 *
 * Hugging Face "Assisted Generation" page, section "Assisted Generation
 * loop": after step 5 adjusts the window the loop returns to step 1, the
 * assistant drafting as many tokens as the window says. Reading (the page
 * speaks of tokens, not of a cache): this call's new tokens are the previous
 * step's last token followed by the n_cand[b] candidates, so the sequence
 * keeps seq_lens[b] - q_lens[b] + 1 + accepted[b] tokens (the cache rows of
 * the rejected candidates are simply overwritten by the next append); the
 * next call opens with next_tok[b] followed by min(window, k_max) candidates.
 * Everything sa_spec_verify_greedy does, plus, per sequence b:
 *   window[b]       <- the adjusted window (as there; required here)
 *   n_cand_next[b]  <- n = min(window[b], k_max)   (device int32 [num_seqs])
 *   q_lens[b]       <- n + 1                       (device int32, in/out)
 *   seq_lens[b]     <- seq_lens[b] - q_lens[b] + 1 + accepted[b] + n + 1
 *                                                  (device int32, in/out)
 * so the next step's kv_append, paged_attn and verify read their lengths
 * straight from these buffers with no host round trip. n_cand_next may be
 * the n_cand buffer itself (every read of n_cand[b] precedes the write). A
 * sequence with q_lens[b] < n_cand[b] + 1 or seq_lens[b] < q_lens[b] gets
 * SA_ERR_QLEN in *err_flag and its window and lengths are left unchanged.
 * Other arguments, the workspace and the errors as in sa_spec_verify_greedy.
 */
SA_API int sa_spec_verify_greedy_advance(const float *logits, const int32_t *candidates,
                                         const int32_t *n_cand, int32_t num_seqs, int32_t k_max,
                                         int32_t vocab, int32_t *accepted, int32_t *next_tok,
                                         int32_t *window, int32_t *seq_lens, int32_t *q_lens,
                                         int32_t *n_cand_next, void *workspace, size_t workspace_bytes,
                                         int32_t *err_flag, void *stream);

/*
 * sa_defrag_moves -- compaction plan for a fragmented cache (host only, no
 * CUDA call).
 *
 * ExLlamaV2 "Dynamic Generator" page, section "Continuous batching": freeing
 * a finished job's pages leaves holes, the block table need not be
 * contiguous, and the cache can be defragmented (the generator does it only
 * when its job queue is empty). The page gives no procedure; this call's
 * reading: a page is live when a table names it within its sequence's
 * length (the first ceil(seq_lens[b] / 256) entries). With L live pages,
 * every live page whose id is L or more moves into a free id below L, the
 * k-th such page (by increasing id) into the k-th free id (by increasing id);
 * live pages below L stay. Tables are rewritten through the same map, so a
 * page shared by several sequences stays shared.
 *   block_table  host int32 [num_seqs, max_pages_per_seq]
 *   seq_lens     host int32 [num_seqs]
 *   new_table    host int32 [num_seqs, max_pages_per_seq] (output): the
 *                remapped table; entries past a sequence's length are -1
 *   moves        host int32 [num_pages][2] (output): (from, to) page pairs,
 *                *n_moves of them, by increasing from; no page is both a
 *                from and a to, and no to repeats
 *   n_moves, n_live  host int32 (outputs)
 * Uses num_seqs, num_pages and max_pages_per_seq of dims. Errors:
 * SA_ERR_ARG (a NULL pointer, a negative length, a length that needs more
 * than max_pages_per_seq pages), SA_ERR_PAGE_OOB (a used entry outside
 * [0, num_pages)); outputs are then unspecified.
 */
SA_API int sa_defrag_moves(const sa_dims *dims, const int32_t *block_table, const int32_t *seq_lens,
                           int32_t *new_table, int32_t *moves, int32_t *n_moves, int32_t *n_live);

/*
 * sa_defrag_apply -- make the moves of a compaction plan: for every (from,
 * to) pair, page `to` of k_pages and of v_pages gets page `from`'s rows
 * (every KV head). Same page and section as sa_defrag_moves.
 *   k_pages, v_pages  device bf16 [num_pages, num_kv_heads, 256, 128]
 *   moves        device int32 [n_moves][2]; no page may be both read and
 *                written and no page written twice (as sa_defrag_moves
 *                gives them); otherwise the result is unspecified
 * A pair naming a page outside [0, num_pages) sets SA_ERR_PAGE_OOB in
 * *err_flag and is skipped. One kernel; n_moves = 0 launches nothing.
 */
SA_API int sa_defrag_apply(const sa_dims *dims, uint16_t *k_pages, uint16_t *v_pages,
                           const int32_t *moves, int32_t n_moves, int32_t *err_flag, void *stream);

/*
 * sa_defrag_apply_bytes -- the same moves on any two pools paged alike:
 * page p of a pool is the page_bytes bytes at p * page_bytes. For int8 pages
 * (sa_kv_append_q8), call it once for the code pools (page_bytes =
 * num_kv_heads * 256 * 128) and once for the scale pools (num_kv_heads * 256
 * * 4). page_bytes a multiple of 16, pools 16-byte aligned (else SA_ERR_ARG);
 * moves and errors as in sa_defrag_apply.
 */
SA_API int sa_defrag_apply_bytes(int32_t num_pages, int64_t page_bytes, void *pool_a, void *pool_b,
                                 const int32_t *moves, int32_t n_moves, int32_t *err_flag, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECATTN_H */
