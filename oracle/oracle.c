/*
 * oracle.c -- CPU fp64 oracle for paged attention and greedy verification.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, includes
 * or calls this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it. It shares no code with the CUDA path.
 *
 * It states the plain definitions, slowly and in double precision:
 *
 *  - kv_append: the K/V rows of a sequence's new tokens are written into
 *    the page that the sequence's block table names for their position,
 *    at slot (position mod page size).  ExLlamaV2 "Dynamic Generator" page,
 *    section "Continuous batching": the cache is indexed through a block
 *    table of fixed 256-token pages, and adding or removing sequences only
 *    touches block indices.
 *
 *  - attention: for every new query token of every sequence, gather the
 *    sequence's keys and values page by page into contiguous arrays, take
 *    softmax(scale * q.K^T) over the keys the token may see, and weight the
 *    values with it.  Same page and section for the block-table gather; the
 *    "Deduplication" section for pages shared between sequences (nothing
 *    special is done: a shared page is simply read by each sequence that
 *    names it).  Query token i of a sequence with q_len new tokens and
 *    seq_len cached tokens sits at position seq_len - q_len + i and sees
 *    keys 0 .. seq_len - q_len + i (causal inside the new tokens): the
 *    Hugging Face "Assisted Generation" page, section "How Assisted
 *    Generation works", says one forward pass over a token sequence yields
 *    logits at every position, which is what this masking gives.
 *    Query head h uses KV head h / (Hq / Hkv) (contiguous grouping; the
 *    pages are silent on grouped heads, this is the plain reading).
 *
 *  - greedy verification: per verifier row take the lowest index of the
 *    largest logit; compare the draft candidates with these left to right;
 *    the accepted count is the length of the matching prefix and the
 *    correction token is the verifier's token at the first mismatch (at the
 *    bonus row when every candidate matched); the draft window grows by 2
 *    when every candidate matched and shrinks by 1 otherwise.  Hugging Face
 *    "Assisted Generation" page, section "Assisted Generation loop", steps
 *    3 (comparison), 4 (correction) and 5 (adjustment); step 1 gives the
 *    initial window of 5.  Readings where the page is silent: the window
 *    never drops below 1; with zero candidates nothing can mismatch, so the
 *    window grows; NaN never wins an argmax and an all-NaN row gives 0;
 *    -0.0 and +0.0 compare equal (a tie).
 *
 *  - the next step of the loop: the same page's loop returns to step 1
 *    after step 5, the assistant drafting as many tokens as the adjusted
 *    window says. Reading of the cache (the page speaks of tokens, not of a
 *    cache): the verify call's new tokens are [the last token of the previous
 *    step, candidate 0 .. candidate n-1], so after step 4 the sequence holds
 *    the tokens before the call, that first token and the accepted
 *    candidates (seq_len - q_len + accepted + 1 tokens); the correction
 *    token opens the next call, followed by min(window, k_max) candidates
 *    (k_max being the most the caller's buffers take), so the next call has
 *    q_len = that count + 1 and seq_len = the kept tokens + q_len.
 *
 *  - int8 pages: the ExLlamaV2 "Dynamic Generator" page, in its setup of the
 *    model and cache, names quantised cache modes (Q4 now, Q8 planned) but
 *    defines no format. Reading: every (page, KV head, token) row of 128 values
 *    is stored as 128 int8 codes and one binary32 scale, scale = amax / 127,
 *    code = round-to-nearest-even(x / scale) in binary32; a cached value is
 *    code * scale, and attention is the plain definition over those values.
 *
 *  - int4 pages (the Q4 mode that page names): the same reading with 4-bit
 *    codes, scale = amax / 7, code = round-to-nearest-even(x / scale) clamped
 *    to [-7, 7], stored as the nibble code + 8; the row's byte c holds value
 *    2c in its low nibble and value 2c + 1 in its high nibble.
 *
 *  - defragmentation: releasing pages leaves holes in the cache; the block
 *    table need not be contiguous, and the cache can be defragmented (the
 *    generator does it only when its job queue is empty).  ExLlamaV2
 *    "Dynamic Generator" page, section "Continuous batching".  Reading (the
 *    page gives no procedure): a page is live when some sequence's table
 *    names it within that sequence's length; with L live pages, every live
 *    page whose id is L or more moves into a free id below L, the k-th such
 *    page (in increasing id) into the k-th free id (in increasing id); live
 *    pages below L stay.  Tables are rewritten through the same map, so
 *    shared pages stay shared; entries past a sequence's length become -1.
 *    Moving copies each moved page's K and V rows for every KV head.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC (no fast-math, so
 * the arithmetic is the order written here on every machine).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_OK = 0, ORACLE_ERR_ARG = 1, ORACLE_ERR_PAGE_OOB = 3, ORACLE_ERR_NOMEM = 7 };

/* bf16 bit pattern -> double, exact: bf16 is the top half of an IEEE binary32. */
double oracle_bf16_to_f64(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Physical page holding position `pos` of sequence `b`, or -1 if the block
 * table entry is out of range. */
static int64_t page_of(const int32_t *block_table, int max_pages_per_seq, int num_pages,
                       int page_size, int b, int64_t pos) {
    int64_t j = pos / page_size;
    if (j >= max_pages_per_seq) return -1;
    int32_t id = block_table[(int64_t)b * max_pages_per_seq + j];
    if (id < 0 || id >= num_pages) return -1;
    return id;
}

/* ---------------------------------------------------------------- kv_append */

int oracle_kv_append(int num_seqs, int num_kv_heads, int head_dim, int page_size,
                     int num_pages, int max_pages_per_seq,
                     const uint16_t *k_new, const uint16_t *v_new,
                     uint16_t *k_pages, uint16_t *v_pages,
                     const int32_t *block_table, const int32_t *pos_start,
                     const int32_t *new_lens) {
    if (num_seqs < 0 || num_kv_heads <= 0 || head_dim <= 0 || page_size <= 0) return ORACLE_ERR_ARG;
    int64_t row = 0; /* new tokens are packed sequence after sequence */
    for (int b = 0; b < num_seqs; ++b) {
        for (int i = 0; i < new_lens[b]; ++i, ++row) {
            int64_t pos = (int64_t)pos_start[b] + i;
            int64_t pg = page_of(block_table, max_pages_per_seq, num_pages, page_size, b, pos);
            if (pg < 0) return ORACLE_ERR_PAGE_OOB;
            int64_t slot = pos % page_size;
            for (int g = 0; g < num_kv_heads; ++g) {
                int64_t dst = ((pg * num_kv_heads + g) * page_size + slot) * head_dim;
                int64_t src = (row * num_kv_heads + g) * head_dim;
                for (int c = 0; c < head_dim; ++c) {
                    k_pages[dst + c] = k_new[src + c];
                    v_pages[dst + c] = v_new[src + c];
                }
            }
        }
    }
    return ORACLE_OK;
}

/* ---------------------------------------------------------------- attention */

typedef struct {
    int num_seqs, num_q_heads, num_kv_heads, head_dim, page_size, num_pages, max_pages_per_seq;
    const uint16_t *q, *k_pages, *v_pages;
    const int32_t *block_table, *seq_lens, *q_lens;
    double scale;
    /* int8 pages (NULL for bf16 pages): value = code * the row's scale */
    const int8_t *k_codes, *v_codes;
    const float *k_scales, *v_scales;
    /* int4 pages (NULL otherwise): packed nibbles, value = (nibble - 8) * scale */
    const uint8_t *k_nib, *v_nib;
} attn_args;

/* One output row: new token i of sequence b, query head h. `kbuf`/`vbuf`
 * hold at least seq_len*head_dim doubles, `s` at least seq_len. */
static int attention_row(const attn_args *a, const int64_t *q_row_of_seq, int b, int i, int h,
                         double *kbuf, double *vbuf, double *s, double *o) {
    const int d = a->head_dim;
    const int group = a->num_q_heads / a->num_kv_heads;
    const int g = h / group;
    const int64_t T = a->seq_lens[b];
    const int64_t n = a->q_lens[b];
    const int64_t p = T - n + i; /* absolute position of this query token */
    const int64_t nkeys = p + 1;

    /* 1. gather keys/values 0..p through the block table into contiguous arrays */
    for (int64_t t = 0; t < nkeys; ++t) {
        int64_t pg = page_of(a->block_table, a->max_pages_per_seq, a->num_pages, a->page_size, b, t);
        if (pg < 0) return ORACLE_ERR_PAGE_OOB;
        int64_t srow = (pg * a->num_kv_heads + g) * a->page_size + t % a->page_size;
        int64_t base = srow * d;
        if (a->k_nib) { /* int4 pages: row srow is d / 2 bytes, value c in nibble c % 2 of byte c / 2 */
            double ks = a->k_scales[srow], vs = a->v_scales[srow];
            const uint8_t *kr = a->k_nib + srow * (d / 2), *vr = a->v_nib + srow * (d / 2);
            for (int c = 0; c < d; ++c) {
                int kn = (c % 2 == 0) ? (kr[c / 2] & 15) : (kr[c / 2] >> 4);
                int vn = (c % 2 == 0) ? (vr[c / 2] & 15) : (vr[c / 2] >> 4);
                kbuf[t * d + c] = (double)(kn - 8) * ks;
                vbuf[t * d + c] = (double)(vn - 8) * vs;
            }
        } else if (a->k_codes) { /* int8 pages: exact in double (an 8-bit integer times an fp32 scale) */
            double ks = a->k_scales[srow], vs = a->v_scales[srow];
            for (int c = 0; c < d; ++c) {
                kbuf[t * d + c] = (double)a->k_codes[base + c] * ks;
                vbuf[t * d + c] = (double)a->v_codes[base + c] * vs;
            }
        } else {
            for (int c = 0; c < d; ++c) {
                kbuf[t * d + c] = oracle_bf16_to_f64(a->k_pages[base + c]);
                vbuf[t * d + c] = oracle_bf16_to_f64(a->v_pages[base + c]);
            }
        }
    }
    /* 2. scores s_t = scale * q . k_t */
    const uint16_t *qr = a->q + ((q_row_of_seq[b] + i) * a->num_q_heads + h) * (int64_t)d;
    for (int64_t t = 0; t < nkeys; ++t) {
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += oracle_bf16_to_f64(qr[c]) * kbuf[t * d + c];
        s[t] = a->scale * dot;
    }
    /* 3. softmax weights w_t = exp(s_t - max) / sum exp(s - max) */
    double mx = -INFINITY;
    for (int64_t t = 0; t < nkeys; ++t) mx = s[t] > mx ? s[t] : mx;
    double sum = 0.0;
    for (int64_t t = 0; t < nkeys; ++t) {
        s[t] = exp(s[t] - mx);
        sum += s[t];
    }
    /* 4. o = sum_t w_t v_t */
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (int64_t t = 0; t < nkeys; ++t) {
        double w = s[t] / sum;
        for (int c = 0; c < d; ++c) o[c] += w * vbuf[t * d + c];
    }
    return ORACLE_OK;
}

static int check_attn_args(const attn_args *a) {
    if (a->num_seqs < 0 || a->num_q_heads <= 0 || a->num_kv_heads <= 0 || a->head_dim <= 0 ||
        a->page_size <= 0 || a->num_q_heads % a->num_kv_heads != 0)
        return ORACLE_ERR_ARG;
    for (int b = 0; b < a->num_seqs; ++b)
        if (a->q_lens[b] < 0 || a->q_lens[b] > a->seq_lens[b]) return ORACLE_ERR_ARG;
    return ORACLE_OK;
}

static int64_t *q_row_offsets(const attn_args *a) {
    int64_t *off = (int64_t *)malloc(sizeof(int64_t) * (a->num_seqs + 1));
    if (!off) return NULL;
    off[0] = 0;
    for (int b = 0; b < a->num_seqs; ++b) off[b + 1] = off[b] + a->q_lens[b];
    return off;
}

/* Rows to compute are given as (packed query token, head) pairs; out is
 * [n_rows, head_dim]. n_threads <= 0 uses the OpenMP default. */
static int attention_rows_impl(attn_args a, const int64_t *row_token, const int32_t *row_head,
                               int64_t n_rows, double *out, int n_threads) {
    const int num_seqs = a.num_seqs, num_q_heads = a.num_q_heads, head_dim = a.head_dim;
    const int32_t *seq_lens = a.seq_lens;
    int rc = check_attn_args(&a);
    if (rc) return rc;
    int64_t *off = q_row_offsets(&a);
    if (!off) return ORACLE_ERR_NOMEM;
    int64_t max_T = 1;
    for (int b = 0; b < num_seqs; ++b) max_T = seq_lens[b] > max_T ? seq_lens[b] : max_T;
    int status = ORACLE_OK;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
#pragma omp parallel
    {
        double *kbuf = (double *)malloc(sizeof(double) * max_T * head_dim);
        double *vbuf = (double *)malloc(sizeof(double) * max_T * head_dim);
        double *s = (double *)malloc(sizeof(double) * max_T);
        int local = (kbuf && vbuf && s) ? ORACLE_OK : ORACLE_ERR_NOMEM;
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n_rows; ++r) {
            if (local) continue;
            int64_t tok = row_token[r];
            int b = 0; /* which sequence owns packed token `tok` */
            while (b < num_seqs && off[b + 1] <= tok) ++b;
            if (b >= num_seqs || row_head[r] < 0 || row_head[r] >= num_q_heads) {
                local = ORACLE_ERR_ARG;
                continue;
            }
            int e = attention_row(&a, off, b, (int)(tok - off[b]), row_head[r], kbuf, vbuf, s,
                                  out + r * head_dim);
            if (e) local = e;
        }
        if (local) {
#pragma omp critical
            status = status ? status : local;
        }
        free(kbuf);
        free(vbuf);
        free(s);
    }
    free(off);
    return status;
}

int oracle_attention_rows(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                          int page_size, int num_pages, int max_pages_per_seq,
                          const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                          const int32_t *block_table, const int32_t *seq_lens,
                          const int32_t *q_lens, double scale,
                          const int64_t *row_token, const int32_t *row_head, int64_t n_rows,
                          double *out, int n_threads) {
    attn_args a = {num_seqs, num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
                   max_pages_per_seq, q, k_pages, v_pages, block_table, seq_lens, q_lens, scale,
                   NULL, NULL, NULL, NULL, NULL, NULL};
    return attention_rows_impl(a, row_token, row_head, n_rows, out, n_threads);
}

/* Every row: out is [total_q, num_q_heads, head_dim]. */
int oracle_paged_attention(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                           int page_size, int num_pages, int max_pages_per_seq,
                           const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                           const int32_t *block_table, const int32_t *seq_lens,
                           const int32_t *q_lens, double scale, double *out, int n_threads) {
    int64_t total_q = 0;
    for (int b = 0; b < num_seqs; ++b) total_q += q_lens[b] > 0 ? q_lens[b] : 0;
    int64_t n_rows = total_q * num_q_heads;
    int64_t *tok = (int64_t *)malloc(sizeof(int64_t) * (n_rows ? n_rows : 1));
    int32_t *head = (int32_t *)malloc(sizeof(int32_t) * (n_rows ? n_rows : 1));
    if (!tok || !head) {
        free(tok);
        free(head);
        return ORACLE_ERR_NOMEM;
    }
    for (int64_t r = 0; r < n_rows; ++r) {
        tok[r] = r / num_q_heads;
        head[r] = (int32_t)(r % num_q_heads);
    }
    int rc = oracle_attention_rows(num_seqs, num_q_heads, num_kv_heads, head_dim, page_size,
                                   num_pages, max_pages_per_seq, q, k_pages, v_pages, block_table,
                                   seq_lens, q_lens, scale, tok, head, n_rows, out, n_threads);
    free(tok);
    free(head);
    return rc;
}

/* ------------------------------------------------------------- int8 pages */

/* One row of d bf16 values -> d int8 codes and one scale: scale = amax / 127
 * and code = round-to-nearest-even(x / scale), both in binary32 (the width
 * the GPU path decides the codes in); a row of zeros gets scale 0 and codes
 * 0. Inputs are finite. */
int oracle_quantize_q8(const uint16_t *x, int64_t n_rows, int d, int8_t *codes, float *scales) {
    for (int64_t r = 0; r < n_rows; ++r) {
        float amax = 0.f;
        for (int c = 0; c < d; ++c) {
            float v = (float)oracle_bf16_to_f64(x[r * d + c]);
            float av = v < 0.f ? -v : v;
            if (av > amax) amax = av;
        }
        float sc = amax / 127.0f;
        scales[r] = sc;
        for (int c = 0; c < d; ++c) {
            float v = (float)oracle_bf16_to_f64(x[r * d + c]);
            float qv = sc > 0.f ? rintf(v / sc) : 0.f;
            if (qv > 127.f) qv = 127.f;
            if (qv < -127.f) qv = -127.f;
            codes[r * d + c] = (int8_t)qv;
        }
    }
    return ORACLE_OK;
}

/* kv_append for int8 pages: each new (token, KV head) row is quantized as
 * above and written, codes and scale, where the block table puts it. */
int oracle_kv_append_q8(int num_seqs, int num_kv_heads, int head_dim, int page_size,
                        int num_pages, int max_pages_per_seq,
                        const uint16_t *k_new, const uint16_t *v_new,
                        int8_t *k_codes, int8_t *v_codes, float *k_scales, float *v_scales,
                        const int32_t *block_table, const int32_t *pos_start,
                        const int32_t *new_lens) {
    if (num_seqs < 0 || num_kv_heads <= 0 || head_dim <= 0 || page_size <= 0) return ORACLE_ERR_ARG;
    int64_t row = 0;
    for (int b = 0; b < num_seqs; ++b) {
        for (int i = 0; i < new_lens[b]; ++i, ++row) {
            int64_t pos = (int64_t)pos_start[b] + i;
            int64_t pg = page_of(block_table, max_pages_per_seq, num_pages, page_size, b, pos);
            if (pg < 0) return ORACLE_ERR_PAGE_OOB;
            for (int g = 0; g < num_kv_heads; ++g) {
                int64_t drow = (pg * num_kv_heads + g) * page_size + pos % page_size;
                int64_t src = (row * num_kv_heads + g) * head_dim;
                oracle_quantize_q8(k_new + src, 1, head_dim, k_codes + drow * head_dim, k_scales + drow);
                oracle_quantize_q8(v_new + src, 1, head_dim, v_codes + drow * head_dim, v_scales + drow);
            }
        }
    }
    return ORACLE_OK;
}

/* Attention over int8 pages: as oracle_attention_rows with every cached value
 * replaced by code * scale (exact in double). */
int oracle_attention_rows_q8(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                             int page_size, int num_pages, int max_pages_per_seq, const uint16_t *q,
                             const int8_t *k_codes, const int8_t *v_codes, const float *k_scales,
                             const float *v_scales, const int32_t *block_table,
                             const int32_t *seq_lens, const int32_t *q_lens, double scale,
                             const int64_t *row_token, const int32_t *row_head, int64_t n_rows,
                             double *out, int n_threads) {
    attn_args a = {num_seqs, num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
                   max_pages_per_seq, q, NULL, NULL, block_table, seq_lens, q_lens, scale,
                   k_codes, v_codes, k_scales, v_scales, NULL, NULL};
    return attention_rows_impl(a, row_token, row_head, n_rows, out, n_threads);
}

/* ------------------------------------------------------------- int4 pages */

/* One row of d (even) bf16 values -> d/2 bytes of nibbles and one scale:
 * scale = amax / 7, code = round-to-nearest-even(x / scale) in binary32,
 * clamped to [-7, 7], nibble = code + 8; byte c = nibble(2c) | nibble(2c+1) << 4.
 * A row of zeros gets scale 0 and every nibble 8. Inputs are finite. */
int oracle_quantize_q4(const uint16_t *x, int64_t n_rows, int d, uint8_t *packed, float *scales) {
    if (d <= 0 || d % 2 != 0) return ORACLE_ERR_ARG;
    for (int64_t r = 0; r < n_rows; ++r) {
        float amax = 0.f;
        for (int c = 0; c < d; ++c) {
            float v = (float)oracle_bf16_to_f64(x[r * d + c]);
            float av = v < 0.f ? -v : v;
            if (av > amax) amax = av;
        }
        float sc = amax / 7.0f;
        scales[r] = sc;
        for (int c = 0; c < d; c += 2) {
            int nib[2];
            for (int e = 0; e < 2; ++e) {
                float v = (float)oracle_bf16_to_f64(x[r * d + c + e]);
                float qv = sc > 0.f ? rintf(v / sc) : 0.f;
                if (qv > 7.f) qv = 7.f;
                if (qv < -7.f) qv = -7.f;
                nib[e] = (int)qv + 8;
            }
            packed[r * (d / 2) + c / 2] = (uint8_t)(nib[0] | (nib[1] << 4));
        }
    }
    return ORACLE_OK;
}

/* kv_append for int4 pages: each new (token, KV head) row is quantized as
 * above and written, nibbles and scale, where the block table puts it. */
int oracle_kv_append_q4(int num_seqs, int num_kv_heads, int head_dim, int page_size,
                        int num_pages, int max_pages_per_seq,
                        const uint16_t *k_new, const uint16_t *v_new,
                        uint8_t *k_nib, uint8_t *v_nib, float *k_scales, float *v_scales,
                        const int32_t *block_table, const int32_t *pos_start,
                        const int32_t *new_lens) {
    if (num_seqs < 0 || num_kv_heads <= 0 || head_dim <= 0 || head_dim % 2 != 0 || page_size <= 0)
        return ORACLE_ERR_ARG;
    int64_t row = 0;
    for (int b = 0; b < num_seqs; ++b) {
        for (int i = 0; i < new_lens[b]; ++i, ++row) {
            int64_t pos = (int64_t)pos_start[b] + i;
            int64_t pg = page_of(block_table, max_pages_per_seq, num_pages, page_size, b, pos);
            if (pg < 0) return ORACLE_ERR_PAGE_OOB;
            for (int g = 0; g < num_kv_heads; ++g) {
                int64_t drow = (pg * num_kv_heads + g) * page_size + pos % page_size;
                int64_t src = (row * num_kv_heads + g) * head_dim;
                oracle_quantize_q4(k_new + src, 1, head_dim, k_nib + drow * (head_dim / 2), k_scales + drow);
                oracle_quantize_q4(v_new + src, 1, head_dim, v_nib + drow * (head_dim / 2), v_scales + drow);
            }
        }
    }
    return ORACLE_OK;
}

/* Attention over int4 pages: as oracle_attention_rows with every cached value
 * replaced by (nibble - 8) * scale (exact in double). */
int oracle_attention_rows_q4(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                             int page_size, int num_pages, int max_pages_per_seq, const uint16_t *q,
                             const uint8_t *k_nib, const uint8_t *v_nib, const float *k_scales,
                             const float *v_scales, const int32_t *block_table,
                             const int32_t *seq_lens, const int32_t *q_lens, double scale,
                             const int64_t *row_token, const int32_t *row_head, int64_t n_rows,
                             double *out, int n_threads) {
    if (head_dim % 2 != 0) return ORACLE_ERR_ARG;
    attn_args a = {num_seqs, num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
                   max_pages_per_seq, q, NULL, NULL, block_table, seq_lens, q_lens, scale,
                   NULL, NULL, k_scales, v_scales, k_nib, v_nib};
    return attention_rows_impl(a, row_token, row_head, n_rows, out, n_threads);
}

/* ------------------------------------------------------- greedy verification */

/* Lowest index of the largest value; NaN never wins; all-NaN gives 0. The
 * comparison is the float comparison itself, so -0.0 == +0.0 is a tie. */
int64_t oracle_argmax(const float *row, int64_t V) {
    int64_t best = -1;
    for (int64_t v = 0; v < V; ++v) {
        if (isnan(row[v])) continue;
        if (best < 0 || row[v] > row[best]) best = v;
    }
    return best < 0 ? 0 : best;
}

/* logits [B, k_max+1, V]; candidates [B, k_max]; n_cand [B] in 0..k_max.
 * window may be NULL; when given it is updated in place. */
int oracle_verify_greedy(const float *logits, const int32_t *candidates, const int32_t *n_cand,
                         int B, int k_max, int64_t V, int32_t *accepted, int32_t *next_tok,
                         int32_t *window) {
    if (B < 0 || k_max < 0 || V <= 0) return ORACLE_ERR_ARG;
    for (int b = 0; b < B; ++b) {
        int n = n_cand[b];
        if (n < 0 || n > k_max) return ORACLE_ERR_ARG;
        const float *rows = logits + (int64_t)b * (k_max + 1) * V;
        /* step 3: compare left to right */
        int a = 0;
        while (a < n && candidates[(int64_t)b * k_max + a] == (int32_t)oracle_argmax(rows + a * V, V))
            ++a;
        accepted[b] = a;
        /* step 4: the verifier's own token where the candidates stopped */
        next_tok[b] = (int32_t)oracle_argmax(rows + (int64_t)a * V, V);
        /* step 5: +2 when everything matched, -1 otherwise (never below 1) */
        if (window) window[b] = (a == n) ? window[b] + 2 : (window[b] - 1 > 1 ? window[b] - 1 : 1);
    }
    return ORACLE_OK;
}

/* The shapes of the next verify call (see the header): window holds the
 * windows after step 5. A sequence whose q_lens < n_cand + 1 or whose
 * seq_lens < q_lens has no consistent cache: ORACLE_ERR_ARG. */
int oracle_spec_advance(int B, int k_max, const int32_t *n_cand, const int32_t *accepted,
                        const int32_t *window, int32_t *seq_lens, int32_t *q_lens, int32_t *n_cand_next) {
    if (B < 0 || k_max < 0) return ORACLE_ERR_ARG;
    for (int b = 0; b < B; ++b) {
        if (q_lens[b] < n_cand[b] + 1 || seq_lens[b] < q_lens[b] || accepted[b] < 0 || accepted[b] > n_cand[b])
            return ORACLE_ERR_ARG;
        /* kept: everything before the call, its first token, the accepted candidates */
        const int32_t kept = seq_lens[b] - q_lens[b] + 1 + accepted[b];
        /* step 1 again: as many candidates as the window says, at most k_max */
        const int32_t n = window[b] < k_max ? window[b] : k_max;
        n_cand_next[b] = n;
        q_lens[b] = n + 1;  /* the correction token, then the candidates */
        seq_lens[b] = kept + n + 1;
    }
    return ORACLE_OK;
}

/* ---------------------------------------------------------- defragmentation */

/* block_table [num_seqs][max_pages]; seq_lens [num_seqs].  Outputs:
 * new_table [num_seqs][max_pages]; moves [num_pages][2] as (from, to) pairs,
 * *n_moves of them; *n_live live pages.  The moves read only pages no move
 * writes, so they may be made in any order. */
int oracle_defrag_plan(int num_seqs, int page_size, int num_pages, int max_pages,
                       const int32_t *block_table, const int32_t *seq_lens, int32_t *new_table,
                       int32_t *moves, int32_t *n_moves, int32_t *n_live) {
    if (num_seqs < 0 || page_size <= 0 || num_pages < 0 || max_pages < 0) return ORACLE_ERR_ARG;
    char *live = calloc((size_t)num_pages + 1, 1);
    int32_t *map = malloc(((size_t)num_pages + 1) * sizeof(int32_t));
    if (!live || !map) {
        free(live);
        free(map);
        return ORACLE_ERR_NOMEM;
    }
    int rc = ORACLE_OK;
    /* 1. live pages: named by a table within its sequence's length */
    for (int b = 0; b < num_seqs && rc == ORACLE_OK; ++b) {
        if (seq_lens[b] < 0) rc = ORACLE_ERR_ARG;
        int64_t used = ((int64_t)seq_lens[b] + page_size - 1) / page_size;
        if (used > max_pages) rc = ORACLE_ERR_ARG;
        for (int64_t j = 0; j < used && rc == ORACLE_OK; ++j) {
            int32_t id = block_table[(int64_t)b * max_pages + j];
            if (id < 0 || id >= num_pages) rc = ORACLE_ERR_PAGE_OOB;
            else live[id] = 1;
        }
    }
    if (rc == ORACLE_OK) {
        int32_t L = 0;
        for (int p = 0; p < num_pages; ++p) L += live[p];
        /* 2. the k-th live page at or above L goes to the k-th free id below L */
        int32_t hole = 0, m = 0;
        for (int p = 0; p < num_pages; ++p) {
            map[p] = p;
            if (!live[p] || p < L) continue;
            while (live[hole]) ++hole; /* a free id below L exists for every page above it */
            map[p] = hole;
            moves[2 * m] = p;
            moves[2 * m + 1] = hole;
            ++m;
            ++hole;
        }
        /* 3. the tables through the map */
        for (int b = 0; b < num_seqs; ++b) {
            int64_t used = ((int64_t)seq_lens[b] + page_size - 1) / page_size;
            for (int64_t j = 0; j < max_pages; ++j) {
                int64_t i = (int64_t)b * max_pages + j;
                new_table[i] = j < used ? map[block_table[i]] : -1;
            }
        }
        *n_moves = m;
        *n_live = L;
    }
    free(live);
    free(map);
    return rc;
}

/* k_pages, v_pages [num_pages][page_elems]: copy page `from` to page `to`
 * for every move. */
int oracle_defrag_move(int num_pages, int64_t page_elems, uint16_t *k_pages, uint16_t *v_pages,
                       const int32_t *moves, int n_moves) {
    for (int m = 0; m < n_moves; ++m) {
        int32_t from = moves[2 * m], to = moves[2 * m + 1];
        if (from < 0 || from >= num_pages || to < 0 || to >= num_pages) return ORACLE_ERR_PAGE_OOB;
        memcpy(k_pages + (int64_t)to * page_elems, k_pages + (int64_t)from * page_elems,
               (size_t)page_elems * sizeof(uint16_t));
        memcpy(v_pages + (int64_t)to * page_elems, v_pages + (int64_t)from * page_elems,
               (size_t)page_elems * sizeof(uint16_t));
    }
    return ORACLE_OK;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
