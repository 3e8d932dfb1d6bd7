// internal.h -- declarations shared by the library's translation units
// (host side). Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "specattn.h"

namespace sa {

constexpr int kHeadDim = 128;
constexpr int kPageSize = 256;
constexpr int kMaxQLen = 512;     // new tokens per sequence in one call (decode 1, verify k+1, prefill chunks)
constexpr int kPlanMaxQLen = 16;  // with a shared-prefix plan
constexpr int kMaxKMax = 15;

constexpr int32_t kErrBitPageOOB = 1 << SA_ERR_PAGE_OOB;
constexpr int32_t kErrBitTimeout = 1 << SA_ERR_TIMEOUT;
constexpr int32_t kErrBitQlen = 1 << SA_ERR_QLEN;

// Device-side description of a plan's shared-prefix work (all arrays live in
// the plan's device buffer).
struct PlanDevice {
    int32_t num_runs;        // shared runs
    int32_t num_tiles;       // tensor-core work items (run, kv head, row tile, page chunk)
    int32_t max_run_slots;   // workspace partial slots used by runs per row
    const int32_t *skip_pages;  // [B] leading logical pages covered by runs
    const int32_t *run_slots;   // [B] number of run partials of each sequence
    const int32_t *run_desc;    // per run: page_lo, page_hi, row_begin, row_count, first member
    const int32_t *run_rows;    // per run row: packed query token, q head (within kv head), key limit, slot
    const int32_t *tiles;       // per work item: run, row tile, page chunk lo, page chunk hi, slot
};

// Parameters of the split-K kernel (page-streamed attention on CUDA cores).
struct SplitParams {
    const uint16_t *q;
    const uint16_t *k_pages;    // [num_pages, Hkv, 256, 128]
    const uint16_t *v_pages;
    uint16_t *out;
    const int32_t *block_table;
    const int32_t *seq_lens;
    const int32_t *q_lens;
    const int32_t *skip_pages;  // nullable: pages [0, skip) handled by the shared-prefix path
    const int32_t *run_slots;   // nullable: partials the shared-prefix path writes per sequence
    float *ws_acc;              // [n_slots][total_q * Hq][128] fp32 unnormalised accumulators
    float *ws_ml;               // [n_slots][total_q * Hq][2] running max (log2 units), sum
    int32_t *err;
    int32_t B, Hq, Hkv, G, num_pages, max_pages, total_q, max_q_len;
    int32_t rows_per_block;     // R, rows of one segment (4, 8 or 16)
    int32_t n_row_blocks;       // row blocks per (sequence, KV head) at max_q_len
    int32_t piece_slots;        // partial slots a segment's pieces may use
    int32_t tc_min_rows;        // > 0: sequences with >= this many rows per KV head were
    int32_t tc_grid;            //   attended on the tensor cores by this many persistent CTAs
                                //   (tc_work.cuh); the combine pass merges their partials
    int32_t slot_base;          // first workspace slot used by pieces
    int32_t n_rows_total;       // total_q * Hq (row stride of a workspace slot)
    float qscale;               // scale * log2(e)
    int32_t evict_first;
    int32_t split_ctas;         // grid of the split kernel (one warp each); the combine
                                // pass recomputes the same cut of the work
    // quantised pages (NULL for bf16 pages): codes [num_pages, Hkv, 256, 128 *
    // code_bits / 8] (int8 codes, or int4 as nibble = code + 8 with value 2c in
    // the low nibble of byte c), one scale per (page, head, token) row
    // [num_pages, Hkv, 256]; value = code * scale
    const uint8_t *k_codes, *v_codes;
    const float *k_scales, *v_scales;
    int32_t code_bits;          // 8 or 4 when k_codes is set
    int32_t pages_ready;        // 1: a kernel of this call that started after the pages were
                                // written ran first, so pages are read without waiting for it
};

// Parameters of the persistent page-streaming kernel (attn_stream.cu): bf16,
// int8 or int4 pages, no plan, fewer than 16 query rows per KV head.
constexpr int kStreamMaxCtas = 256;   // grid cap (one CTA per SM); workspace is sized for it
// partial slots: two per CTA (the pieces it shares with its neighbours)
constexpr int kStreamSlots = 2 * kStreamMaxCtas;
struct StreamParams {
    const uint16_t *q;
    const uint16_t *k_pages;    // [num_pages, Hkv, 256, 128]
    const uint16_t *v_pages;
    uint16_t *out;
    const int32_t *block_table;
    const int32_t *seq_lens;
    const int32_t *q_lens;
    float *part_acc;            // [kStreamSlots][R][128] fp32 partials of cut segments
    float *part_ml;             // [kStreamSlots][R][2] (max in log2 units, sum)
    int32_t *counters;          // [kStreamMaxCtas] pieces finished per cut segment, zero
                                // between calls
    int32_t *err;
    int32_t B, Hq, Hkv, G, num_pages, max_pages, total_q, max_q_len;
    int32_t R;                  // rows per segment (4, 8 or 16)
    float qscale;               // scale * log2(e)
    int32_t n_ctas;             // grid: one CTA per SM, at most kStreamMaxCtas
    int32_t evict_first;
    // quantised pages (code_bits 8 or 4; 16: bf16 pages): the tensor maps view
    // the code pools, and one fp32 scale per (page, head, token) row
    // [num_pages, Hkv, 256]; value = code * scale
    int32_t code_bits;
    const float *k_scales, *v_scales;
};
// Tensor maps of the K and V pools, each viewed as [num_pages * Hkv * 256
// rows] of 128 bf16 values (box kind i: 64 columns x (16 << i) rows, 128-byte
// swizzle), of 128 int8 codes (128 bytes x (16 << i) rows, 128-byte swizzle)
// or of 64 bytes of int4 codes (64 bytes x (16 << i) rows, 64-byte swizzle).
constexpr int kStreamBoxKinds = 5;
struct StreamMaps {
    CUtensorMap k[kStreamBoxKinds];
    CUtensorMap v[kStreamBoxKinds];
};
cudaError_t launch_stream_attn(const StreamParams &p, const StreamMaps &maps, cudaStream_t stream);
int stream_units_per_tile();
int stream_segment_cost();
int stream_tile_tokens();  // tokens per cut tile (the work is counted in these)
int stream_box_rows();     // rows of the smallest TMA box

// Split kernel over p.split_ctas one-warp CTAs, then the combine pass that
// merges the partials of segments cut into pieces (two kernels).
cudaError_t launch_split_attn(const SplitParams &p, cudaStream_t stream);
cudaError_t split_occupancy(int R, int code_bits, int *ctas_per_sm);  // code_bits 16: bf16 pages
int split_tile_tokens();  // tokens per K/V tile of the split kernel
int split_units_per_tile();  // balancing units of one tile and of a segment start
int split_segment_cost();

// Cache compaction (defrag.cu): the host planner and the page-copy kernel.
int defrag_plan_host(int num_seqs, int num_pages, int max_pages, const int32_t *block_table,
                     const int32_t *seq_lens, int32_t *new_table, int32_t *moves, int32_t *n_moves,
                     int32_t *n_live);
cudaError_t launch_defrag(void *k_pages, void *v_pages, const int32_t *moves, int n_moves,
                          int num_pages, int64_t page_bytes, int32_t *err, int sms, cudaStream_t stream);

// kv_append for quantised pages: code_bits 8 (int8) or 4 (int4 nibbles)
cudaError_t launch_kv_append_quant(const sa_dims &d, int code_bits, const uint16_t *k_new,
                                   const uint16_t *v_new, uint8_t *k_codes, uint8_t *v_codes,
                                   float *k_scales, float *v_scales, const int32_t *block_table,
                                   const int32_t *seq_lens, const int32_t *q_lens, int32_t *err,
                                   cudaStream_t stream);
cudaError_t launch_kv_append(const sa_dims &d, const uint16_t *k_new, const uint16_t *v_new,
                             uint16_t *k_pages, uint16_t *v_pages, const int32_t *block_table,
                             const int32_t *seq_lens, const int32_t *q_lens, int32_t *err,
                             cudaStream_t stream);

struct VerifyParams {
    const float *logits;
    const int32_t *candidates;
    const int32_t *n_cand;
    int32_t *accepted;
    int32_t *next_tok;
    int32_t *window;
    int32_t *seq_lens;    // nullable: in/out, the next call's lengths (with q_lens, n_cand_next)
    int32_t *q_lens;
    int32_t *n_cand_next;
    float *part_val;      // [B * (k_max + 1)][n_chunks]
    int32_t *part_idx;    // same shape
    int32_t *counters;    // [B], zero between calls
    int32_t *err;
    int32_t B, k_max, V, n_chunks, chunk;
};
cudaError_t launch_verify(const VerifyParams &p, cudaStream_t stream);

// Driver entry point for tensor-map encoding (resolved once, no -lcuda).
CUresult encode_tensor_map_2d(CUtensorMap *map, CUtensorMapDataType dtype, void *base,
                              uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                              uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);
// A 3-D tiled map: dims innermost first, byte strides of dims 1 and 2, box
// extents, no interleave, zero fill outside the tensor.
CUresult encode_tensor_map_3d(CUtensorMap *map, CUtensorMapDataType dtype, void *base, const uint64_t dims[3],
                              const uint64_t strides_bytes[2], const uint32_t box[3], CUtensorMapSwizzle swizzle);

int device_sm_count();

}  // namespace sa
