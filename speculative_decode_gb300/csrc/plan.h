// plan.h -- host planner for shared page runs (deduplicated prefixes) and the
// launcher of the tensor-core shared-prefix kernel. Not part of the public ABI.
#pragma once

#include <vector>

#include "internal.h"

namespace sa {

// Rows of one shared run, per KV head: member sequences' query tokens x the
// G query heads of the KV head.
struct RunRow {
    int32_t token;      // packed query row (index into q / out)
    int32_t head_local; // 0 .. G-1; the query head is kv_head * G + head_local
    int32_t limit;      // last key position this row may see (causal)
    int32_t slot;       // workspace slot of this row's partial for chunk 0 of the run
};

struct PlanHost {
    sa_dims dims;
    int32_t num_runs = 0, num_members = 0, num_run_pages = 0;
    int32_t max_run_slots = 0;
    std::vector<int32_t> skip_pages, run_slots;
    // per run: page_lo, page_hi, row_begin, row_count, chunk_pages, first member's table row
    std::vector<int32_t> run_desc;
    std::vector<RunRow> rows;
    // per work item: run, kv head, first row of the 128-row tile, page chunk lo,
    // page chunk hi, chunk index, and the first token of the tile's rows when
    // they are consecutive tokens each with its G heads in order (the rows are
    // then one box of the queries), else -1
    std::vector<int32_t> tiles;
};

int plan_run_slots(const sa_plan *plan);
bool plan_matches(const sa_plan *plan, const sa_dims &d);
const PlanDevice *plan_device(const sa_plan *plan);

// Pure host function (no CUDA): find the shared runs of a batch. Runs that
// would give fewer than `min_rows` rows per KV head stay on the split path.
PlanHost build_plan(const sa_dims &d, const int32_t *block_table, const int32_t *seq_lens,
                    const int32_t *q_lens, int sms, int min_rows);

// Launch the tensor-core shared-prefix kernel over the plan's work items.
// tmk / tmv view the K / V pools as [num_pages*Hkv*256 rows][128] bf16 with
// 64 x prefix_key_tile() boxes and 128-byte swizzle.
cudaError_t launch_prefix_tc(const sa_dims &d, const PlanDevice &pd, const uint16_t *q,
                             const CUtensorMap &tmk, const CUtensorMap &tmv, float scale,
                             float *ws_acc, float *ws_ml, int64_t rows_total, int32_t *err,
                             const int32_t *block_table, cudaStream_t stream);
int prefix_tile_rows();  // query rows per work item (tensor-memory lanes)
int prefix_key_tile();   // keys per K/V tile

// Sequence mode of the tensor-core kernel: sequences with at least min_rows
// query rows per KV head (G heads x new tokens, e.g. q_len = k+1 verification)
// are attended entirely on the tensor cores by `grid` persistent CTAs, each
// walking one contiguous range of the sequence of (sequence, KV head, 128-row
// tile) segments' 64-key tiles (tc_work.cuh); the combine pass merges their
// partials (up to kTcMaxPieces per segment).
struct SeqTcConfig {
    int min_rows;  // 0 disables the mode
    int grid;      // CTAs (one per SM)
};
// (segments a CTA attends whole, in the waves of tc_work.cuh, are written to
// `out` directly; the combine pass skips them)
cudaError_t launch_seq_tc(const sa_dims &d, const SeqTcConfig &c, const uint16_t *q,
                          const CUtensorMap &tmk, const CUtensorMap &tmv, float scale,
                          float *ws_acc, float *ws_ml, int64_t rows_total, int32_t *err,
                          const int32_t *block_table, const int32_t *seq_lens,
                          const int32_t *q_lens, uint16_t *out, cudaStream_t stream);

constexpr int kRunDescInts = 6;
constexpr int kTileInts = 7;
constexpr int kPrefixTileRows = 128;

}  // namespace sa
