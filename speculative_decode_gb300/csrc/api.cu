// api.cu -- the C ABI (include/specattn.h): argument checks, work
// decomposition, tensor maps and kernel launches. Host code only.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "plan.h"
#include "tc_work.cuh"

namespace sa {

namespace {

bool debug_sync() {
    static const bool on = [] {
        const char *v = std::getenv("SA_DEBUG");
        return v != nullptr && std::strcmp(v, "1") == 0;
    }();
    return on;
}

// Under SA_DEBUG=1: wait for the stream and turn the device flag into a status.
int finish(cudaStream_t stream, const int32_t *err_flag) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return SA_ERR_CUDA;
    if (!debug_sync()) return SA_OK;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return SA_ERR_CUDA;
    if (err_flag == nullptr) return SA_OK;
    int32_t flag = 0;
    if (cudaMemcpy(&flag, err_flag, sizeof flag, cudaMemcpyDeviceToHost) != cudaSuccess)
        return SA_ERR_CUDA;
    for (int s = 1; s < 31; ++s)
        if (flag & (1 << s)) return s;
    return SA_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_dims(const sa_dims *d) {
    if (d == nullptr) return SA_ERR_ARG;
    if (d->num_seqs < 0 || d->num_q_heads <= 0 || d->num_kv_heads <= 0 || d->num_pages < 0 ||
        d->max_pages_per_seq < 0 || d->total_q < 0 || d->max_q_len < 0)
        return SA_ERR_ARG;
    if (d->num_q_heads % d->num_kv_heads != 0) return SA_ERR_ARG;
    if (d->head_dim != kHeadDim || d->page_size != kPageSize) return SA_ERR_UNSUPPORTED;
    if (d->max_q_len > kMaxQLen) return SA_ERR_UNSUPPORTED;
    // the pool is addressed as num_pages * Hkv * 256 rows with 32-bit coordinates
    if (static_cast<int64_t>(d->num_pages) * d->num_kv_heads * kPageSize >= (int64_t{1} << 31))
        return SA_ERR_UNSUPPORTED;
    if (d->num_q_heads / d->num_kv_heads * d->max_q_len > 16 * kMaxQLen) return SA_ERR_UNSUPPORTED;
    return SA_OK;
}

// Work decomposition of the split kernel: rows per segment and the partial
// slots pieces may use (a pure function of the shapes).
struct SplitConfig {
    int R, nrb, piece_slots, run_slots, n_slots;
    SeqTcConfig tc;
};

constexpr int kPieceSlots = 8;
// A batch whose largest sequence has at least this many query rows per KV
// head (G heads x new tokens: q_len = k+1 verification, prefill chunks) is a
// dense contraction: without a plan all of its sequences go to the tensor
// cores (persistent CTAs over an even cut of their tiles), the ones with few
// rows too, so that a mixed batch is one even cut of all its keys. Smaller
// batches go to the persistent page-streaming kernel.
constexpr int kTcMinRows = 16;

// Quantised pages are attended on the CUDA cores only: sequences with many
// query rows per KV head take several 16-row blocks, each streaming the pages
// again, up to this many rows (verification blocks; not prefill chunks).
constexpr int kQuantMaxRows = 128;

SplitConfig split_config(const sa_dims &d, const sa_plan *plan, bool quant = false) {
    SplitConfig c{};
    const int G = d.num_q_heads / d.num_kv_heads;
    const int rows = G * std::max(1, d.max_q_len);
    c.R = rows <= 4 ? 4 : rows <= 8 ? 8 : 16;
    c.nrb = (rows + c.R - 1) / c.R;
    const int max_tiles = std::max(1, d.max_pages_per_seq) * (kPageSize / split_tile_tokens());
    c.piece_slots = std::min(kPieceSlots, max_tiles);
    c.tc = SeqTcConfig{0, 0};  // grid is set at launch (one CTA per SM)
    if (!quant && plan == nullptr && G * std::max(1, d.max_q_len) >= kTcMinRows) c.tc.min_rows = 1;
    c.run_slots = plan ? plan_run_slots(plan) : (c.tc.min_rows > 0 ? kTcMaxPieces : 0);
    c.n_slots = c.run_slots + c.piece_slots;
    return c;
}

// Partials one output row may have to merge (the combine pass merges at most
// kMaxMergeSlotsHost of them).
constexpr int kMaxMergeSlotsHost = 16;
bool merge_fits(const SplitConfig &c) { return c.n_slots <= kMaxMergeSlotsHost;
}

// Workspace layout. The first kCounterBytes hold the persistent kernel's
// counters (one per cut segment; zero between calls: every call leaves them at
// zero, so the workspace must be zero-filled once before its first use); no
// other kernel touches them, so one workspace serves calls of any shape. Then
// the partials: for the persistent kernel, fp32 accumulators [slots][R][128]
// and (max, sum) pairs [slots][R][2] (two slots per CTA); for the split kernel,
// accumulators [n_slots][total_q * Hq][128] and pairs [n_slots][total_q * Hq]
// [2]. Every partial a call reads was written earlier in the same call. The
// sizes are for the finest split any device could choose, so sizing needs no
// device.
constexpr size_t kCounterBytes = 4096;
static_assert(kStreamMaxCtas * 4 <= static_cast<int>(kCounterBytes), "counters fit their region");

struct WsLayout {
    size_t acc_offset, ml_offset, total;
};

// Calls with no plan and fewer than kTcMinRows query rows per KV head (over
// bf16, int8 or int4 pages) go to the persistent page-streaming kernel.
bool use_stream(const sa_dims &d, const sa_plan *plan, bool quant) {
    (void)quant;
    return plan == nullptr && d.num_q_heads / d.num_kv_heads * std::max(1, d.max_q_len) < kTcMinRows;
}

size_t align256(size_t n) { return (n + 255) / 256 * 256; }

WsLayout attn_ws_layout(const sa_dims &d, const sa_plan *plan, bool quant) {
    WsLayout w{};
    const SplitConfig c = split_config(d, plan, quant);
    w.acc_offset = kCounterBytes;
    if (use_stream(d, plan, quant)) {
        const size_t rows = static_cast<size_t>(kStreamSlots) * c.R;
        w.ml_offset = w.acc_offset + align256(rows * kHeadDim * 4);
        w.total = w.ml_offset + align256(rows * 2 * 4);
        return w;
    }
    const int64_t rows = static_cast<int64_t>(d.total_q) * d.num_q_heads;
    const size_t acc = static_cast<size_t>(c.n_slots * rows * kHeadDim * 4);
    const size_t ml = static_cast<size_t>(c.n_slots * rows * 2 * 4);
    w.ml_offset = w.acc_offset + align256(acc);
    w.total = w.ml_offset + align256(ml);
    return w;
}

// The size sa_paged_attn_workspace_size reports: without a plan it covers
// both bf16 and quantised pages (the quantised calls take the same size).
size_t attn_ws_bytes(const sa_dims &d, const sa_plan *plan) {
    size_t n = attn_ws_layout(d, plan, false).total;
    if (plan == nullptr) n = std::max(n, attn_ws_layout(d, plan, true).total);
    return n;
}

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                              const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                              const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
    static EncodeFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeFn>(p);
    }();
    return fn;
}

}  // namespace

CUresult encode_tensor_map_2d(CUtensorMap *map, CUtensorMapDataType dtype, void *base,
                              uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                              uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
    EncodeFn fn = encode_fn();
    if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dtype, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode_tensor_map_3d(CUtensorMap *map, CUtensorMapDataType dtype, void *base, const uint64_t dims[3],
                              const uint64_t strides_bytes[2], const uint32_t box[3], CUtensorMapSwizzle swizzle) {
    EncodeFn fn = encode_fn();
    if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
    const cuuint64_t gd[3] = {dims[0], dims[1], dims[2]};
    const cuuint64_t gs[2] = {strides_bytes[0], strides_bytes[1]};
    const cuuint32_t bx[3] = {box[0], box[1], box[2]};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, dtype, 3, base, gd, gs, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// Tensor maps of the persistent kernel for one pair of pools: bf16 pages
// (bits 16: rows of 128 values, boxes of 64 columns with 128-byte swizzle),
// int8 codes (bits 8: rows of 128 bytes, 128-byte swizzle) or int4 codes
// (bits 4: rows of 64 bytes, 64-byte swizzle). A decode loop calls with the
// same pools every step, so the last pair's maps are kept (per host thread;
// a map holds only the pool's address and shape).
const StreamMaps *stream_maps(const void *k_pool, const void *v_pool, uint64_t rows, int bits) {
    struct Entry {
        const void *k = nullptr, *v = nullptr;
        uint64_t rows = 0;
        int bits = 0;
        StreamMaps maps;
    };
    thread_local Entry e;
    if (e.k == k_pool && e.v == v_pool && e.rows == rows && e.bits == bits) return &e.maps;
    e.k = nullptr;
    for (int i = 0; i < kStreamBoxKinds; ++i) {
        const uint32_t box_rows = static_cast<uint32_t>(stream_box_rows()) << i;
        CUresult rk, rv;
        if (bits == 16) {
            rk = encode_tensor_map_2d(&e.maps.k[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void *>(k_pool),
                                      kHeadDim, rows, kHeadDim * 2, 64, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
            rv = encode_tensor_map_2d(&e.maps.v[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void *>(v_pool),
                                      kHeadDim, rows, kHeadDim * 2, 64, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
        } else {
            const uint32_t row_bytes = kHeadDim * bits / 8;
            const CUtensorMapSwizzle sw = bits == 8 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
            rk = encode_tensor_map_2d(&e.maps.k[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<void *>(k_pool),
                                      row_bytes, rows, row_bytes, row_bytes, box_rows, sw);
            rv = encode_tensor_map_2d(&e.maps.v[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<void *>(v_pool),
                                      row_bytes, rows, row_bytes, row_bytes, box_rows, sw);
        }
        if (rk != CUDA_SUCCESS || rv != CUDA_SUCCESS) return nullptr;
    }
    e.k = k_pool;
    e.v = v_pool;
    e.rows = rows;
    e.bits = bits;
    return &e.maps;
}

int device_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

}  // namespace sa

using namespace sa;

namespace sa {

// One CTA waits on an mbarrier that nothing completes, with the bounded wait
// every kernel of the library uses; when it gives up the CTA flags the
// timeout and returns.
__global__ void bounded_wait_selftest_kernel(int32_t *err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    const bool done = __all_sync(0xffffffffu, mbar_wait(&bar, 0));
    if (!done && threadIdx.x == 0) flag_error(err, kErrBitTimeout);
}

}  // namespace sa

extern "C" {

const char *sa_status_string(int status) {
    switch (status) {
        case SA_OK: return "ok";
        case SA_ERR_ARG: return "invalid argument";
        case SA_ERR_UNSUPPORTED: return "unsupported shape";
        case SA_ERR_PAGE_OOB: return "block-table entry out of range";
        case SA_ERR_CUDA: return "CUDA error";
        case SA_ERR_TIMEOUT: return "bounded wait timed out inside a kernel";
        case SA_ERR_WORKSPACE: return "workspace missing or too small";
        case SA_ERR_QLEN: return "query length or candidate count out of range";
        default: return "unknown status";
    }
}

int sa_device_sm_count(void) { return device_sm_count(); }

int sa_selftest_bounded_wait(int32_t *err_flag, void *stream) {
    if (err_flag == nullptr) return SA_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    sa::bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(err_flag);
    if (cudaGetLastError() != cudaSuccess) return SA_ERR_CUDA;
    return finish(s, err_flag);
}

int sa_kv_append(const sa_dims *dims, const uint16_t *k_new, const uint16_t *v_new,
                 uint16_t *k_pages, uint16_t *v_pages, const int32_t *block_table,
                 const int32_t *seq_lens, const int32_t *q_lens, int32_t *err_flag, void *stream) {
    int rc = check_dims(dims);
    if (rc) return rc;
    if (dims->num_seqs == 0 || dims->total_q == 0) return SA_OK;
    if (!k_new || !v_new || !k_pages || !v_pages || !block_table || !seq_lens || !q_lens)
        return SA_ERR_ARG;
    if (!aligned(k_new, 8) || !aligned(v_new, 8) || !aligned(k_pages, 8) || !aligned(v_pages, 8))
        return SA_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (launch_kv_append(*dims, k_new, v_new, k_pages, v_pages, block_table, seq_lens, q_lens,
                         err_flag, s) != cudaSuccess)
        return SA_ERR_CUDA;
    return finish(s, err_flag);
}

size_t sa_paged_attn_workspace_size(const sa_dims *dims, const sa_plan *plan) {
    if (check_dims(dims) != SA_OK) return 0;
    return attn_ws_bytes(*dims, plan);
}

// quantised pools of sa_paged_attn_q8 / _q4 (all NULL for bf16 pages)
struct QuantPools {
    const uint8_t *k_codes, *v_codes;
    const float *k_scales, *v_scales;
    int bits;  // 8 or 4
};

static int paged_attn_impl(const sa_dims *dims, const uint16_t *q, const uint16_t *k_pages,
                           const uint16_t *v_pages, const QuantPools &qp, const int32_t *block_table,
                           const int32_t *seq_lens, const int32_t *q_lens, float scale, uint16_t *out,
                           const sa_plan *plan, void *workspace, size_t workspace_bytes,
                           int32_t *err_flag, void *stream) {
    int rc = check_dims(dims);
    if (rc) return rc;
    const sa_dims &d = *dims;
    if (d.num_seqs == 0 || d.total_q == 0) return SA_OK;
    const bool quant = qp.k_codes != nullptr;
    if (!q || !block_table || !seq_lens || !q_lens || !out) return SA_ERR_ARG;
    if (quant ? (!qp.v_codes || !qp.k_scales || !qp.v_scales) : (!k_pages || !v_pages)) return SA_ERR_ARG;
    if (d.num_pages == 0 || d.max_pages_per_seq == 0) return SA_ERR_ARG;
    if (!aligned(q, 16) || !aligned(out, 16)) return SA_ERR_ARG;
    if (quant ? (!aligned(qp.k_codes, 16) || !aligned(qp.v_codes, 16) || !aligned(qp.k_scales, 16) ||
                 !aligned(qp.v_scales, 16))
              : (!aligned(k_pages, 16) || !aligned(v_pages, 16)))
        return SA_ERR_ARG;
    // quantised pages are attended on the CUDA cores only: no plan, at most
    // kQuantMaxRows query rows per KV head
    if (quant && (plan != nullptr || d.num_q_heads / d.num_kv_heads * std::max(1, d.max_q_len) > kQuantMaxRows))
        return SA_ERR_UNSUPPORTED;
    if (plan && !plan_matches(plan, d)) return SA_ERR_ARG;
    const WsLayout wl = attn_ws_layout(d, plan, quant);
    if (workspace == nullptr || workspace_bytes < wl.total || !aligned(workspace, 256))
        return SA_ERR_WORKSPACE;
    const int sms = device_sm_count();
    if (sms <= 0) return SA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);

    const SplitConfig c = split_config(d, plan, quant);
    if (use_stream(d, plan, quant)) {
        // the work is counted in 32-bit balancing units
        const int64_t max_units = static_cast<int64_t>(d.num_seqs) * d.num_kv_heads * c.nrb *
                                  (static_cast<int64_t>(d.max_pages_per_seq) * (kPageSize / stream_tile_tokens()) *
                                       stream_units_per_tile() + stream_segment_cost());
        if (max_units > INT32_MAX / 2) return SA_ERR_UNSUPPORTED;
        StreamParams p{};
        p.q = q;
        p.k_pages = k_pages;
        p.v_pages = v_pages;
        p.out = out;
        p.block_table = block_table;
        p.seq_lens = seq_lens;
        p.q_lens = q_lens;
        p.part_acc = reinterpret_cast<float *>(ws + wl.acc_offset);
        p.part_ml = reinterpret_cast<float *>(ws + wl.ml_offset);
        p.counters = reinterpret_cast<int32_t *>(ws);
        p.err = err_flag;
        p.B = d.num_seqs;
        p.Hq = d.num_q_heads;
        p.Hkv = d.num_kv_heads;
        p.G = d.num_q_heads / d.num_kv_heads;
        p.num_pages = d.num_pages;
        p.max_pages = d.max_pages_per_seq;
        p.total_q = d.total_q;
        p.max_q_len = d.max_q_len;
        p.R = c.R;
        p.qscale = scale * 1.4426950408889634f;
        p.n_ctas = std::min(sms, kStreamMaxCtas);
        p.evict_first = c.nrb == 1;
        p.code_bits = quant ? qp.bits : 16;
        p.k_scales = qp.k_scales;
        p.v_scales = qp.v_scales;
        const uint64_t rows = static_cast<uint64_t>(d.num_pages) * d.num_kv_heads * kPageSize;
        const StreamMaps *maps = quant ? stream_maps(qp.k_codes, qp.v_codes, rows, qp.bits)
                                       : stream_maps(k_pages, v_pages, rows, 16);
        if (maps == nullptr) return SA_ERR_CUDA;
        if (launch_stream_attn(p, *maps, s) != cudaSuccess) return SA_ERR_CUDA;
        return finish(s, err_flag);
    }
    if (!merge_fits(c)) return SA_ERR_UNSUPPORTED;  // too many partials per row to merge
    // the split kernel counts work in 32-bit balancing units
    const int64_t max_work = static_cast<int64_t>(d.num_seqs) * d.num_kv_heads * c.nrb *
                             (static_cast<int64_t>(d.max_pages_per_seq) * (kPageSize / split_tile_tokens()) *
                                  split_units_per_tile() + split_segment_cost());
    if (max_work > INT32_MAX) return SA_ERR_UNSUPPORTED;
    const int64_t rows_total = static_cast<int64_t>(d.total_q) * d.num_q_heads;
    float *ws_acc = reinterpret_cast<float *>(ws + wl.acc_offset);
    float *ws_ml = reinterpret_cast<float *>(ws + wl.ml_offset);

    const uint64_t pool_rows = static_cast<uint64_t>(d.num_pages) * d.num_kv_heads * kPageSize;
    const PlanDevice *pd = plan ? plan_device(plan) : nullptr;
    if ((pd && pd->num_tiles > 0) || c.tc.min_rows > 0) {
        // tensor-core work first: the combine pass reads its partials
        CUtensorMap pk, pv;
        if (encode_tensor_map_2d(&pk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<uint16_t *>(k_pages),
                                 kHeadDim, pool_rows, kHeadDim * 2, 64, prefix_key_tile(),
                                 CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
            encode_tensor_map_2d(&pv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<uint16_t *>(v_pages),
                                 kHeadDim, pool_rows, kHeadDim * 2, 64, prefix_key_tile(),
                                 CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
            return SA_ERR_CUDA;
        if (pd && pd->num_tiles > 0 &&
            launch_prefix_tc(d, *pd, q, pk, pv, scale, ws_acc, ws_ml, rows_total, err_flag,
                             block_table, s) != cudaSuccess)
            return SA_ERR_CUDA;
        if (c.tc.min_rows > 0 &&
            launch_seq_tc(d, SeqTcConfig{c.tc.min_rows, sms}, q, pk, pv, scale, ws_acc, ws_ml, rows_total, err_flag,
                          block_table, seq_lens, q_lens, out, s) != cudaSuccess)
            return SA_ERR_CUDA;
    }

    SplitParams p{};
    p.q = q;
    p.k_pages = k_pages;
    p.k_codes = qp.k_codes;
    p.v_codes = qp.v_codes;
    p.k_scales = qp.k_scales;
    p.v_scales = qp.v_scales;
    p.code_bits = qp.bits;
    p.v_pages = v_pages;
    p.out = out;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.q_lens = q_lens;
    p.skip_pages = pd ? pd->skip_pages : nullptr;
    p.run_slots = pd ? pd->run_slots : nullptr;
    p.ws_acc = ws_acc;
    p.ws_ml = ws_ml;
    p.err = err_flag;
    p.B = d.num_seqs;
    p.Hq = d.num_q_heads;
    p.Hkv = d.num_kv_heads;
    p.G = d.num_q_heads / d.num_kv_heads;
    p.num_pages = d.num_pages;
    p.max_pages = d.max_pages_per_seq;
    p.total_q = d.total_q;
    p.max_q_len = d.max_q_len;
    p.rows_per_block = c.R;
    p.n_row_blocks = c.nrb;
    p.piece_slots = c.piece_slots;
    p.tc_min_rows = c.tc.min_rows;
    p.tc_grid = sms;
    p.slot_base = c.run_slots;
    p.n_rows_total = static_cast<int32_t>(rows_total);
    p.qscale = scale * 1.4426950408889634f;
    p.evict_first = c.nrb == 1;

    int per_sm = 0;
    if (split_occupancy(c.R, quant ? qp.bits : 16, &per_sm) != cudaSuccess || per_sm <= 0) return SA_ERR_CUDA;
    // one warp per CTA, all resident; after a plan's tensor-core kernel two
    // fewer per SM, so that combine CTAs fit beside them and scan early
    p.split_ctas = sms * ((pd && pd->num_tiles > 0 && per_sm > 2) ? per_sm - 2 : per_sm);
    p.pages_ready = ((pd && pd->num_tiles > 0) || c.tc.min_rows > 0) ? 1 : 0;
    if (launch_split_attn(p, s) != cudaSuccess)
        return SA_ERR_CUDA;
    return finish(s, err_flag);
}

int sa_paged_attn(const sa_dims *dims, const uint16_t *q, const uint16_t *k_pages,
                  const uint16_t *v_pages, const int32_t *block_table, const int32_t *seq_lens,
                  const int32_t *q_lens, float scale, uint16_t *out, const sa_plan *plan,
                  void *workspace, size_t workspace_bytes, int32_t *err_flag, void *stream) {
    return paged_attn_impl(dims, q, k_pages, v_pages, QuantPools{nullptr, nullptr, nullptr, nullptr, 16},
                           block_table, seq_lens, q_lens, scale, out, plan, workspace, workspace_bytes,
                           err_flag, stream);
}

int sa_paged_attn_q8(const sa_dims *dims, const uint16_t *q, const int8_t *k_codes,
                     const int8_t *v_codes, const float *k_scales, const float *v_scales,
                     const int32_t *block_table, const int32_t *seq_lens, const int32_t *q_lens,
                     float scale, uint16_t *out, void *workspace, size_t workspace_bytes,
                     int32_t *err_flag, void *stream) {
    if (k_codes == nullptr) return SA_ERR_ARG;
    return paged_attn_impl(dims, q, nullptr, nullptr,
                           QuantPools{reinterpret_cast<const uint8_t *>(k_codes),
                                      reinterpret_cast<const uint8_t *>(v_codes), k_scales, v_scales, 8},
                           block_table, seq_lens, q_lens, scale, out, nullptr, workspace,
                           workspace_bytes, err_flag, stream);
}

int sa_paged_attn_q4(const sa_dims *dims, const uint16_t *q, const uint8_t *k_codes,
                     const uint8_t *v_codes, const float *k_scales, const float *v_scales,
                     const int32_t *block_table, const int32_t *seq_lens, const int32_t *q_lens,
                     float scale, uint16_t *out, void *workspace, size_t workspace_bytes,
                     int32_t *err_flag, void *stream) {
    if (k_codes == nullptr) return SA_ERR_ARG;
    return paged_attn_impl(dims, q, nullptr, nullptr, QuantPools{k_codes, v_codes, k_scales, v_scales, 4},
                           block_table, seq_lens, q_lens, scale, out, nullptr, workspace,
                           workspace_bytes, err_flag, stream);
}

static int kv_append_quant(const sa_dims *dims, int bits, const uint16_t *k_new, const uint16_t *v_new,
                           uint8_t *k_codes, uint8_t *v_codes, float *k_scales, float *v_scales,
                           const int32_t *block_table, const int32_t *seq_lens, const int32_t *q_lens,
                           int32_t *err_flag, void *stream) {
    int rc = check_dims(dims);
    if (rc) return rc;
    if (dims->num_seqs == 0 || dims->total_q == 0) return SA_OK;
    if (!k_new || !v_new || !k_codes || !v_codes || !k_scales || !v_scales || !block_table ||
        !seq_lens || !q_lens)
        return SA_ERR_ARG;
    if (!aligned(k_new, 8) || !aligned(v_new, 8) || !aligned(k_codes, 4) || !aligned(v_codes, 4) ||
        !aligned(k_scales, 4) || !aligned(v_scales, 4))
        return SA_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (launch_kv_append_quant(*dims, bits, k_new, v_new, k_codes, v_codes, k_scales, v_scales, block_table,
                               seq_lens, q_lens, err_flag, s) != cudaSuccess)
        return SA_ERR_CUDA;
    return finish(s, err_flag);
}

int sa_kv_append_q8(const sa_dims *dims, const uint16_t *k_new, const uint16_t *v_new,
                    int8_t *k_codes, int8_t *v_codes, float *k_scales, float *v_scales,
                    const int32_t *block_table, const int32_t *seq_lens, const int32_t *q_lens,
                    int32_t *err_flag, void *stream) {
    return kv_append_quant(dims, 8, k_new, v_new, reinterpret_cast<uint8_t *>(k_codes),
                           reinterpret_cast<uint8_t *>(v_codes), k_scales, v_scales, block_table, seq_lens,
                           q_lens, err_flag, stream);
}

int sa_kv_append_q4(const sa_dims *dims, const uint16_t *k_new, const uint16_t *v_new,
                    uint8_t *k_codes, uint8_t *v_codes, float *k_scales, float *v_scales,
                    const int32_t *block_table, const int32_t *seq_lens, const int32_t *q_lens,
                    int32_t *err_flag, void *stream) {
    return kv_append_quant(dims, 4, k_new, v_new, k_codes, v_codes, k_scales, v_scales, block_table,
                           seq_lens, q_lens, err_flag, stream);
}

int sa_paged_attn_kernel_count(const sa_dims *dims, const sa_plan *plan) {
    if (check_dims(dims) != SA_OK) return -1;
    const int sms = device_sm_count();
    if (sms <= 0) return -1;
    const PlanDevice *pd = plan ? plan_device(plan) : nullptr;
    if (use_stream(*dims, plan, false)) return 1;
    const SplitConfig c = split_config(*dims, plan);
    return 2 + ((pd && pd->num_tiles > 0) ? 1 : 0) + (c.tc.min_rows > 0 ? 1 : 0);
}

size_t sa_spec_verify_workspace_size(int32_t num_seqs, int32_t k_max, int32_t vocab) {
    if (num_seqs < 0 || k_max < 0 || k_max > kMaxKMax || vocab <= 0) return 0;
    const int64_t chunks = (static_cast<int64_t>(vocab) + 1023) / 1024;
    const int64_t parts = static_cast<int64_t>(num_seqs) * (k_max + 1) * chunks;
    const size_t a = ((static_cast<size_t>(parts) * 4 + 255) / 256) * 256;
    const size_t c = ((static_cast<size_t>(num_seqs) * 4 + 255) / 256) * 256;
    return 2 * a + c;
}

static int verify_impl(const float *logits, const int32_t *candidates, const int32_t *n_cand,
                       int32_t num_seqs, int32_t k_max, int32_t vocab, int32_t *accepted,
                       int32_t *next_tok, int32_t *window, int32_t *seq_lens, int32_t *q_lens,
                       int32_t *n_cand_next, void *workspace, size_t workspace_bytes, int32_t *err_flag,
                       void *stream) {
    if (num_seqs < 0 || k_max < 0 || vocab <= 0) return SA_ERR_ARG;
    if (k_max > kMaxKMax) return SA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return SA_OK;
    if (!logits || !n_cand || !accepted || !next_tok || (k_max > 0 && !candidates))
        return SA_ERR_ARG;
    if (!aligned(logits, 16)) return SA_ERR_ARG;
    const size_t need = sa_spec_verify_workspace_size(num_seqs, k_max, vocab);
    if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256))
        return SA_ERR_WORKSPACE;
    const int sms = device_sm_count();
    if (sms <= 0) return SA_ERR_CUDA;
    const int64_t rows = static_cast<int64_t>(num_seqs) * (k_max + 1);
    const int64_t max_chunks = (static_cast<int64_t>(vocab) + 1023) / 1024;
    // about five CTAs per SM in total (one wave), each chunk a multiple of 1024 elements
    int64_t n_chunks = std::min<int64_t>(max_chunks, std::max<int64_t>(1, (5 * sms + rows - 1) / rows));
    const int64_t chunk = ((vocab + n_chunks - 1) / n_chunks + 1023) / 1024 * 1024;
    n_chunks = (vocab + chunk - 1) / chunk;
    const int64_t parts = rows * max_chunks;
    const size_t a = ((static_cast<size_t>(parts) * 4 + 255) / 256) * 256;

    VerifyParams p{};
    p.logits = logits;
    p.candidates = candidates;
    p.n_cand = n_cand;
    p.accepted = accepted;
    p.next_tok = next_tok;
    p.window = window;
    p.seq_lens = seq_lens;
    p.q_lens = q_lens;
    p.n_cand_next = n_cand_next;
    p.part_val = static_cast<float *>(workspace);
    p.part_idx = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + a);
    p.counters = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + 2 * a);
    p.err = err_flag;
    p.B = num_seqs;
    p.k_max = k_max;
    p.V = vocab;
    p.n_chunks = static_cast<int32_t>(n_chunks);
    p.chunk = static_cast<int32_t>(chunk);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (launch_verify(p, s) != cudaSuccess) return SA_ERR_CUDA;
    return finish(s, err_flag);
}

int sa_spec_verify_greedy(const float *logits, const int32_t *candidates, const int32_t *n_cand,
                          int32_t num_seqs, int32_t k_max, int32_t vocab, int32_t *accepted,
                          int32_t *next_tok, int32_t *window, void *workspace,
                          size_t workspace_bytes, int32_t *err_flag, void *stream) {
    return verify_impl(logits, candidates, n_cand, num_seqs, k_max, vocab, accepted, next_tok, window,
                       nullptr, nullptr, nullptr, workspace, workspace_bytes, err_flag, stream);
}

int sa_spec_verify_greedy_advance(const float *logits, const int32_t *candidates, const int32_t *n_cand,
                                  int32_t num_seqs, int32_t k_max, int32_t vocab, int32_t *accepted,
                                  int32_t *next_tok, int32_t *window, int32_t *seq_lens, int32_t *q_lens,
                                  int32_t *n_cand_next, void *workspace, size_t workspace_bytes,
                                  int32_t *err_flag, void *stream) {
    if (num_seqs > 0 && (!window || !seq_lens || !q_lens || !n_cand_next)) return SA_ERR_ARG;
    return verify_impl(logits, candidates, n_cand, num_seqs, k_max, vocab, accepted, next_tok, window,
                       seq_lens, q_lens, n_cand_next, workspace, workspace_bytes, err_flag, stream);
}

int sa_defrag_moves(const sa_dims *dims, const int32_t *block_table, const int32_t *seq_lens,
                    int32_t *new_table, int32_t *moves, int32_t *n_moves, int32_t *n_live) {
    if (dims == nullptr || n_moves == nullptr || n_live == nullptr) return SA_ERR_ARG;
    if (dims->num_seqs < 0 || dims->num_pages < 0 || dims->max_pages_per_seq < 0) return SA_ERR_ARG;
    if (dims->num_seqs > 0 && (!block_table || !seq_lens || !new_table)) return SA_ERR_ARG;
    if (dims->num_pages > 0 && !moves) return SA_ERR_ARG;
    return defrag_plan_host(dims->num_seqs, dims->num_pages, dims->max_pages_per_seq, block_table,
                            seq_lens, new_table, moves, n_moves, n_live);
}

int sa_defrag_apply(const sa_dims *dims, uint16_t *k_pages, uint16_t *v_pages, const int32_t *moves,
                    int32_t n_moves, int32_t *err_flag, void *stream) {
    int rc = check_dims(dims);
    if (rc) return rc;
    if (n_moves < 0) return SA_ERR_ARG;
    if (n_moves == 0) return SA_OK;
    if (!k_pages || !v_pages || !moves) return SA_ERR_ARG;
    if (!aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(moves, 4)) return SA_ERR_ARG;
    const int sms = device_sm_count();
    if (sms <= 0) return SA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t page_bytes = static_cast<int64_t>(dims->num_kv_heads) * kPageSize * kHeadDim * 2;
    if (launch_defrag(k_pages, v_pages, moves, n_moves, dims->num_pages, page_bytes, err_flag, sms, s) !=
        cudaSuccess)
        return SA_ERR_CUDA;
    return finish(s, err_flag);
}

int sa_defrag_apply_bytes(int32_t num_pages, int64_t page_bytes, void *pool_a, void *pool_b,
                          const int32_t *moves, int32_t n_moves, int32_t *err_flag, void *stream) {
    if (num_pages < 0 || page_bytes <= 0 || page_bytes % 16 != 0 || n_moves < 0) return SA_ERR_ARG;
    if (n_moves == 0) return SA_OK;
    if (!pool_a || !pool_b || !moves) return SA_ERR_ARG;
    if (!aligned(pool_a, 16) || !aligned(pool_b, 16) || !aligned(moves, 4)) return SA_ERR_ARG;
    const int sms = device_sm_count();
    if (sms <= 0) return SA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (launch_defrag(pool_a, pool_b, moves, n_moves, num_pages, page_bytes, err_flag, sms, s) != cudaSuccess)
        return SA_ERR_CUDA;
    return finish(s, err_flag);
}

// ---------------------------------------------------------------------------
// Paged attention without any allocation by the caller or the library.
//
// Some callers cannot allocate device memory at all: a plugin that runs inside
// a serving process whose memory pool already owns every byte of the GPU, or a
// decode loop that may not call cudaMalloc because it synchronises the whole
// device. For them the kernels' scratch (partial accumulators, their maxima
// and sums, and the counters) lives in one fixed array in this file. The
// array belongs to this file's module, which the driver loads on a device at
// the first lookup of its address there (the first call of the entry point on
// that device): from then on the 16 MiB stay reserved on that device until
// the process exits. The array is zero when loaded and every call that
// completes without a device error leaves its counters at zero.
// ---------------------------------------------------------------------------
constexpr size_t kStaticScratchBytes = size_t{16} << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
struct ScratchEntry {
    CUcontext ctx;  // the context the address belongs to (a device reset makes a new one)
    void *ptr;      // device address of g_static_scratch in it
};
ScratchEntry g_scratch[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
CtxGetCurrentFn ctx_get_current_fn() {
    static CtxGetCurrentFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<CtxGetCurrentFn>(p);
    }();
    return fn;
}

// Device address of the fixed scratch on the current device, looked up with
// that device current (the host-side name of the array is not a device address
// and is never passed to a kernel) and kept until the device's context
// changes.
int static_scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SA_ERR_UNSUPPORTED;
    if (cudaFree(nullptr) != cudaSuccess) return SA_ERR_CUDA;  // makes the device's context current (frees nothing)
    CUcontext ctx = nullptr;
    CtxGetCurrentFn get = ctx_get_current_fn();
    if (get == nullptr || get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return SA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchEntry &e = g_scratch[dev];
    if (e.ptr == nullptr || e.ctx != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return SA_ERR_CUDA;
        e.ctx = ctx;
        e.ptr = p;
    }
    *out = e.ptr;
    return SA_OK;
}

}  // namespace

int sa_paged_attn_noalloc(const sa_dims *dims, const uint16_t *q, const uint16_t *k_pages,
                          const uint16_t *v_pages, const int32_t *block_table,
                          const int32_t *seq_lens, const int32_t *q_lens, float scale,
                          uint16_t *out, int32_t *err_flag, void *stream) {
    int rc = check_dims(dims);
    if (rc) return rc;
    if (attn_ws_bytes(*dims, nullptr) > kStaticScratchBytes) return SA_ERR_WORKSPACE;  // shapes exceed the fixed scratch
    void *ws = nullptr;
    rc = static_scratch_address(&ws);
    if (rc) return rc;
    return sa_paged_attn(dims, q, k_pages, v_pages, block_table, seq_lens, q_lens, scale, out,
                         nullptr, ws, kStaticScratchBytes, err_flag, stream);
}

}  // extern "C"
