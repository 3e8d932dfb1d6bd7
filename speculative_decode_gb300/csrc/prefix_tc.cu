// prefix_tc.cu -- shared-prefix attention on the tcgen05 tensor cores.
//
// ExLlamaV2 "Dynamic Generator" page, "Deduplication": many sequences index
// the same physical pages for a common prefix. Attention over such a run of
// pages is one dense contraction: the query rows of every member sequence
// (G heads x its new tokens, all for one KV head) against the run's keys and
// values. This kernel streams each shared 128-token K/V tile from HBM once per
// 128-row tile of queries (row tiles of one run share their tiles through L2)
// and computes
//     S = Q K^T          (tcgen05.mma, bf16 x bf16 -> fp32 in tensor memory)
//     P = exp2(S*scale*log2e - m)  online, one thread per row, bf16 to smem
//     O += P V           (tcgen05.mma, fp32 accumulator in tensor memory)
// and stores, per row, an fp32 partial (O, m, l) that the split kernel merges
// with the rest of the sequence's keys.
//
// CTA = 6 warps: warps 0-3 softmax and epilogue (thread t owns row t, which is
// tensor-memory lane t), warp 4 the TMA producer, warp 5 allocates tensor
// memory and issues the MMAs (one elected thread). S is double-buffered in
// tensor memory, so Q K^T of the next tile and P V of the previous one run on
// the tensor cores while the softmax of the current tile runs on the CUDA
// cores. Operands sit in shared
// memory in the 128-byte-swizzled K-major layout the TMA writes (Q, K and P)
// or the MN-major one (V), described to the tensor core by shared-memory
// matrix descriptors. Every wait is bounded; on timeout the CTA flags
// SA_ERR_TIMEOUT, drains what it issued and frees its tensor memory.
#include <cuda_bf16.h>

#include "common.cuh"
#include "plan.h"

namespace sa {

namespace {

constexpr int kM = 128;                       // rows per tile (tensor-memory lanes)
constexpr int kN = 128;                       // keys per K/V tile
constexpr int kSub = kN * 128;                // one 64-wide bf16 column block: 128 rows x 128 B = 16 KiB
constexpr int kQBytes = 2 * kSub;             // Q [128 rows][128 d]
constexpr int kPBytes = 2 * kSub;             // P [128 rows][128 keys]
constexpr int kKVStage = 4 * kSub;            // K (2 blocks) + V (2 blocks) = 64 KiB
constexpr int kStagesTC = 2;
constexpr int kTmemCols = 512;                // S0: columns 0-127, S1: 128-255, O: 256-383
constexpr int kThreads = 192;

constexpr int kOffQ = 0;
constexpr int kOffP = kOffQ + kQBytes;
constexpr int kOffKV = kOffP + kPBytes;
constexpr int kOffBar = kOffKV + kStagesTC * kKVStage;
constexpr int kSmemBytes = kOffBar + 256 + 1024;  // barriers, tensor-memory address, alignment slack

// ------------------------------------------------------------ tcgen05 helpers
// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor for kind::f16: fp32 accumulate, bf16 A and B, A
// K-major, B K-major or MN-major, M = 128, N = 128.
__host__ __device__ constexpr uint32_t idesc_bf16(bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn_major ? (1u << 16) : 0u) |
           (static_cast<uint32_t>(kN >> 3) << 17) | (static_cast<uint32_t>(kM >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive 32-bit columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
        "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
        "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])),
        "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
        "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])),
        "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

struct PrefixParams {
    const uint16_t *q;
    const int32_t *block_table;
    // plan mode: work items and rows from a shared-run plan
    const int32_t *run_desc;
    const int32_t *run_rows;
    const int32_t *tiles;
    // sequence mode: one work item per (sequence, KV head, row tile, page chunk)
    const int32_t *seq_lens;
    const int32_t *q_lens;
    int32_t seq_mode, B, max_q_len, total_q, min_rows, mtiles, max_chunks, chunk_pages;
    float *ws_acc;
    float *ws_ml;
    int32_t *err;
    int32_t Hq, Hkv, G, max_pages, num_pages;
    int64_t n_rows_total;
    float qscale;  // scale * log2(e)
};

__global__ void __launch_bounds__(kThreads, 1)
    prefix_tc_kernel(const PrefixParams P, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint64_t *kv_full = bars;           // [2] K/V tile landed
    uint64_t *kv_empty = bars + 2;      // [2] K/V stage free again
    uint64_t *q_full = bars + 4;        // Q rows written
    uint64_t *s_full = bars + 5;        // [2] S buffer holds Q K^T of a tile
    uint64_t *p_full = bars + 7;        // P written (and its S buffer read)
    uint64_t *p_free = bars + 8;        // P V finished: P free, O up to date
    uint64_t *mma_done = bars + 9;      // every MMA finished (before freeing tensor memory)
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(bars + 10);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(bars + 11);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    // ---- the work item
    int g, row0, pc_lo, pc_hi, chunk, member, row_count, rows_begin = 0;
    int key_end = 0x7fffffff;  // keys at or past this position are not in the cache
    int seq_n = 0, seq_qstart = 0;
    if (!P.seq_mode) {  // (run, KV head, 128-row tile, page chunk) from the plan
        const int32_t *it = P.tiles + static_cast<int64_t>(blockIdx.x) * kTileInts;
        const int run = it[0];
        g = it[1];
        row0 = it[2];
        pc_lo = it[3];
        pc_hi = it[4];
        chunk = it[5];
        const int32_t *rd = P.run_desc + static_cast<int64_t>(run) * kRunDescInts;
        rows_begin = rd[2];
        row_count = rd[3];
        member = rd[5];
    } else {  // (sequence, KV head, 128-row tile, page chunk): rows = G heads x new tokens
        int idx = blockIdx.x;
        chunk = idx % P.max_chunks;
        idx /= P.max_chunks;
        const int mt = idx % P.mtiles;
        idx /= P.mtiles;
        g = idx % P.Hkv;
        member = idx / P.Hkv;
        const int T = P.seq_lens[member];
        seq_n = P.q_lens[member];
        const int npages = (T + kPageSize - 1) / kPageSize;
        row_count = P.G * seq_n;
        row0 = mt * kM;
        pc_lo = chunk * P.chunk_pages;
        pc_hi = min(npages, pc_lo + P.chunk_pages);
        key_end = T;
        // packed query row of the sequence's first new token (block reduction)
        __shared__ int red[kThreads / 32];
        int part = 0;
        for (int k = tid; k < member; k += kThreads) part += P.q_lens[k];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0) red[warp] = part;
        __syncthreads();
        for (int w = 0; w < kThreads / 32; ++w) seq_qstart += red[w];
        // the same eligibility rule as the split kernel's, which merges these partials
        const bool work = seq_n > 0 && seq_n <= T && seq_n <= P.max_q_len && npages <= P.max_pages &&
                          row_count >= P.min_rows && seq_qstart + seq_n <= P.total_q && pc_lo < pc_hi &&
                          row0 < row_count;
        if (!work) return;  // uniform over the CTA: nothing allocated yet
    }
    // 128-key tiles of the chunk that hold keys below key_end
    const int n_kv = (min(pc_hi * kPageSize, key_end) - pc_lo * kPageSize + kN - 1) / kN;

    if (tid == 0) {
        for (int s = 0; s < kStagesTC; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        mbar_init(q_full, kM);
        mbar_init(&s_full[0], 1);
        mbar_init(&s_full[1], 1);
        mbar_init(p_full, kM);
        mbar_init(p_free, 1);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 5) {  // tensor memory for S and O
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(const_cast<uint32_t *>(tmem_slot))),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_o = tmem + 2 * kN;  // S buffers at columns 0 and kN

    const uint32_t sQ = smem_u32(smem + kOffQ), sP = smem_u32(smem + kOffP), sKV = smem_u32(smem + kOffKV);

    if (warp < 4) {
        // ================= softmax / epilogue warps: thread t owns row t
        const int t = tid;
        const int r = row0 + t;
        const bool valid = r < row_count;
        const bool warp_valid = __any_sync(0xffffffffu, valid);  // warps without rows skip the softmax
        int32_t token = 0, hl = 0, limit = -1, slot = 0;
        if (valid) {
            if (!P.seq_mode) {
                const int32_t *rr = P.run_rows + static_cast<int64_t>(rows_begin + r) * 4;
                token = rr[0];
                hl = rr[1];
                limit = rr[2];
                slot = rr[3] + chunk;
            } else {
                token = seq_qstart + r / P.G;
                hl = r % P.G;
                limit = key_end - seq_n + r / P.G;
                slot = chunk;
            }
        }
        if (!warp_valid) {  // P rows of rows that do not exist stay zero
#pragma unroll
            for (int c = 0; c < kN / 8; ++c)
                *reinterpret_cast<uint4 *>(smem + kOffP + (c >> 3) * kSub + sw128_offset(t, c & 7)) = make_uint4(0, 0, 0, 0);
        }
        // Q row t -> shared memory, 128-byte swizzled K-major (two 64-column blocks)
        {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                P.q + (static_cast<int64_t>(token) * P.Hq + g * P.G + hl) * kHeadDim);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const uint4 w = valid ? src[c] : make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4 *>(smem + kOffQ + (c >> 3) * kSub + sw128_offset(t, c & 7)) = w;
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(q_full);
        }
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        float m_ref = -INFINITY, lsum = 0.f;
        bool ok = true;
        for (int i = 0; i < n_kv && ok; ++i) {
            ok = __all_sync(0xffffffffu, mbar_wait(&s_full[i & 1], (i >> 1) & 1));
            if (!ok) break;
            tc_fence_after();
            const int pos0 = pc_lo * kPageSize + i * kN;
            if (!warp_valid) {
                if (i > 0) {
                    ok = __all_sync(0xffffffffu, mbar_wait(p_free, (i - 1) & 1));
                    if (!ok) break;
                }
                if (pos0 + t >= key_end) {  // keys past the end may hold stale data: zero their V row
                    uint8_t *vrow = smem + kOffKV + (i % kStagesTC) * kKVStage + 2 * kSub + t * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        *reinterpret_cast<uint4 *>(vrow + c * 16) = make_uint4(0, 0, 0, 0);
                        *reinterpret_cast<uint4 *>(vrow + kSub + c * 16) = make_uint4(0, 0, 0, 0);
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                tc_fence_before();
                mbar_arrive(p_full);
                continue;
            }
            const uint32_t tmem_s = tmem + (i & 1) * kN;
            float x[kN];
            const bool whole = pos0 + kN - 1 <= limit;  // no key of this tile is masked for row t
#pragma unroll
            for (int c = 0; c < kN / 32; ++c) {
                float v[32];
                tmem_ld32(tmem_s + lane_base + c * 32, v);
                if (whole) {
#pragma unroll
                    for (int k = 0; k < 32; ++k) x[c * 32 + k] = v[k] * P.qscale;
                } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k)
                        x[c * 32 + k] = pos0 + c * 32 + k <= limit ? v[k] * P.qscale : -INFINITY;
                }
            }
            float tmax = -INFINITY;
#pragma unroll
            for (int k = 0; k < kN; ++k) tmax = fmaxf(tmax, x[k]);
            // move the reference max only when it grows by more than 2^8, so
            // that tensor-memory O is rarely rescaled (p stays below 256)
            const bool grow = tmax > m_ref + 8.f;
            const float m_new = grow ? tmax : m_ref;
            const float alpha = grow ? exp2f(m_ref - m_new) : 1.f;  // 0 when m_ref was -inf
            const float m_use = m_new == -INFINITY ? 0.f : m_new;
            // probabilities, packed to bf16 pairs while the tensor cores finish P V
            uint32_t pw[kN / 2];
            float psum = 0.f;
#pragma unroll
            for (int k = 0; k < kN / 2; ++k) {
                const float a = exp2f(x[2 * k] - m_use), b = exp2f(x[2 * k + 1] - m_use);
                psum += a + b;
                const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
                pw[k] = *reinterpret_cast<const uint32_t *>(&h);
            }
            if (i > 0) {  // P V of the previous tile must be done before P and O change
                ok = __all_sync(0xffffffffu, mbar_wait(p_free, (i - 1) & 1));
                if (!ok) break;
                tc_fence_after();
                if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
                    for (int c = 0; c < kHeadDim / 32; ++c) {
                        float o[32];
                        tmem_ld32(tmem_o + lane_base + c * 32, o);
#pragma unroll
                        for (int k = 0; k < 32; ++k) o[k] *= alpha;
                        tmem_st32(tmem_o + lane_base + c * 32, o);
                    }
                }
            }
            lsum = lsum * alpha + psum;
            m_ref = m_new;
            // P row t -> shared memory (bf16, 128-byte swizzled K-major)
#pragma unroll
            for (int c = 0; c < kN / 8; ++c)
                *reinterpret_cast<uint4 *>(smem + kOffP + (c >> 3) * kSub + sw128_offset(t, c & 7)) =
                    make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
            if (pos0 + t >= key_end) {  // keys past the end may hold stale data: zero their V row
                uint8_t *vrow = smem + kOffKV + (i % kStagesTC) * kKVStage + 2 * kSub + t * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    *reinterpret_cast<uint4 *>(vrow + c * 16) = make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4 *>(vrow + kSub + c * 16) = make_uint4(0, 0, 0, 0);
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            tc_fence_before();
            mbar_arrive(p_full);
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(p_free, (n_kv - 1) & 1));  // the last P V
        if (!ok) {
            *abort_flag = 1;
            if (lane == 0) flag_error(P.err, kErrBitTimeout);
        } else if (warp_valid) {
            tc_fence_after();
            // epilogue: fp32 partial (O, m, l) of this row for the merge
            const int64_t orow = static_cast<int64_t>(token) * P.Hq + g * P.G + hl;
            const int64_t wi = static_cast<int64_t>(slot) * P.n_rows_total + orow;
#pragma unroll
            for (int c = 0; c < kHeadDim / 32; ++c) {
                float o[32];
                tmem_ld32(tmem_o + lane_base + c * 32, o);
                if (valid) {
                    float4 *dst = reinterpret_cast<float4 *>(P.ws_acc + wi * kHeadDim + c * 32);
#pragma unroll
                    for (int k = 0; k < 8; ++k) dst[k] = make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
                }
            }
            if (valid) *reinterpret_cast<float2 *>(P.ws_ml + wi * 2) = make_float2(m_ref, lsum);
        }
    } else if (warp == 4) {
        // ================= TMA producer
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_last();  // row tiles of the run re-read these
            int issued = 0;
            for (int i = 0; i < n_kv; ++i) {
                const int s = i % kStagesTC;
                if (i >= kStagesTC && !mbar_wait(&kv_empty[s], ((i / kStagesTC) - 1) & 1)) {
                    *abort_flag = 1;
                    flag_error(P.err, kErrBitTimeout);
                    break;
                }
                if (*abort_flag) break;
                const int page = pc_lo + (i >> 1);
                const int pid = P.block_table[static_cast<int64_t>(member) * P.max_pages + page];
                // (sequence mode: the last tile may reach past the sequence's keys; the
                // rows past the end are zeroed in shared memory before P V)
                uint8_t *dst = smem + kOffKV + s * kKVStage;
                if (pid < 0 || pid >= P.num_pages) {  // the planner only takes valid pages
                    flag_error(P.err, kErrBitPageOOB);
                    mbar_arrive(&kv_full[s]);
                } else {
                    const int y = (pid * P.Hkv + g) * kPageSize + (i & 1) * kN;
                    mbar_arrive_expect_tx(&kv_full[s], kKVStage);
                    tma_load_2d(dst, &tmk, &kv_full[s], 0, y, policy);
                    tma_load_2d(dst + kSub, &tmk, &kv_full[s], 64, y, policy);
                    tma_load_2d(dst + 2 * kSub, &tmv, &kv_full[s], 0, y, policy);
                    tma_load_2d(dst + 3 * kSub, &tmv, &kv_full[s], 64, y, policy);
                }
                ++issued;
            }
            // copies still in flight finish before the CTA can leave
            for (int i = issued - kStagesTC < 0 ? 0 : issued - kStagesTC; i < issued; ++i)
                (void)mbar_wait(&kv_full[i % kStagesTC], (i / kStagesTC) & 1);
        }
    } else {
        // ================= MMA issuer (one thread). Order: QK(0), then for
        // each tile i >= 1: QK(i) into the other S buffer, PV(i-1).
        if (lane == 0) {
            constexpr uint32_t kIdQK = idesc_bf16(false), kIdPV = idesc_bf16(true);
            bool ok = mbar_wait(q_full, 0);
            for (int i = 0; ok && i <= n_kv; ++i) {
                if (i < n_kv) {  // S[i&1] = Q K(i)^T; S[i&1] was last read by softmax(i-2)
                    const int s = i % kStagesTC;
                    ok = mbar_wait(&kv_full[s], (i / kStagesTC) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t sK = sKV + s * kKVStage;
#pragma unroll
                    for (int k = 0; k < kHeadDim / 16; ++k) {
                        const uint64_t a = smem_desc(sQ + (k >> 2) * kSub + (k & 3) * 32, 16, 1024);
                        const uint64_t b = smem_desc(sK + (k >> 2) * kSub + (k & 3) * 32, 16, 1024);
                        mma_bf16(tmem + (i & 1) * kN, a, b, kIdQK, k > 0);
                    }
                    mma_commit(&s_full[i & 1]);
                }
                if (i > 0) {  // O += P(i-1) V(i-1) once the softmax has written P(i-1)
                    ok = mbar_wait(p_full, (i - 1) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t sV = sKV + ((i - 1) % kStagesTC) * kKVStage + 2 * kSub;
#pragma unroll
                    for (int k = 0; k < kN / 16; ++k) {
                        const uint64_t a = smem_desc(sP + (k >> 2) * kSub + (k & 3) * 32, 16, 1024);
                        const uint64_t b = smem_desc(sV + k * 16 * 128, kSub, 1024);
                        mma_bf16(tmem_o, a, b, kIdPV, i > 1 || k > 0);
                    }
                    mma_commit(&kv_empty[(i - 1) % kStagesTC]);
                    mma_commit(p_free);
                }
            }
            if (!ok) {
                *abort_flag = 1;
                flag_error(P.err, kErrBitTimeout);
            }
            // every MMA this thread issued completes before tensor memory is freed
            mma_commit(mma_done);
        }
    }
    if (warp == 5 && lane == 0) (void)mbar_wait(mma_done, 0);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

}  // namespace

cudaError_t launch_prefix_tc(const sa_dims &d, const PlanDevice &pd, const uint16_t *q,
                             const CUtensorMap &tmk, const CUtensorMap &tmv, float scale,
                             float *ws_acc, float *ws_ml, int64_t rows_total, int32_t *err,
                             const int32_t *block_table, cudaStream_t stream) {
    static cudaError_t attr = cudaFuncSetAttribute(prefix_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   kSmemBytes);
    if (attr != cudaSuccess) return attr;
    PrefixParams p{};
    p.q = q;
    p.block_table = block_table;
    p.run_desc = pd.run_desc;
    p.run_rows = pd.run_rows;
    p.tiles = pd.tiles;
    p.ws_acc = ws_acc;
    p.ws_ml = ws_ml;
    p.err = err;
    p.Hq = d.num_q_heads;
    p.Hkv = d.num_kv_heads;
    p.G = d.num_q_heads / d.num_kv_heads;
    p.max_pages = d.max_pages_per_seq;
    p.num_pages = d.num_pages;
    p.n_rows_total = rows_total;
    p.qscale = scale * 1.4426950408889634f;
    prefix_tc_kernel<<<pd.num_tiles, kThreads, kSmemBytes, stream>>>(p, tmk, tmv);
    return cudaGetLastError();
}

cudaError_t launch_seq_tc(const sa_dims &d, const SeqTcConfig &c, const uint16_t *q,
                          const CUtensorMap &tmk, const CUtensorMap &tmv, float scale,
                          float *ws_acc, float *ws_ml, int64_t rows_total, int32_t *err,
                          const int32_t *block_table, const int32_t *seq_lens,
                          const int32_t *q_lens, cudaStream_t stream) {
    static cudaError_t attr = cudaFuncSetAttribute(prefix_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   kSmemBytes);
    if (attr != cudaSuccess) return attr;
    PrefixParams p{};
    p.q = q;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.q_lens = q_lens;
    p.seq_mode = 1;
    p.B = d.num_seqs;
    p.max_q_len = d.max_q_len;
    p.total_q = d.total_q;
    p.min_rows = c.min_rows;
    p.mtiles = c.mtiles;
    p.max_chunks = c.max_chunks;
    p.chunk_pages = c.chunk_pages;
    p.ws_acc = ws_acc;
    p.ws_ml = ws_ml;
    p.err = err;
    p.Hq = d.num_q_heads;
    p.Hkv = d.num_kv_heads;
    p.G = d.num_q_heads / d.num_kv_heads;
    p.max_pages = d.max_pages_per_seq;
    p.num_pages = d.num_pages;
    p.n_rows_total = rows_total;
    p.qscale = scale * 1.4426950408889634f;
    const int64_t grid = static_cast<int64_t>(d.num_seqs) * d.num_kv_heads * c.mtiles * c.max_chunks;
    if (grid == 0) return cudaSuccess;
    prefix_tc_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(p, tmk, tmv);
    return cudaGetLastError();
}

int prefix_tile_rows() { return kN; }

}  // namespace sa
