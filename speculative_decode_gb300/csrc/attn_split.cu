// attn_split.cu -- page-streamed attention on the CUDA cores (split-K over
// pages), for decode (q_len = 1) and causal multi-query verification
// (q_len = k + 1), plus the combine pass that merges split partials.
//
// What it computes: for each sequence b, new query token i and query head h,
// softmax(scale * q . K_b^T) V_b over the keys at positions
// 0 .. seq_len - q_len + i, with K_b/V_b gathered through the block table
// (ExLlamaV2 "Dynamic Generator" page, "Continuous batching"; causal rows as
// in the Hugging Face "Assisted Generation" page, "How Assisted Generation
// works"). The softmax is evaluated online over 32-token tiles and the pages
// of a sequence are cut into splits whose partial (max, sum, accumulator)
// states are merged exactly by the combine pass.
//
// Design (sm_103a):
//  * Work unit = (sequence, KV head, row block, split of `pages_per_split`
//    pages). Rows are the G query heads of the KV head times the sequence's
//    query tokens, so each K/V byte read serves all of them.
//  * One warp owns a unit from start to finish: lane 0 streams the unit's
//    32-token K and V tiles with TMA (2-D tensor copies, 128-byte swizzle)
//    into a private ring of `S` stages; all 32 lanes compute. Warps are
//    independent (no block barriers), the grid is persistent and each warp
//    walks units gw, gw + total_warps, ... with the copies of its next tiles
//    already in flight while it computes, across unit boundaries.
//  * QK^T: lane = token; each lane reads its key row chunk by chunk from the
//    swizzled tile (conflict-free) while the pre-scaled fp32 queries are
//    broadcast from shared memory. Online softmax in log2 units with warp
//    shuffles for the tile maxima. PV: lane = 4 output dims; p broadcast from
//    shared memory, V read from the swizzled tile (conflict-free).
//  * Every wait on a TMA barrier is bounded (common.cuh); on timeout the
//    warp flags SA_ERR_TIMEOUT, drains its copies in flight and leaves.
#include "common.cuh"

namespace sa {

namespace {

constexpr int kTile = 32;                     // tokens per stage, one per lane
constexpr int kHalfBytes = kTile * 128;       // 32 rows x 64 bf16 (one 128-byte swizzle span)
constexpr int kStageBytes = 4 * kHalfBytes;   // K[0:64], K[64:128], V[0:64], V[64:128]
constexpr int kStages = 2;

template <int R>
struct WarpLayout {
    static constexpr int kStageOff = 0;
    static constexpr int kQOff = kStages * kStageBytes;                 // fp32 [R][128]
    static constexpr int kPOff = kQOff + R * kHeadDim * 4;             // fp32 [32][R]
    static constexpr int kBarOff = kPOff + kTile * R * 4;              // uint64 [kStages]
    static constexpr int kBytes = ((kBarOff + kStages * 8) + 1023) / 1024 * 1024;
};

struct Unit {
    int b, kvh, rb, T, n, t_lo, t_hi, n_tiles, slot;
    bool direct, ok;
};

__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Packed query rows that precede sequence b (sum of q_lens[0..b)).
__device__ __forceinline__ int q_row_start(const int32_t *q_lens, int b, int lane) {
    int s = 0;
    for (int k = lane; k < b; k += 32) s += q_lens[k];
    return warp_sum_i(s);
}

// Decode unit u. Returns false when the unit has no work at all. Warp-uniform;
// every lane must call it. Sets U.ok = false when a page id is out of range.
template <int R>
__device__ bool decode_unit(const SplitParams &P, int64_t u, Unit &U, int lane) {
    const int per_split = P.B * P.Hkv * P.n_row_blocks;
    const int split = static_cast<int>(u / per_split);
    int rem = static_cast<int>(u % per_split);
    U.b = rem / (P.Hkv * P.n_row_blocks);
    rem %= P.Hkv * P.n_row_blocks;
    U.kvh = rem / P.n_row_blocks;
    U.rb = rem % P.n_row_blocks;
    U.T = P.seq_lens[U.b];
    U.n = P.q_lens[U.b];
    if (U.n <= 0 || U.n > U.T || U.n > P.max_q_len) return false;
    if (U.rb * R >= P.G * U.n) return false;
    const int npages = (U.T + kPageSize - 1) / kPageSize;
    const int skip = P.skip_pages ? P.skip_pages[U.b] : 0;
    const int p_lo = skip + split * P.pages_per_split;
    if (p_lo >= npages) return false;
    const int p_hi = min(p_lo + P.pages_per_split, npages);
    U.t_lo = p_lo * kPageSize;
    U.t_hi = min(p_hi * kPageSize, U.T);
    U.n_tiles = (U.t_hi - U.t_lo + kTile - 1) / kTile;
    const int nsplit = (npages - skip + P.pages_per_split - 1) / P.pages_per_split;
    const int runs = P.run_slots ? P.run_slots[U.b] : 0;
    U.direct = (nsplit == 1 && runs == 0);
    U.slot = P.slot_base + split;
    bool ok = npages <= P.max_pages;
    for (int j = p_lo + lane; ok && j < p_hi; j += 32) {
        const int id = P.block_table[static_cast<int64_t>(U.b) * P.max_pages + j];
        ok = id >= 0 && id < P.num_pages;
    }
    U.ok = __all_sync(0xffffffffu, ok);
    return true;
}

template <int R>
__global__ void __launch_bounds__(32) split_attn_kernel(const SplitParams P,
                                                        const __grid_constant__ CUtensorMap tmk,
                                                        const __grid_constant__ CUtensorMap tmv) {
    using L = WarpLayout<R>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int lane = threadIdx.x & 31;
    uint8_t *stage_base = smem + L::kStageOff;
    float(*qs)[kHeadDim] = reinterpret_cast<float(*)[kHeadDim]>(smem + L::kQOff);
    float(*pbuf)[R] = reinterpret_cast<float(*)[R]>(smem + L::kPOff);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kBarOff);

    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
    }
    __syncwarp();

    const int64_t gw = blockIdx.x;          // one warp per CTA
    const int64_t TW = gridDim.x;
    // K/V are streamed once unless several row blocks share a tile
    const uint64_t policy = P.evict_first ? l2_policy_evict_first() : l2_policy_evict_normal();

    // ---- issue cursor: walks the same (unit, tile) sequence as the consumer
    int64_t iu = gw - TW;
    int itile = 0, intiles = 0;
    Unit IU;
    uint32_t issued = 0;
    auto issue_next = [&]() {
        while (itile >= intiles) {
            iu += TW;
            if (iu >= P.n_units) return;
            intiles = 0;
            if (decode_unit<R>(P, iu, IU, lane) && IU.ok) intiles = IU.n_tiles;
            itile = 0;
        }
        const int t0 = IU.t_lo + itile * kTile;
        const int pid = P.block_table[static_cast<int64_t>(IU.b) * P.max_pages + t0 / kPageSize];
        const int y = (pid * P.Hkv + IU.kvh) * kPageSize + (t0 % kPageSize);
        const int s = issued % kStages;
        if (lane == 0) {
            uint8_t *dst = stage_base + s * kStageBytes;
            mbar_arrive_expect_tx(&full[s], kStageBytes);
            tma_load_2d(dst, &tmk, &full[s], 0, y, policy);
            tma_load_2d(dst + kHalfBytes, &tmk, &full[s], 64, y, policy);
            tma_load_2d(dst + 2 * kHalfBytes, &tmv, &full[s], 0, y, policy);
            tma_load_2d(dst + 3 * kHalfBytes, &tmv, &full[s], 64, y, policy);
        }
        ++issued;
        ++itile;
    };
    auto issue_has_more = [&]() -> bool {
        while (itile >= intiles) {
            if (iu + TW >= P.n_units) return false;
            iu += TW;
            intiles = 0;
            if (decode_unit<R>(P, iu, IU, lane) && IU.ok) intiles = IU.n_tiles;
            itile = 0;
        }
        return true;
    };
    for (int s = 0; s < kStages; ++s)
        if (issue_has_more()) issue_next();

    uint32_t consumed = 0;
    // Bounded-wait failure: flag, wait (bounded) for the copies still in
    // flight into this warp's ring, and leave.
    auto bail_out = [&]() {
        flag_error(P.err, kErrBitTimeout);
        for (uint32_t c = consumed; c < issued; ++c)
            (void)mbar_wait(&full[c % kStages], (c / kStages) & 1);
    };

    const int d0 = lane * 4;  // output dims owned by this lane in PV
    const uint32_t v_lane_off = 2 * kHalfBytes + (lane >> 4) * kHalfBytes + ((lane & 1) << 3);
    const uint32_t v_chunk = (lane & 15) >> 1;

    for (int64_t u = gw; u < P.n_units; u += TW) {
        Unit U;
        if (!decode_unit<R>(P, u, U, lane)) {
            if (lane == 0) {
                const int n = P.q_lens[U.b], T = P.seq_lens[U.b];
                if (n > T || n > P.max_q_len) flag_error(P.err, kErrBitQlen);
            }
            continue;
        }
        const int qstart = q_row_start(P.q_lens, U.b, lane);
        const int rows = P.G * U.n;
        if (qstart + U.n > P.total_q) {  // q_lens disagree with dims.total_q
            if (lane == 0) flag_error(P.err, kErrBitQlen);
            continue;
        }
        if (!U.ok) {
            // Unit skipped: report it and leave an empty partial (or zeros).
            if (lane == 0) flag_error(P.err, kErrBitPageOOB);
            for (int r = 0; r < R; ++r) {
                const int rr = U.rb * R + r;
                if (rr >= rows) break;
                const int64_t row = static_cast<int64_t>(qstart + rr / P.G) * P.Hq + U.kvh * P.G + rr % P.G;
                if (U.direct) {
                    *reinterpret_cast<uint2 *>(P.out + row * kHeadDim + d0) = make_uint2(0, 0);
                } else {
                    const int64_t w = static_cast<int64_t>(U.slot) * P.n_rows_total + row;
                    *reinterpret_cast<float4 *>(P.ws_acc + w * kHeadDim + d0) = make_float4(0, 0, 0, 0);
                    if (lane == 0) *reinterpret_cast<float2 *>(P.ws_ml + w * 2) = make_float2(-INFINITY, 0.f);
                }
            }
            continue;
        }

        // ---- queries of this unit -> shared memory, pre-scaled by scale*log2(e)
        const int nvr = min(R, rows - U.rb * R);   // valid rows of this block
        const int lim0 = U.T - U.n;                // last key visible to query token 0
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int rr = U.rb * R + r;
            float4 qv = make_float4(0, 0, 0, 0);
            if (r < nvr) {
                const int64_t row = static_cast<int64_t>(qstart + rr / P.G) * P.Hq + U.kvh * P.G + rr % P.G;
                const uint2 w = *reinterpret_cast<const uint2 *>(P.q + row * kHeadDim + d0);
                qv = make_float4(bf16_lo(w.x) * P.qscale, bf16_hi(w.x) * P.qscale,
                                 bf16_lo(w.y) * P.qscale, bf16_hi(w.y) * P.qscale);
            }
            *reinterpret_cast<float4 *>(&qs[r][d0]) = qv;
        }
        __syncwarp();

        float m[R], l[R], acc[R][4];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            m[r] = -INFINITY;
            l[r] = 0.f;
            acc[r][0] = acc[r][1] = acc[r][2] = acc[r][3] = 0.f;
        }

        for (int k = 0; k < U.n_tiles; ++k) {
            const int s = consumed % kStages;
            const bool arrived = mbar_wait(&full[s], (consumed / kStages) & 1);
            if (!__all_sync(0xffffffffu, arrived)) {
                bail_out();
                return;
            }
            const uint8_t *st = stage_base + s * kStageBytes;
            const int t0 = U.t_lo + k * kTile;

            // ---- S = q . K^T for this lane's token
            float sc[R];
#pragma unroll
            for (int r = 0; r < R; ++r) sc[r] = 0.f;
            constexpr int kUnrollC = R <= 4 ? 16 : R <= 8 ? 4 : 2;
#pragma unroll kUnrollC
            for (int c = 0; c < 16; ++c) {
                const uint4 kw = *reinterpret_cast<const uint4 *>(
                    st + (c >> 3) * kHalfBytes + sw128_offset(lane, c & 7));
                const float k0 = bf16_lo(kw.x), k1 = bf16_hi(kw.x), k2 = bf16_lo(kw.y),
                            k3 = bf16_hi(kw.y), k4 = bf16_lo(kw.z), k5 = bf16_hi(kw.z),
                            k6 = bf16_lo(kw.w), k7 = bf16_hi(kw.w);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float4 qa = *reinterpret_cast<const float4 *>(&qs[r][c * 8]);
                    const float4 qb = *reinterpret_cast<const float4 *>(&qs[r][c * 8 + 4]);
                    float a = sc[r];
                    a = fmaf(qa.x, k0, a);
                    a = fmaf(qa.y, k1, a);
                    a = fmaf(qa.z, k2, a);
                    a = fmaf(qa.w, k3, a);
                    a = fmaf(qb.x, k4, a);
                    a = fmaf(qb.y, k5, a);
                    a = fmaf(qb.z, k6, a);
                    a = fmaf(qb.w, k7, a);
                    sc[r] = a;
                }
            }
            // ---- causal / length mask and online softmax (log2 units). Only
            // tiles that reach past the first query's last key, or blocks with
            // padding rows, need the per-row test.
            const int pos = t0 + lane;
            const bool edge = t0 + kTile - 1 > lim0 || nvr < R;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float sv = sc[r];
                if (edge) {
                    const int i_r = (U.rb * R + r) / P.G;
                    if (r >= nvr || pos > lim0 + i_r) sv = -INFINITY;
                }
                const float m_new = fmaxf(m[r], warp_max_f(sv));
                const float m_use = m_new == -INFINITY ? 0.f : m_new;
                const float alpha = exp2f(m[r] - m_use);
                const float pr = exp2f(sv - m_use);
                l[r] = l[r] * alpha + pr;
                acc[r][0] *= alpha;
                acc[r][1] *= alpha;
                acc[r][2] *= alpha;
                acc[r][3] *= alpha;
                m[r] = m_new;
                pbuf[lane][r] = pr;
            }
            __syncwarp();

            // ---- O += P V over the valid tokens of the tile
            const int nvalid = min(kTile, U.t_hi - t0);
            for (int t = 0; t < nvalid; ++t) {
                const uint2 vw = *reinterpret_cast<const uint2 *>(st + v_lane_off + sw128_offset(t, v_chunk));
                const float v0 = bf16_lo(vw.x), v1 = bf16_hi(vw.x), v2 = bf16_lo(vw.y), v3 = bf16_hi(vw.y);
#pragma unroll
                for (int r4 = 0; r4 < R / 4; ++r4) {
                    const float4 pp = *reinterpret_cast<const float4 *>(&pbuf[t][r4 * 4]);
                    const float pr[4] = {pp.x, pp.y, pp.z, pp.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int r = r4 * 4 + j;
                        acc[r][0] = fmaf(pr[j], v0, acc[r][0]);
                        acc[r][1] = fmaf(pr[j], v1, acc[r][1]);
                        acc[r][2] = fmaf(pr[j], v2, acc[r][2]);
                        acc[r][3] = fmaf(pr[j], v3, acc[r][3]);
                    }
                }
            }
            __syncwarp();
            ++consumed;
            // refill the stage just released with the next tile of this warp's stream
            if (issue_has_more()) issue_next();
        }

        // ---- finalize: direct bf16 output or fp32 partial for the combine pass
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float lt = warp_sum_f(l[r]);
            const int rr = U.rb * R + r;
            if (rr < rows) {
                const int64_t row = static_cast<int64_t>(qstart + rr / P.G) * P.Hq + U.kvh * P.G + rr % P.G;
                if (U.direct) {
                    const float inv = 1.f / lt;
                    const uint32_t lo = f32_to_bf16_rne(acc[r][0] * inv) | (static_cast<uint32_t>(f32_to_bf16_rne(acc[r][1] * inv)) << 16);
                    const uint32_t hi = f32_to_bf16_rne(acc[r][2] * inv) | (static_cast<uint32_t>(f32_to_bf16_rne(acc[r][3] * inv)) << 16);
                    *reinterpret_cast<uint2 *>(P.out + row * kHeadDim + d0) = make_uint2(lo, hi);
                } else {
                    const int64_t w = static_cast<int64_t>(U.slot) * P.n_rows_total + row;
                    *reinterpret_cast<float4 *>(P.ws_acc + w * kHeadDim + d0) =
                        make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
                    if (lane == 0) *reinterpret_cast<float2 *>(P.ws_ml + w * 2) = make_float2(m[r], lt);
                }
            }
        }
        __syncwarp();  // q buffer is rewritten by the next unit
    }
}

// One warp per output row (sequence b, query token i, head h): merge the
// partials of the shared-prefix runs and of the splits.
__global__ void __launch_bounds__(256) combine_kernel(const CombineParams P) {
    const int lane = threadIdx.x & 31;
    const int64_t w = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int h = static_cast<int>(w % P.Hq);
    const int64_t bi = w / P.Hq;
    const int i = static_cast<int>(bi % P.max_q_len);
    const int b = static_cast<int>(bi / P.max_q_len);
    if (b >= P.B) return;
    const int n = P.q_lens[b], T = P.seq_lens[b];
    if (i >= n || n > T || n > P.max_q_len) return;
    const int npages = (T + kPageSize - 1) / kPageSize;
    const int skip = P.skip_pages ? P.skip_pages[b] : 0;
    const int runs = P.run_slots ? P.run_slots[b] : 0;
    const int nsplit = npages > skip ? (npages - skip + P.pages_per_split - 1) / P.pages_per_split : 0;
    if (nsplit == 1 && runs == 0) return;  // written directly by the split kernel
    const int qstart = q_row_start(P.q_lens, b, lane);
    if (qstart + n > P.total_q) return;  // flagged by the split kernel
    const int64_t row = static_cast<int64_t>(qstart + i) * P.Hq + h;
    const int nslots = runs + nsplit;
    auto slot_of = [&](int k) { return k < runs ? k : P.slot_base + (k - runs); };

    float M = -INFINITY;
    for (int k = 0; k < nslots; ++k) {
        const float2 ml = *reinterpret_cast<const float2 *>(P.ws_ml + (static_cast<int64_t>(slot_of(k)) * P.n_rows_total + row) * 2);
        if (ml.y > 0.f) M = fmaxf(M, ml.x);
    }
    float L = 0.f;
    float4 o = make_float4(0, 0, 0, 0);
    for (int k = 0; k < nslots; ++k) {
        const int64_t wi = static_cast<int64_t>(slot_of(k)) * P.n_rows_total + row;
        const float2 ml = *reinterpret_cast<const float2 *>(P.ws_ml + wi * 2);
        if (!(ml.y > 0.f)) continue;
        const float sc = exp2f(ml.x - M);
        const float4 a = *reinterpret_cast<const float4 *>(P.ws_acc + wi * kHeadDim + lane * 4);
        L += ml.y * sc;
        o.x += a.x * sc;
        o.y += a.y * sc;
        o.z += a.z * sc;
        o.w += a.w * sc;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const uint32_t lo = f32_to_bf16_rne(o.x * inv) | (static_cast<uint32_t>(f32_to_bf16_rne(o.y * inv)) << 16);
    const uint32_t hi = f32_to_bf16_rne(o.z * inv) | (static_cast<uint32_t>(f32_to_bf16_rne(o.w * inv)) << 16);
    *reinterpret_cast<uint2 *>(P.out + row * kHeadDim + lane * 4) = make_uint2(lo, hi);
}

template <int R>
cudaError_t launch_r(const SplitParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                     int num_ctas, cudaStream_t stream) {
    const size_t smem = WarpLayout<R>::kBytes + 1024;
    cudaError_t e = cudaFuncSetAttribute(split_attn_kernel<R>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    split_attn_kernel<R><<<num_ctas, 32, smem, stream>>>(p, tk, tv);
    return cudaGetLastError();
}

template <int R>
cudaError_t occupancy_r(int *ctas_per_sm) {
    const size_t smem = WarpLayout<R>::kBytes + 1024;
    cudaError_t e = cudaFuncSetAttribute(split_attn_kernel<R>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, split_attn_kernel<R>, 32, smem);
}

}  // namespace

int max_rows_per_block() { return 16; }

size_t split_smem_bytes(int R, int) {
    switch (R) {
        case 4: return WarpLayout<4>::kBytes + 1024;
        case 8: return WarpLayout<8>::kBytes + 1024;
        case 12: return WarpLayout<12>::kBytes + 1024;
        default: return WarpLayout<16>::kBytes + 1024;
    }
}

cudaError_t split_occupancy(int R, int, int *ctas_per_sm) {
    switch (R) {
        case 4: return occupancy_r<4>(ctas_per_sm);
        case 8: return occupancy_r<8>(ctas_per_sm);
        case 12: return occupancy_r<12>(ctas_per_sm);
        case 16: return occupancy_r<16>(ctas_per_sm);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_split_attn(const SplitParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                              int num_ctas, int, cudaStream_t stream) {
    switch (p.rows_per_block) {
        case 4: return launch_r<4>(p, tk, tv, num_ctas, stream);
        case 8: return launch_r<8>(p, tk, tv, num_ctas, stream);
        case 12: return launch_r<12>(p, tk, tv, num_ctas, stream);
        case 16: return launch_r<16>(p, tk, tv, num_ctas, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_combine(const CombineParams &p, cudaStream_t stream) {
    const int64_t warps = static_cast<int64_t>(p.B) * p.max_q_len * p.Hq;
    if (warps == 0) return cudaSuccess;
    const int64_t blocks = (warps + 7) / 8;
    combine_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace sa
