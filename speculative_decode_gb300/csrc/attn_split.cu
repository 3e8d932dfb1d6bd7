// attn_split.cu -- page-streamed attention on the CUDA cores (split-K over
// pages) for decode (q_len = 1) and causal multi-query verification
// (q_len = k + 1).
//
// What it computes: for each sequence b, new query token i and query head h,
// softmax(scale * q . K_b^T) V_b over the keys at positions
// 0 .. seq_len - q_len + i, with K_b/V_b gathered through the block table
// (ExLlamaV2 "Dynamic Generator" page, "Continuous batching"; causal rows as
// in the Hugging Face "Assisted Generation" page, "How Assisted Generation
// works"). The softmax is evaluated online over 32-token tiles; the pages of a
// sequence are cut into splits whose partial (max, sum, accumulator) states
// are merged exactly, in this kernel, by whichever warp finishes a
// sequence's last split.
//
// Design (sm_103a):
//  * Work unit = (sequence, KV head, row block, split of `pages_per_split`
//    pages). Rows are the G query heads of the KV head times the sequence's
//    query tokens, so every K/V byte read serves all of them.
//  * One warp owns a unit from start to finish. Lane 0 streams the unit's
//    32-token K and V tiles with TMA (2-D tensor copies, 128-byte swizzle)
//    into the warp's private ring of S stages; warps claim units dynamically
//    from a global counter and keep copies of their next units in flight
//    while computing, across unit boundaries.
//  * Lane mapping: a token is handled by L = 2R lanes (8, 16 or 32), each
//    owning 128/L head dimensions, so the pre-scaled queries and the output
//    accumulators live in registers. Q.K partial dots are combined with a
//    shuffle reduce-scatter, after which each lane holds one (token, row)
//    score; P.V reuses the same mapping with p broadcast from shared memory.
//    Products use packed fp32x2 FMAs (bf16 inputs converted exactly).
//  * Every wait on a TMA barrier is bounded (common.cuh); on timeout the
//    warp flags SA_ERR_TIMEOUT, drains its copies in flight and leaves.
#include <cstdlib>

#include "common.cuh"

namespace sa {

namespace {

constexpr int kTile = 32;                     // tokens per stage
constexpr int kHalfBytes = kTile * 128;       // 32 rows x 64 bf16 (one 128-byte swizzle span)
constexpr int kStageBytes = 4 * kHalfBytes;   // K[0:64], K[64:128], V[0:64], V[64:128]
constexpr int kRing = 8;                      // claimed-unit FIFO depth per warp

template <int R>
struct Geo {
    static constexpr int L = R <= 4 ? 8 : (R <= 8 ? 16 : 32);  // lanes per token
    static constexpr int TG = 32 / L;                          // tokens per warp step
    static constexpr int NS = kTile / TG;                      // steps per tile
    static constexpr int NW = kHeadDim / L / 2;                // bf16x2 words per lane
};

template <int R, int S>
struct Layout {
    static constexpr int kPOff = S * kStageBytes;               // fp32 p [32][R]
    static constexpr int kRowOff = kPOff + kTile * R * 4;       // fp32 [2][R] row exchange
    static constexpr int kRingOff = kRowOff + 2 * R * 4;        // int32 [kRing]
    static constexpr int kBarOff = (kRingOff + kRing * 4 + 7) / 8 * 8;
    static constexpr int kBytes = (kBarOff + S * 8 + 1023) / 1024 * 1024;
};

struct Unit {
    int b, kvh, rb, T, n, qstart, t_lo, t_hi, n_tiles, slot, nsplit, runs;
    bool direct, ok;
};

__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Packed fp32x2 fused multiply-add: d = a * b + c elementwise, one rounding each.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    unsigned long long ra = *reinterpret_cast<unsigned long long *>(&a);
    unsigned long long rb = *reinterpret_cast<unsigned long long *>(&b);
    unsigned long long rc = *reinterpret_cast<unsigned long long *>(&c);
    unsigned long long rd;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
    return *reinterpret_cast<float2 *>(&rd);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t w) { return make_float2(bf16_lo(w), bf16_hi(w)); }

// Load this lane's bf16 words of row t from a swizzled two-half tile. Lane j
// of an L-lane token group owns: L=8 -> d 8j..8j+7 and 64+8j..64+8j+7;
// L=16 -> d 64(j/8)+8(j%8) .. +7; L=32 -> d 4j..4j+3. Each quarter-warp then
// touches eight distinct 16-byte chunks of the swizzle span (conflict-free).
template <int L>
__device__ __forceinline__ void load_tile_row(const uint8_t *tile, int t, int j, uint32_t (&w)[64 / L]) {
    if constexpr (L == 8) {
        const uint4 a = *reinterpret_cast<const uint4 *>(tile + sw128_offset(t, j));
        const uint4 b = *reinterpret_cast<const uint4 *>(tile + kHalfBytes + sw128_offset(t, j));
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
        w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
    } else if constexpr (L == 16) {
        const uint4 a = *reinterpret_cast<const uint4 *>(tile + (j >> 3) * kHalfBytes + sw128_offset(t, j & 7));
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    } else {
        const uint2 a = *reinterpret_cast<const uint2 *>(tile + (j >> 4) * kHalfBytes +
                                                         sw128_offset(t, (j & 15) >> 1) + (j & 1) * 8);
        w[0] = a.x; w[1] = a.y;
    }
}

// Element offset (within a 128-wide row) of this lane's word k.
template <int L>
__device__ __forceinline__ int lane_dim_of_word(int j, int k) {
    if constexpr (L == 8) return (k < 4 ? 8 * j : 64 + 8 * j) + 2 * (k & 3);
    else if constexpr (L == 16) return 64 * (j >> 3) + 8 * (j & 7) + 2 * k;
    else return 4 * j + 2 * k;
}

// Packed query rows that precede sequence b (sum of q_lens[0..b)).
__device__ __forceinline__ int q_row_start(const int32_t *q_lens, int b, int lane) {
    int s = 0;
    for (int k = lane; k < b; k += 32) s += q_lens[k];
    return warp_sum_i(s);
}

// Decode unit u (warp-uniform; every lane calls). Returns false when the
// unit has no work; U.ok = false when a page id is out of range.
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
    if (U.n <= 0) return false;
    if (U.n > U.T || U.n > P.max_q_len) {
        if (lane == 0) flag_error(P.err, kErrBitQlen);
        return false;
    }
    if (U.rb * R >= P.G * U.n) return false;
    const int npages = (U.T + kPageSize - 1) / kPageSize;
    const int skip = P.skip_pages ? P.skip_pages[U.b] : 0;
    const int p_lo = skip + split * P.pages_per_split;
    if (p_lo >= npages) return false;
    U.qstart = q_row_start(P.q_lens, U.b, lane);
    if (U.qstart + U.n > P.total_q) {  // q_lens disagree with dims.total_q
        if (lane == 0) flag_error(P.err, kErrBitQlen);
        return false;
    }
    const int p_hi = min(p_lo + P.pages_per_split, npages);
    U.t_lo = p_lo * kPageSize;
    U.t_hi = min(p_hi * kPageSize, U.T);
    U.n_tiles = (U.t_hi - U.t_lo + kTile - 1) / kTile;
    U.nsplit = (npages - skip + P.pages_per_split - 1) / P.pages_per_split;
    U.runs = P.run_slots ? P.run_slots[U.b] : 0;
    U.direct = (U.nsplit == 1 && U.runs == 0);
    U.slot = P.slot_base + split;
    bool ok = npages <= P.max_pages;
    for (int jp = p_lo + lane; ok && jp < p_hi; jp += 32) {
        const int id = P.block_table[static_cast<int64_t>(U.b) * P.max_pages + jp];
        ok = id >= 0 && id < P.num_pages;
    }
    U.ok = __all_sync(0xffffffffu, ok);
    return true;
}

__device__ __forceinline__ int64_t out_row(const SplitParams &P, const Unit &U, int rr) {
    return static_cast<int64_t>(U.qstart + rr / P.G) * P.Hq + U.kvh * P.G + rr % P.G;
}

// Merge every partial of rows [rb*R, rb*R + nvr) of (b, kvh): the slots of the
// shared-prefix runs and of the splits, with exact max-shifted rescaling.
__device__ void merge_rows(const SplitParams &P, const Unit &U, int R, int nvr, int lane) {
    const int nslots = U.runs + U.nsplit;
    for (int r = 0; r < nvr; ++r) {
        const int64_t row = out_row(P, U, U.rb * R + r);
        float M = -INFINITY;
        for (int k = 0; k < nslots; ++k) {
            const int slot = k < U.runs ? k : P.slot_base + (k - U.runs);
            const float2 ml = __ldcg(reinterpret_cast<const float2 *>(
                P.ws_ml + (static_cast<int64_t>(slot) * P.n_rows_total + row) * 2));
            if (ml.y > 0.f) M = fmaxf(M, ml.x);
        }
        float Lsum = 0.f;
        float4 o = make_float4(0, 0, 0, 0);
        for (int k = 0; k < nslots; ++k) {
            const int slot = k < U.runs ? k : P.slot_base + (k - U.runs);
            const int64_t wi = static_cast<int64_t>(slot) * P.n_rows_total + row;
            const float2 ml = __ldcg(reinterpret_cast<const float2 *>(P.ws_ml + wi * 2));
            if (!(ml.y > 0.f)) continue;
            const float sc = exp2f(ml.x - M);
            const float4 a = __ldcg(reinterpret_cast<const float4 *>(P.ws_acc + wi * kHeadDim + lane * 4));
            Lsum += ml.y * sc;
            o.x += a.x * sc;
            o.y += a.y * sc;
            o.z += a.z * sc;
            o.w += a.w * sc;
        }
        const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
        const uint32_t lo = f32_to_bf16_rne(o.x * inv) | (static_cast<uint32_t>(f32_to_bf16_rne(o.y * inv)) << 16);
        const uint32_t hi = f32_to_bf16_rne(o.z * inv) | (static_cast<uint32_t>(f32_to_bf16_rne(o.w * inv)) << 16);
        *reinterpret_cast<uint2 *>(P.out + row * kHeadDim + lane * 4) = make_uint2(lo, hi);
    }
}

// After a split's partial is stored: count it; the last split of (b, kvh,
// row block) merges all partials and resets the counter for the next call.
__device__ void count_and_merge(const SplitParams &P, const Unit &U, int R, int nvr, int lane) {
    __threadfence();
    __syncwarp();
    int last = 0;
    if (lane == 0) {
        int32_t *ctr = P.merge_ctr + (static_cast<int64_t>(U.b) * P.Hkv + U.kvh) * P.n_row_blocks + U.rb;
        last = atomicAdd(ctr, 1) == U.nsplit - 1;
        if (last) atomicExch(ctr, 0);
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __threadfence();
    merge_rows(P, U, R, nvr, lane);
}

template <int R, int S>
__global__ void __launch_bounds__(32) split_attn_kernel(const SplitParams P,
                                                        const __grid_constant__ CUtensorMap tmk,
                                                        const __grid_constant__ CUtensorMap tmv) {
    using Gm = Geo<R>;
    using Lay = Layout<R, S>;
    constexpr int L = Gm::L, TG = Gm::TG, NS = Gm::NS, NW = Gm::NW;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int lane = threadIdx.x & 31;
    const int tg = lane / L;   // token group
    const int j = lane % L;    // lane within the token group
    float(*pbuf)[R] = reinterpret_cast<float(*)[R]>(smem + Lay::kPOff);
    float *rowx = reinterpret_cast<float *>(smem + Lay::kRowOff);
    int32_t *ring = reinterpret_cast<int32_t *>(smem + Lay::kRingOff);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Lay::kBarOff);

    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
    }
    __syncwarp();

    // row of the reduce-scatter result this lane ends up holding
    int rj = 0;
    {
        int n = R;
#pragma unroll
        for (int o = L / 2; o >= 2; o >>= 1) {
            n >>= 1;
            if (j & o) rj += n;
        }
    }
    const uint64_t policy = P.evict_first ? l2_policy_evict_first() : l2_policy_evict_normal();

    // ---- issue side: claims units, pushes them to the ring, streams tiles
    uint32_t issued = 0, consumed = 0;
    int ring_head = 0, ring_tail = 0;   // pushed / popped unit counts
    bool exhausted = false;
    Unit IU;
    int itile = 0, intiles = 0;
    auto issue_next = [&]() -> bool {
        while (itile >= intiles) {
            if (exhausted || ring_head - ring_tail >= kRing) return false;
            int u = 0;
            if (lane == 0) u = atomicAdd(P.sched, 1);
            u = __shfl_sync(0xffffffffu, u, 0);
            if (u >= P.n_units) {
                exhausted = true;
                return false;
            }
            if (!decode_unit<R>(P, u, IU, lane)) continue;
            if (lane == 0) ring[ring_head % kRing] = u;
            ++ring_head;
            intiles = IU.ok ? IU.n_tiles : 0;
            itile = 0;
        }
        const int t0 = IU.t_lo + itile * kTile;
        const int pid = P.block_table[static_cast<int64_t>(IU.b) * P.max_pages + t0 / kPageSize];
        const int y = (pid * P.Hkv + IU.kvh) * kPageSize + (t0 % kPageSize);
        const int s = issued % S;
        if (lane == 0) {
            uint8_t *dst = smem + s * kStageBytes;
            mbar_arrive_expect_tx(&full[s], kStageBytes);
            tma_load_2d(dst, &tmk, &full[s], 0, y, policy);
            tma_load_2d(dst + kHalfBytes, &tmk, &full[s], 64, y, policy);
            tma_load_2d(dst + 2 * kHalfBytes, &tmv, &full[s], 0, y, policy);
            tma_load_2d(dst + 3 * kHalfBytes, &tmv, &full[s], 64, y, policy);
        }
        ++issued;
        ++itile;
        return true;
    };
    auto top_up = [&]() {
        while (issued - consumed < static_cast<uint32_t>(S) && issue_next()) {
        }
        __syncwarp();
    };

    top_up();
    while (true) {
        if (ring_tail == ring_head) top_up();
        if (ring_tail == ring_head) break;  // nothing claimed and nothing left
        const int u = ring[ring_tail % kRing];
        ++ring_tail;
        Unit U;
        decode_unit<R>(P, u, U, lane);
        const int rows = P.G * U.n;
        const int nvr = min(R, rows - U.rb * R);  // valid rows of this block

        if (!U.ok) {
            // pages out of range: report, leave an empty partial (or zeros)
            if (lane == 0) flag_error(P.err, kErrBitPageOOB);
            for (int r = 0; r < nvr; ++r) {
                const int64_t row = out_row(P, U, U.rb * R + r);
                if (U.direct) {
                    *reinterpret_cast<uint2 *>(P.out + row * kHeadDim + lane * 4) = make_uint2(0, 0);
                } else {
                    const int64_t w = static_cast<int64_t>(U.slot) * P.n_rows_total + row;
                    *reinterpret_cast<float4 *>(P.ws_acc + w * kHeadDim + lane * 4) = make_float4(0, 0, 0, 0);
                    if (lane == 0) *reinterpret_cast<float2 *>(P.ws_ml + w * 2) = make_float2(-INFINITY, 0.f);
                }
            }
            if (!U.direct) count_and_merge(P, U, R, nvr, lane);
            continue;
        }

        // ---- this lane's slice of the unit's queries, pre-scaled by scale*log2(e)
        float2 q2[R][NW];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int rr = U.rb * R + r;
#pragma unroll
            for (int k = 0; k < NW; ++k) q2[r][k] = make_float2(0.f, 0.f);
            if (r < nvr) {
                const uint16_t *qrow = P.q + out_row(P, U, rr) * kHeadDim;
#pragma unroll
                for (int k = 0; k < NW; ++k) {
                    const uint32_t w = *reinterpret_cast<const uint32_t *>(qrow + lane_dim_of_word<L>(j, k));
                    q2[r][k] = make_float2(bf16_lo(w) * P.qscale, bf16_hi(w) * P.qscale);
                }
            }
        }
        const int lim0 = U.T - U.n;                      // last key visible to query token 0
        const bool row_ok = rj < nvr;
        const int lim = row_ok ? lim0 + (U.rb * R + rj) / P.G : -1;
        float m = -INFINITY, lsum = 0.f;
        float2 acc[R][NW];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int k = 0; k < NW; ++k) acc[r][k] = make_float2(0.f, 0.f);

        for (int kt = 0; kt < U.n_tiles; ++kt) {
            top_up();
            const int s = consumed % S;
            const bool arrived = mbar_wait(&full[s], (consumed / S) & 1);
            if (!__all_sync(0xffffffffu, arrived)) {
                flag_error(P.err, kErrBitTimeout);
                for (uint32_t c = consumed + 1; c < issued; ++c) (void)mbar_wait(&full[c % S], (c / S) & 1);
                return;
            }
            const uint8_t *st = smem + s * kStageBytes;
            const int t0 = U.t_lo + kt * kTile;

            // ---- scores: partial dots over this lane's dims, reduce-scatter over L lanes
            float sv[NS];
#pragma unroll
            for (int step = 0; step < NS; ++step) {
                const int t = step * TG + tg;
                uint32_t kw[NW];
                load_tile_row<L>(st, t, j, kw);
                float2 a2[R];
#pragma unroll
                for (int r = 0; r < R; ++r) a2[r] = make_float2(0.f, 0.f);
#pragma unroll
                for (int k = 0; k < NW; ++k) {
                    const float2 kf = unpack_bf16x2(kw[k]);
#pragma unroll
                    for (int r = 0; r < R; ++r) a2[r] = ffma2(q2[r][k], kf, a2[r]);
                }
                float v[R];
#pragma unroll
                for (int r = 0; r < R; ++r) v[r] = a2[r].x + a2[r].y;
                int n = R;
#pragma unroll
                for (int o = L / 2; o >= 2; o >>= 1) {
                    const int h = n >> 1;
                    const bool up = (j & o) != 0;
#pragma unroll
                    for (int i = 0; i < h; ++i) {
                        const float send = up ? v[i] : v[i + h];
                        const float keep = up ? v[i + h] : v[i];
                        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                    }
                    n = h;
                }
                v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
                sv[step] = t0 + t <= lim ? v[0] : -INFINITY;
            }

            // ---- online softmax for this lane's row (log2 units)
            float tmax = -INFINITY;
#pragma unroll
            for (int step = 0; step < NS; ++step) tmax = fmaxf(tmax, sv[step]);
#pragma unroll
            for (int o = L; o < 32; o <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
            const float m_new = fmaxf(m, tmax);
            const float m_use = m_new == -INFINITY ? 0.f : m_new;
            const float alpha = exp2f(m - m_use);
            lsum *= alpha;
            m = m_new;
#pragma unroll
            for (int step = 0; step < NS; ++step) {
                const float p = exp2f(sv[step] - m_use);
                lsum += p;
                if ((j & 1) == 0) pbuf[step * TG + tg][rj] = p;
            }
            if (tg == 0 && (j & 1) == 0) rowx[rj] = alpha;
            __syncwarp();
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float a = rowx[r];
#pragma unroll
                    for (int k = 0; k < NW; ++k) acc[r][k] = make_float2(acc[r][k].x * a, acc[r][k].y * a);
                }
            }

            // ---- O += P V over the valid tokens of the tile
            const int nvalid = min(kTile, U.t_hi - t0);
#pragma unroll
            for (int step = 0; step < NS; ++step) {
                const int t = step * TG + tg;
                if (t < nvalid) {
                    uint32_t vw[NW];
                    load_tile_row<L>(st + 2 * kHalfBytes, t, j, vw);
                    float pr[R];
#pragma unroll
                    for (int r4 = 0; r4 < R / 4; ++r4) {
                        const float4 pp = *reinterpret_cast<const float4 *>(&pbuf[t][r4 * 4]);
                        pr[r4 * 4 + 0] = pp.x;
                        pr[r4 * 4 + 1] = pp.y;
                        pr[r4 * 4 + 2] = pp.z;
                        pr[r4 * 4 + 3] = pp.w;
                    }
#pragma unroll
                    for (int k = 0; k < NW; ++k) {
                        const float2 vf = unpack_bf16x2(vw[k]);
#pragma unroll
                        for (int r = 0; r < R; ++r) acc[r][k] = ffma2(make_float2(pr[r], pr[r]), vf, acc[r][k]);
                    }
                }
            }
            __syncwarp();   // stage and p buffer are reused by the next tile
            ++consumed;
        }

        // ---- finish the unit: sum over token groups, then output or partial
#pragma unroll
        for (int o = L; o < 32; o <<= 1) {
            lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int k = 0; k < NW; ++k) {
                    acc[r][k].x += __shfl_xor_sync(0xffffffffu, acc[r][k].x, o);
                    acc[r][k].y += __shfl_xor_sync(0xffffffffu, acc[r][k].y, o);
                }
        }
        if (tg == 0 && (j & 1) == 0) {
            rowx[rj] = m;
            rowx[R + rj] = lsum;
        }
        __syncwarp();
        if (tg == 0) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (r < nvr) {
                    const int64_t row = out_row(P, U, U.rb * R + r);
                    if (U.direct) {
                        const float inv = 1.f / rowx[R + r];
#pragma unroll
                        for (int k = 0; k < NW; ++k) {
                            const uint32_t w = f32_to_bf16_rne(acc[r][k].x * inv) |
                                               (static_cast<uint32_t>(f32_to_bf16_rne(acc[r][k].y * inv)) << 16);
                            *reinterpret_cast<uint32_t *>(P.out + row * kHeadDim + lane_dim_of_word<L>(j, k)) = w;
                        }
                    } else {
                        const int64_t wi = static_cast<int64_t>(U.slot) * P.n_rows_total + row;
#pragma unroll
                        for (int k = 0; k < NW; ++k)
                            *reinterpret_cast<float2 *>(P.ws_acc + wi * kHeadDim + lane_dim_of_word<L>(j, k)) = acc[r][k];
                        if (j == 0) *reinterpret_cast<float2 *>(P.ws_ml + wi * 2) = make_float2(rowx[r], rowx[R + r]);
                    }
                }
            }
        }
        if (!U.direct) count_and_merge(P, U, R, nvr, lane);
        __syncwarp();
    }

    // ---- last warp out resets the unit counter for the next call
    if (lane == 0) {
        __threadfence();
        if (atomicAdd(P.sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
            atomicExch(P.sched, 0);
            atomicExch(P.sched + 1, 0);
        }
    }
}

template <int R, int S>
constexpr size_t smem_bytes() { return Layout<R, S>::kBytes + 1024; }

template <int R, int S>
cudaError_t prepare() {
    static cudaError_t err = cudaFuncSetAttribute(split_attn_kernel<R, S>,
                                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  static_cast<int>(smem_bytes<R, S>()));
    return err;
}

template <int R, int S>
cudaError_t launch_rs(const SplitParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                      int num_ctas, cudaStream_t stream) {
    cudaError_t e = prepare<R, S>();
    if (e != cudaSuccess) return e;
    split_attn_kernel<R, S><<<num_ctas, 32, smem_bytes<R, S>(), stream>>>(p, tk, tv);
    return cudaGetLastError();
}

template <int R, int S>
cudaError_t occupancy_rs(int *ctas_per_sm) {
    cudaError_t e = prepare<R, S>();
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, split_attn_kernel<R, S>, 32,
                                                         smem_bytes<R, S>());
}

// Pipeline depth per warp (stages of 16 KiB). SA_SPLIT_STAGES=3 selects three.
int split_stages() {
    static const int s = [] {
        const char *v = std::getenv("SA_SPLIT_STAGES");
        return (v != nullptr && v[0] == '3') ? 3 : 2;
    }();
    return s;
}

}  // namespace

cudaError_t split_occupancy(int R, int, int *ctas_per_sm) {
    const bool s3 = split_stages() == 3;
    switch (R) {
        case 4: return s3 ? occupancy_rs<4, 3>(ctas_per_sm) : occupancy_rs<4, 2>(ctas_per_sm);
        case 8: return s3 ? occupancy_rs<8, 3>(ctas_per_sm) : occupancy_rs<8, 2>(ctas_per_sm);
        case 16: return s3 ? occupancy_rs<16, 3>(ctas_per_sm) : occupancy_rs<16, 2>(ctas_per_sm);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_split_attn(const SplitParams &p, const CUtensorMap &tk, const CUtensorMap &tv,
                              int num_ctas, int, cudaStream_t stream) {
    const bool s3 = split_stages() == 3;
    switch (p.rows_per_block) {
        case 4: return s3 ? launch_rs<4, 3>(p, tk, tv, num_ctas, stream) : launch_rs<4, 2>(p, tk, tv, num_ctas, stream);
        case 8: return s3 ? launch_rs<8, 3>(p, tk, tv, num_ctas, stream) : launch_rs<8, 2>(p, tk, tv, num_ctas, stream);
        case 16: return s3 ? launch_rs<16, 3>(p, tk, tv, num_ctas, stream) : launch_rs<16, 2>(p, tk, tv, num_ctas, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sa
