// attn_split.cu -- page-streamed attention on the CUDA cores for decode
// (q_len = 1) and causal multi-query verification (q_len = k + 1).
//
// What it computes: for each sequence b, new query token i and query head h,
// softmax(scale * q . K_b^T) V_b over the keys at positions
// 0 .. seq_len - q_len + i, with K_b/V_b gathered through the block table
// (ExLlamaV2 "Dynamic Generator" page, "Continuous batching"; causal rows as
// in the Hugging Face "Assisted Generation" page, "How Assisted Generation
// works"). The softmax is evaluated online over 32-token tiles; where a
// sequence's keys are cut into pieces, the partial (max, sum, accumulator)
// states are merged exactly, in this kernel, by whichever warp finishes the
// last piece.
//
// Design (sm_103a):
//  * Segment = (sequence, KV head, row block): the G query heads of the KV
//    head times the sequence's new tokens (up to R rows), so every K/V byte
//    read serves all of them. All segments' 32-token tiles form one sequence
//    of work that is cut into equal contiguous ranges, one per warp
//    (stream-K): perfectly balanced whatever the context lengths, with at
//    most two partial pieces per warp and no scheduling atomics.
//  * One warp owns its range. Lane 0 streams each tile's K rows and V rows
//    (each one contiguous run inside a page) with two 1-D bulk copies into
//    the warp's private ring of S stages, and bulk-copies each piece's query
//    rows ahead of use; all 32 lanes compute.
//  * Lane mapping: a token is handled by L = 2R lanes (8, 16 or 32), each
//    owning 128/L head dims, so pre-scaled queries and output accumulators
//    live in registers. Q.K partial dots are combined with a shuffle
//    reduce-scatter, after which each lane holds one (token, row) score; P.V
//    reuses the mapping with p broadcast from shared memory. Products use
//    packed fp32x2 FMAs on exactly converted bf16 inputs.
//  * A piece that is not a whole segment stores an fp32 partial and counts
//    itself with a release atomic whose result is examined one piece later,
//    so the round trip is hidden; the last piece merges.
//  * Every wait on a barrier is bounded (common.cuh); on timeout the warp
//    flags SA_ERR_TIMEOUT, drains its copies in flight and leaves.
#include "common.cuh"

namespace sa {

namespace {

// Tuning constants (measured on GB300: 16-token tiles, two stages per warp and
// 2R lanes per token were fastest for the decode batch).
#ifndef SA_SPLIT_TILE
#define SA_SPLIT_TILE 16
#endif
#ifndef SA_SPLIT_MIN_WARPS
#define SA_SPLIT_MIN_WARPS 1
#endif
constexpr int kTile = SA_SPLIT_TILE;          // tokens per stage (16 or 32)
constexpr int kRowBytes = kHeadDim * 2;       // one K or V row: 256 bytes
constexpr int kKVBytes = kTile * kRowBytes;   // K (or V) rows of one tile, contiguous in a page
constexpr int kStageBytes = 2 * kKVBytes;     // K tile, then V tile
#ifndef SA_SPLIT_STAGES
#define SA_SPLIT_STAGES 2
#endif
constexpr int kStages = SA_SPLIT_STAGES;      // pipeline depth per warp
constexpr int kRing = kStages + 2;            // piece descriptors in flight (>= kStages + 1)
constexpr int kPieceInts = 16;

#ifndef SA_SPLIT_LPT
#define SA_SPLIT_LPT 2
#endif
template <int R>
struct Geo {
    static constexpr int L = SA_SPLIT_LPT * R < 32 ? SA_SPLIT_LPT * R : 32;  // lanes per token
    static constexpr int DUP = L / R;                          // lanes holding each row's score
    static constexpr int TG = 32 / L;                          // tokens per warp step
    static constexpr int NS = kTile / TG;                      // steps per tile
    static constexpr int NW = kHeadDim / L / 2;                // bf16x2 words per lane
};

template <int R>
struct Layout {
    static constexpr int kQOff = kStages * kStageBytes;                  // bf16 q [S][R][128]
    static constexpr int kPOff = kQOff + kStages * R * kHeadDim * 2;     // fp32 p [32][R]
    static constexpr int kRowOff = kPOff + kTile * R * 4;                // fp32 [2][R]
    static constexpr int kRingOff = kRowOff + 2 * R * 4;                 // int32 [kRing][16]
    static constexpr int kFlagOff = kRingOff + kRing * kPieceInts * 4;   // int32 [kStages] tile loaded?
    static constexpr int kBarOff = (kFlagOff + kStages * 4 + 7) / 8 * 8;  // uint64 [2][kStages]
    static constexpr int kBytes = (kBarOff + 2 * kStages * 8 + 1023) / 1024 * 1024;
};

// A piece: the part of one segment inside this warp's range.
struct Piece {
    int b, kvh, rb, T, n, qstart, t_lo, n_tiles, piece, pieces, nvr, runs;
};

struct SeqInfo {
    int T, n, skip_tok, tiles, nrb, runs;
};

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    unsigned long long ra = *reinterpret_cast<unsigned long long *>(&a);
    unsigned long long rb = *reinterpret_cast<unsigned long long *>(&b);
    unsigned long long rc = *reinterpret_cast<unsigned long long *>(&c);
    unsigned long long rd;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
    return *reinterpret_cast<float2 *>(&rd);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t w) { return make_float2(bf16_lo(w), bf16_hi(w)); }

// Load this lane's bf16 words of row t of a tile held as plain 256-byte rows.
// Lane j of an L-lane token group owns: L=8 -> d 8j..8j+7 and 64+8j..64+8j+7;
// L=16 -> d 8j..8j+7; L=32 -> d 4j..4j+3. The lanes of a token group read
// consecutive 16-byte (8-byte) pieces of one row, so each quarter-warp touches
// one 128-byte span: no bank conflicts.
template <int L>
__device__ __forceinline__ void load_tile_row(const uint8_t *tile, int t, int j, uint32_t (&w)[64 / L]) {
    const uint8_t *row = tile + t * kRowBytes;
    if constexpr (L == 8) {
        const uint4 a = *reinterpret_cast<const uint4 *>(row + j * 16);
        const uint4 b = *reinterpret_cast<const uint4 *>(row + 128 + j * 16);
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
        w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
    } else if constexpr (L == 16) {
        const uint4 a = *reinterpret_cast<const uint4 *>(row + j * 16);
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    } else {
        const uint2 a = *reinterpret_cast<const uint2 *>(row + j * 8);
        w[0] = a.x; w[1] = a.y;
    }
}

// Element offset (within a 128-wide row) of this lane's word k.
template <int L>
__device__ __forceinline__ int lane_dim_of_word(int j, int k) {
    if constexpr (L == 8) return (k < 4 ? 8 * j : 64 + 8 * j) + 2 * (k & 3);
    else if constexpr (L == 16) return 8 * j + 2 * k;
    else return 4 * j + 2 * k;
}

__device__ __forceinline__ int64_t out_row(const SplitParams &P, const Piece &U, int rr) {
    return static_cast<int64_t>(U.qstart + rr / P.G) * P.Hq + U.kvh * P.G + rr % P.G;
}

// Per-sequence shape of the work; tiles = 0 when the sequence has none.
template <int R>
__device__ __forceinline__ SeqInfo seq_info(const SplitParams &P, int b, int qstart, bool flag) {
    SeqInfo s;
    s.T = P.seq_lens[b];
    s.n = P.q_lens[b];
    s.tiles = 0;
    s.nrb = 0;
    s.skip_tok = 0;
    s.runs = 0;
    if (s.n <= 0) return s;
    const int npages = (s.T + kPageSize - 1) / kPageSize;
    if (s.n > s.T || s.n > P.max_q_len || qstart + s.n > P.total_q || npages > P.max_pages) {
        if (flag) flag_error(P.err, kErrBitQlen);
        return s;
    }
    int skip = P.skip_pages ? P.skip_pages[b] : 0;
    int runs = P.run_slots ? P.run_slots[b] : 0;
    if (P.tc_min_rows > 0 && P.G * s.n >= P.tc_min_rows) {  // attended on the tensor cores
        skip = npages;
        runs = (npages + P.tc_chunk_pages - 1) / P.tc_chunk_pages;
    }
    s.runs = runs;
    s.skip_tok = skip * kPageSize;
    const int keys = s.T - s.skip_tok;
    s.tiles = keys > 0 ? (keys + kTile - 1) / kTile : (runs > 0 ? 1 : 0);  // one empty tile carries the merge
    s.nrb = (P.G * s.n + R - 1) / R;
    return s;
}

__device__ __forceinline__ int64_t seq_work(const SplitParams &P, const SeqInfo &s) {
    return static_cast<int64_t>(s.tiles) * P.Hkv * s.nrb;
}

// Merge every partial of the piece's rows: the tensor-core runs' slots and the
// pieces' slots, with exact max-shifted rescaling. Eight lanes per row (16
// head dims each), four rows at a time, every load of a row's slots in flight
// together so the merge costs about two memory round trips per four rows.
constexpr int kMaxMergeSlots = 16;

__device__ __forceinline__ const float *ws_slot_row(const SplitParams &P, const Piece &U, int k, int64_t row,
                                                    const float *base, int width) {
    const int slot = k < U.runs ? k : P.slot_base + (k - U.runs);
    return base + (static_cast<int64_t>(slot) * P.n_rows_total + row) * width;
}

__device__ void merge_rows(const SplitParams &P, const Piece &U, int R, int lane) {
    const int nslots = U.runs + U.pieces;
    const int sub = lane & 7;
    for (int r0 = 0; r0 < U.nvr; r0 += 4) {
        const int r = r0 + (lane >> 3);
        if (r >= U.nvr) continue;
        const int64_t row = out_row(P, U, U.rb * R + r);
        float ms[kMaxMergeSlots], ls[kMaxMergeSlots];
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < kMaxMergeSlots; ++k) {
            ms[k] = -INFINITY;
            ls[k] = 0.f;
            if (k < nslots) {
                const float2 ml = __ldcg(reinterpret_cast<const float2 *>(ws_slot_row(P, U, k, row, P.ws_ml, 2)));
                ms[k] = ml.x;
                ls[k] = ml.y;
            }
        }
#pragma unroll
        for (int k = 0; k < kMaxMergeSlots; ++k)
            if (ls[k] > 0.f) M = fmaxf(M, ms[k]);
        float Lsum = 0.f;
        float4 o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) o[q] = make_float4(0, 0, 0, 0);
#pragma unroll
        for (int k = 0; k < kMaxMergeSlots; ++k) {
            if (ls[k] > 0.f) {
                const float w = exp2f(ms[k] - M);
                Lsum += ls[k] * w;
                const float4 *a = reinterpret_cast<const float4 *>(ws_slot_row(P, U, k, row, P.ws_acc, kHeadDim) + sub * 16);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 v = __ldcg(a + q);
                    o[q].x += v.x * w;
                    o[q].y += v.y * w;
                    o[q].z += v.z * w;
                    o[q].w += v.w * w;
                }
            }
        }
        const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
        uint32_t wv[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            wv[2 * q] = f32_to_bf16_rne(o[q].x * inv) | (static_cast<uint32_t>(f32_to_bf16_rne(o[q].y * inv)) << 16);
            wv[2 * q + 1] = f32_to_bf16_rne(o[q].z * inv) | (static_cast<uint32_t>(f32_to_bf16_rne(o[q].w * inv)) << 16);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(P.out + row * kHeadDim + sub * 16);
        dst[0] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        dst[1] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
    }
}

__device__ __forceinline__ int32_t *merge_counter(const SplitParams &P, const Piece &U) {
    return P.merge_ctr + (static_cast<int64_t>(U.b) * P.Hkv + U.kvh) * P.n_row_blocks + U.rb;
}

// A counted piece whose atomic result is examined later.
struct Pending {
    Piece U;
    int old;
    bool live;
};

__device__ void resolve(const SplitParams &P, Pending &pd, int R, int lane) {
    if (!pd.live) return;
    pd.live = false;
    const int old = __shfl_sync(0xffffffffu, pd.old, 0);
    if (old != pd.U.pieces - 1) return;
    asm volatile("fence.acq_rel.gpu;" ::: "memory");  // acquire: every other piece's partial is visible
    merge_rows(P, pd.U, R, lane);
    if (lane == 0) atomicExch(merge_counter(P, pd.U), 0);
}

template <int R>
__global__ void __launch_bounds__(32, SA_SPLIT_MIN_WARPS) split_attn_kernel(const SplitParams P) {
    using Gm = Geo<R>;
    using Lay = Layout<R>;
    constexpr int L = Gm::L, TG = Gm::TG, NS = Gm::NS, NW = Gm::NW, DUP = Gm::DUP;
    constexpr int S = kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int lane = threadIdx.x & 31;
    const int tg = lane / L;   // token group
    const int j = lane % L;    // lane within the token group
    uint16_t *qbuf = reinterpret_cast<uint16_t *>(smem + Lay::kQOff);
    float(*pbuf)[R] = reinterpret_cast<float(*)[R]>(smem + Lay::kPOff);
    float *rowx = reinterpret_cast<float *>(smem + Lay::kRowOff);
    int32_t *ring = reinterpret_cast<int32_t *>(smem + Lay::kRingOff);
    int32_t *stage_ok = reinterpret_cast<int32_t *>(smem + Lay::kFlagOff);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Lay::kBarOff);
    uint64_t *qfull = full + S;

    if (lane == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&qfull[s], 1);
        }
        fence_barrier_init();
    }

    // ---- 1. total work and this warp's range [g_begin, g_end) of tiles
    // lanes take contiguous chunks of sequences; two passes: query offsets, then work
    const int per = (P.B + 31) / 32;
    const int c_lo = min(P.B, lane * per), c_hi = min(P.B, c_lo + per);
    int cq = 0;
    for (int b = c_lo; b < c_hi; ++b) cq += max(0, P.q_lens[b]);
    int q_pre = cq;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, q_pre, o);
        if (lane >= o) q_pre += v;
    }
    q_pre -= cq;  // exclusive
    int64_t cw = 0;
    int max_tiles = 0;  // longest segment, in tiles
    {
        int qs = q_pre;
        for (int b = c_lo; b < c_hi; ++b) {
            const SeqInfo si = seq_info<R>(P, b, qs, true);
            cw += seq_work(P, si);
            max_tiles = max(max_tiles, si.tiles);
            qs += max(0, si.n);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) max_tiles = max(max_tiles, __shfl_xor_sync(0xffffffffu, max_tiles, o));
    int64_t w_pre = cw;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t v = __shfl_up_sync(0xffffffffu, w_pre, o);
        if (lane >= o) w_pre += v;
    }
    const int64_t total = __shfl_sync(0xffffffffu, w_pre, 31);
    w_pre -= cw;
    const int64_t W = gridDim.x;
    // a segment of s tiles spans at most ceil(s / C) + 1 ranges: C is at least
    // ceil(longest / (slots - 1)) so that no segment has more pieces than the
    // workspace has partial slots
    const int64_t C_min = P.piece_slots > 1 ? (max_tiles + P.piece_slots - 2) / (P.piece_slots - 1) : max_tiles;
    const int64_t C = max((total + W - 1) / W, max(C_min, int64_t{1}));
    const int64_t g_begin = static_cast<int64_t>(blockIdx.x) * C;
    const int64_t g_end = min(total, g_begin + C);
    __syncwarp();
    if (g_begin >= g_end) return;

    // ---- 2. locate the first tile: sequence, segment, tile within segment
    int b0 = 0, q0 = 0;
    int64_t ws0 = 0;
    {
        const bool mine = cw > 0 && w_pre <= g_begin && g_begin < w_pre + cw;
        const int src = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
        if (lane == src) {
            int64_t pos = w_pre;
            int qs = q_pre;
            int b = c_lo;
            for (; b < c_hi; ++b) {
                const SeqInfo si = seq_info<R>(P, b, qs, false);
                const int64_t wb = seq_work(P, si);
                if (g_begin < pos + wb) break;
                pos += wb;
                qs += max(0, si.n);
            }
            b0 = b;
            q0 = qs;
            ws0 = pos;
        }
        b0 = __shfl_sync(0xffffffffu, b0, src);
        q0 = __shfl_sync(0xffffffffu, q0, src);
        ws0 = __shfl_sync(0xffffffffu, ws0, src);
    }

    // row of the reduce-scatter result this lane ends up holding
    int rj = 0;
    {
        int n = R;
#pragma unroll
        for (int o = L / 2; o >= 1; o >>= 1) {
            if (n > 1) {
                n >>= 1;
                if (j & o) rj += n;
            }
        }
    }
    const bool row_writer = (j % DUP) == 0;  // one of the DUP lanes that hold row rj
    const uint64_t policy = P.evict_first ? l2_policy_evict_first() : l2_policy_evict_normal();

    // ---- issue cursor: walks tiles g_begin .. g_end-1 ahead of the consumer
    int ib = b0, iq = q0;
    int64_t iws = ws0;
    SeqInfo isi = seq_info<R>(P, ib, iq, false);
    int64_t ig = g_begin;
    int iseg, itile, ikvh, irb;
    {
        const int64_t off = g_begin - iws;
        iseg = static_cast<int>(off / isi.tiles);
        itile = static_cast<int>(off % isi.tiles);
        ikvh = iseg / isi.nrb;
        irb = iseg % isi.nrb;
    }
    uint32_t issued = 0, consumed = 0, pieces_pushed = 0;
    // physical page of the issue cursor's current logical page, and the next
    // page's id loaded one page ahead so the block-table read never stalls a tile
    int pg_b = -1, pg_j = -1, pg_id = -1, pg_next = -1;
    auto page_id = [&](int b, int jp, int npages) -> int {
        if (b == pg_b && jp == pg_j) return pg_id;
        const int64_t base = static_cast<int64_t>(b) * P.max_pages;
        pg_id = (b == pg_b && jp == pg_j + 1) ? pg_next : P.block_table[base + jp];
        pg_b = b;
        pg_j = jp;
        pg_next = jp + 1 < npages ? P.block_table[base + jp + 1] : -1;
        return pg_id;
    };
    auto issue_next = [&]() -> bool {
        if (ig >= g_end) return false;
        if (itile == isi.tiles) {  // next segment
            itile = 0;
            ++iseg;
            if (++irb == isi.nrb) {
                irb = 0;
                ++ikvh;
            }
            if (iseg == P.Hkv * isi.nrb) {  // next sequence with work
                iseg = 0;
                ikvh = 0;
                irb = 0;
                do {
                    iws += seq_work(P, isi);
                    iq += max(0, isi.n);
                    if (++ib >= P.B) return false;  // unreachable while ig < g_end
                    isi = seq_info<R>(P, ib, iq, false);
                } while (seq_work(P, isi) == 0);
            }
        }
        const int kvh = ikvh, rb = irb;
        if (ig == g_begin || itile == 0) {
            // a new piece: describe it for the consumer and fetch its query rows
            const int64_t seg0 = iws + static_cast<int64_t>(iseg) * isi.tiles;
            const int64_t seg1 = seg0 + isi.tiles;
            const int first = static_cast<int>(seg0 / C), last = static_cast<int>((seg1 - 1) / C);
            const int nvr = min(R, P.G * isi.n - rb * R);
            const int qs = pieces_pushed % S;
            if (lane == 0) {
                int32_t *d = ring + (pieces_pushed % kRing) * kPieceInts;
                d[0] = ib; d[1] = kvh; d[2] = rb; d[3] = isi.T; d[4] = isi.n; d[5] = iq;
                d[6] = isi.skip_tok + itile * kTile;
                d[7] = static_cast<int>(min(seg1, g_end) - ig);
                d[8] = static_cast<int>(blockIdx.x) - first;
                d[9] = last - first + 1;
                d[10] = nvr;
                d[11] = isi.runs;
                mbar_arrive_expect_tx(&qfull[qs], nvr * kHeadDim * 2);
                const int r0 = rb * R;
                for (int i = r0 / P.G; i <= (r0 + nvr - 1) / P.G; ++i) {
                    const int lo = max(r0, i * P.G), hi = min(r0 + nvr, (i + 1) * P.G);
                    const uint16_t *src = P.q + (static_cast<int64_t>(iq + i) * P.Hq + kvh * P.G + (lo - i * P.G)) * kHeadDim;
                    bulk_load(qbuf + (qs * R + (lo - r0)) * kHeadDim, src, (hi - lo) * kHeadDim * 2, &qfull[qs]);
                }
            }
            ++pieces_pushed;
        }
        // the tile: K and V rows [t0, t0 + 32) of KV head kvh
        const int t0 = isi.skip_tok + itile * kTile;
        const int s = issued % S;
        const int pid = t0 < isi.T ? page_id(ib, t0 / kPageSize, (isi.T + kPageSize - 1) / kPageSize) : -1;
        const bool ok = pid >= 0 && pid < P.num_pages;
        if (t0 < isi.T && !ok && lane == 0) flag_error(P.err, kErrBitPageOOB);
        if (lane == 0) {
            stage_ok[s] = ok;
            if (ok) {
                // the tile's K rows and V rows are each one contiguous run in the page
                const int64_t row = static_cast<int64_t>(pid * P.Hkv + kvh) * kPageSize + (t0 % kPageSize);
                uint8_t *dst = smem + s * kStageBytes;
                mbar_arrive_expect_tx(&full[s], kStageBytes);
                bulk_load_hint(dst, P.k_pages + row * kHeadDim, kKVBytes, &full[s], policy);
                bulk_load_hint(dst + kKVBytes, P.v_pages + row * kHeadDim, kKVBytes, &full[s], policy);
            } else {
                mbar_arrive(&full[s]);  // nothing to load: the consumer skips this tile
            }
        }
        ++issued;
        ++itile;
        ++ig;
        return true;
    };
    auto top_up = [&]() {
        while (issued - consumed < static_cast<uint32_t>(S) && issue_next()) {
        }
        __syncwarp();
    };
    uint32_t pieces_done = 0;
    auto bail_out = [&]() {
        flag_error(P.err, kErrBitTimeout);
        for (uint32_t c = consumed; c < issued; ++c) (void)mbar_wait(&full[c % S], (c / S) & 1);
        for (uint32_t c = pieces_done; c < pieces_pushed; ++c) (void)mbar_wait(&qfull[c % S], (c / S) & 1);
    };

    Pending pend;
    pend.live = false;
    pend.old = 0;
    top_up();
    while (consumed < issued) {
        Piece U;
        {
            const int32_t *d = ring + (pieces_done % kRing) * kPieceInts;
            U.b = d[0]; U.kvh = d[1]; U.rb = d[2]; U.T = d[3]; U.n = d[4]; U.qstart = d[5];
            U.t_lo = d[6]; U.n_tiles = d[7]; U.piece = d[8]; U.pieces = d[9]; U.nvr = d[10]; U.runs = d[11];
        }
        const bool direct = U.pieces == 1 && U.runs == 0;

        // ---- this piece's queries: bf16 rows in shared memory -> fp32 registers, scaled
        const int qs = pieces_done % S;
        if (!__all_sync(0xffffffffu, mbar_wait(&qfull[qs], (pieces_done / S) & 1))) {
            bail_out();
            return;
        }
        float2 q2[R][NW];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint16_t *qrow = qbuf + (qs * R + r) * kHeadDim;
#pragma unroll
            for (int k = 0; k < NW; ++k) {
                const uint32_t w = r < U.nvr ? *reinterpret_cast<const uint32_t *>(qrow + lane_dim_of_word<L>(j, k)) : 0u;
                q2[r][k] = make_float2(bf16_lo(w) * P.qscale, bf16_hi(w) * P.qscale);
            }
        }
        __syncwarp();
        ++pieces_done;
        const int lim = rj < U.nvr ? U.T - U.n + (U.rb * R + rj) / P.G : -1;  // last key of this lane's row
        float m = -INFINITY, lsum = 0.f;
        float2 acc[R][NW];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int k = 0; k < NW; ++k) acc[r][k] = make_float2(0.f, 0.f);

        for (int kt = 0; kt < U.n_tiles; ++kt) {
            top_up();
            const int s = consumed % S;
            if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (consumed / S) & 1))) {
                bail_out();
                return;
            }
            const uint8_t *st = smem + s * kStageBytes;
            const int t0 = U.t_lo + kt * kTile;
            if (stage_ok[s]) {
                // ---- scores: partial dots over this lane's dims for a batch of
                // steps, then the reduce-scatter over L lanes level by level across
                // the batch, so that independent shuffles overlap
                float sv[NS];
                constexpr int NB = (32 / R) < NS ? (32 / R) : NS;  // steps per batch
#pragma unroll
                for (int b0 = 0; b0 < NS; b0 += NB) {
                    float v[NB][R];
#pragma unroll
                    for (int bi = 0; bi < NB; ++bi) {
                        const int t = (b0 + bi) * TG + tg;
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
#pragma unroll
                        for (int r = 0; r < R; ++r) v[bi][r] = a2[r].x + a2[r].y;
                    }
                    // halve the values while more than one is left, then all-reduce
                    int n = R;
#pragma unroll
                    for (int o = L / 2; o >= 1; o >>= 1) {
                        if (n > 1) {
                            const int h = n >> 1;
                            const bool up = (j & o) != 0;
#pragma unroll
                            for (int bi = 0; bi < NB; ++bi)
#pragma unroll
                                for (int i = 0; i < h; ++i) {
                                    const float send = up ? v[bi][i] : v[bi][i + h];
                                    const float keep = up ? v[bi][i + h] : v[bi][i];
                                    v[bi][i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                                }
                            n = h;
                        } else {
#pragma unroll
                            for (int bi = 0; bi < NB; ++bi) v[bi][0] += __shfl_xor_sync(0xffffffffu, v[bi][0], o);
                        }
                    }
#pragma unroll
                    for (int bi = 0; bi < NB; ++bi) {
                        const int t = (b0 + bi) * TG + tg;
                        sv[b0 + bi] = t0 + t <= lim ? v[bi][0] : -INFINITY;
                    }
                }

                // ---- online softmax for this lane's row (log2 units)
                float tmax = -INFINITY;
#pragma unroll
                for (int step = 0; step < NS; ++step) tmax = fmaxf(tmax, sv[step]);
#pragma unroll
                for (int o = L; o < 32; o <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
                // the reference max m only moves when the tile max exceeds it by
                // more than 2^8, so p stays below 256 and the accumulators are
                // rescaled a few times per segment instead of on most tiles
                const bool grow = tmax > m + 8.f;
                const float m_new = grow ? tmax : m;
                const float alpha = grow ? exp2f(m - m_new) : 1.f;  // 0 when m was -inf
                const float m_use = m_new == -INFINITY ? 0.f : m_new;
                lsum *= alpha;
                m = m_new;
#pragma unroll
                for (int step = 0; step < NS; ++step) {
                    const float p = exp2f(sv[step] - m_use);
                    lsum += p;
                    if (row_writer) pbuf[step * TG + tg][rj] = p;
                }
                if (__any_sync(0xffffffffu, grow)) {
                    if (tg == 0 && row_writer) rowx[rj] = alpha;
                    __syncwarp();
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const float a = rowx[r];
#pragma unroll
                        for (int k = 0; k < NW; ++k) acc[r][k] = make_float2(acc[r][k].x * a, acc[r][k].y * a);
                    }
                }
                __syncwarp();  // p visible to the whole warp

                // ---- O += P V over the valid tokens of the tile
                const int nvalid = min(kTile, U.T - t0);
#pragma unroll
                for (int step = 0; step < NS; ++step) {
                    const int t = step * TG + tg;
                    if (t < nvalid) {
                        uint32_t vw[NW];
                        load_tile_row<L>(st + kKVBytes, t, j, vw);
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
            }
            __syncwarp();   // stage and p buffer are reused by later tiles
            ++consumed;
        }

        // ---- finish the piece: sum over token groups, then output or partial
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
        if (tg == 0 && row_writer) {
            rowx[rj] = m;
            rowx[R + rj] = lsum;
        }
        __syncwarp();
        if (tg == 0) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (r < U.nvr) {
                    const int64_t row = out_row(P, U, U.rb * R + r);
                    if (direct) {
                        const float inv = 1.f / rowx[R + r];
#pragma unroll
                        for (int k = 0; k < NW; ++k) {
                            const uint32_t w = f32_to_bf16_rne(acc[r][k].x * inv) |
                                               (static_cast<uint32_t>(f32_to_bf16_rne(acc[r][k].y * inv)) << 16);
                            *reinterpret_cast<uint32_t *>(P.out + row * kHeadDim + lane_dim_of_word<L>(j, k)) = w;
                        }
                    } else {
                        const int64_t wi = static_cast<int64_t>(P.slot_base + U.piece) * P.n_rows_total + row;
#pragma unroll
                        for (int k = 0; k < NW; ++k)
                            *reinterpret_cast<float2 *>(P.ws_acc + wi * kHeadDim + lane_dim_of_word<L>(j, k)) = acc[r][k];
                        if (j == 0) *reinterpret_cast<float2 *>(P.ws_ml + wi * 2) = make_float2(rowx[r], rowx[R + r]);
                    }
                }
            }
        }
        __syncwarp();
        resolve(P, pend, R, lane);  // the previous piece's count has long returned
        if (!direct) {
            pend.U = U;
            pend.live = true;
            if (lane == 0) pend.old = atomic_add_release(merge_counter(P, U), 1);
        }
    }
    resolve(P, pend, R, lane);
}

template <int R>
constexpr size_t smem_bytes() { return Layout<R>::kBytes + 1024; }

template <int R>
cudaError_t prepare() {
    static cudaError_t err = cudaFuncSetAttribute(split_attn_kernel<R>,
                                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  static_cast<int>(smem_bytes<R>()));
    return err;
}

template <int R>
cudaError_t launch_r(const SplitParams &p, int num_ctas, cudaStream_t stream) {
    cudaError_t e = prepare<R>();
    if (e != cudaSuccess) return e;
    split_attn_kernel<R><<<num_ctas, 32, smem_bytes<R>(), stream>>>(p);
    return cudaGetLastError();
}

template <int R>
cudaError_t occupancy_r(int *ctas_per_sm) {
    cudaError_t e = prepare<R>();
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, split_attn_kernel<R>, 32,
                                                         smem_bytes<R>());
}

}  // namespace

int split_tile_tokens() { return kTile; }

cudaError_t split_occupancy(int R, int, int *ctas_per_sm) {
    switch (R) {
        case 4: return occupancy_r<4>(ctas_per_sm);
        case 8: return occupancy_r<8>(ctas_per_sm);
        case 16: return occupancy_r<16>(ctas_per_sm);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_split_attn(const SplitParams &p, int num_ctas, cudaStream_t stream) {
    switch (p.rows_per_block) {
        case 4: return launch_r<4>(p, num_ctas, stream);
        case 8: return launch_r<8>(p, num_ctas, stream);
        case 16: return launch_r<16>(p, num_ctas, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sa
