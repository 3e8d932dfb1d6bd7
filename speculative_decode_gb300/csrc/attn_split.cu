// attn_split.cu -- page-streamed attention on the CUDA cores for decode
// (q_len = 1) and causal multi-query verification (q_len = k + 1).
//
// What it computes: for each sequence b, new query token i and query head h,
// softmax(scale * q . K_b^T) V_b over the keys at positions
// 0 .. seq_len - q_len + i, with K_b/V_b gathered through the block table
// (ExLlamaV2 "Dynamic Generator" page, "Continuous batching"; causal rows as
// in the Hugging Face "Assisted Generation" page, "How Assisted Generation
// works"). The softmax is evaluated online over 16-token tiles; where a
// sequence's keys are cut into pieces, the partial (max, sum, accumulator)
// states are merged exactly by a combine pass, a second kernel.
//
// Design (sm_103a):
//  * Segment = (sequence, KV head, row block): the G query heads of the KV
//    head times the sequence's new tokens (up to R rows), so every K/V byte
//    read serves all of them. All segments' 16-token tiles form one sequence
//    of work that is cut into equal contiguous ranges, one per warp
//    (stream-K): perfectly balanced whatever the context lengths, with at
//    most two partial pieces per warp and no scheduling atomics.
//  * One warp owns its range. It streams each tile's K rows and V rows (each
//    one contiguous run inside a page) into its private ring of S stages with
//    two 1-D bulk copies issued by lanes 0 and 1 in one instruction, and
//    bulk-copies each piece's query rows ahead of use; all 32 lanes compute.
//  * int8 and int4 pages (KB = 8 and 4 instances): the same kernel over codes
//    with one fp32 scale per (page, head, token) row; lanes 2 and 3 also copy
//    the tile's K and V scales, the loops run on codes converted exactly to
//    floats, and the row scales multiply the scores (K) and the
//    probabilities (V).
//  * Lane mapping: a token is handled by L = 2R lanes (8, 16 or 32), each
//    owning 128/L head dims, so pre-scaled queries and output accumulators
//    live in registers. Q.K partial dots are combined with a shuffle
//    reduce-scatter, after which each lane holds one (token, row) score; P.V
//    reuses the mapping with p broadcast from shared memory. Products use
//    packed fp32x2 FMAs on exactly converted bf16 inputs.
//  * A piece that is not a whole segment stores an fp32 partial; nothing in
//    the split kernel waits on another warp. The combine kernel, launched as
//    a programmatic dependent, repeats the (cheap) work scan while the split
//    kernel runs, waits for the grid, and merges each cut segment's partials
//    (and the tensor-core kernels' partials) in one or two memory round trips.
//  * Every wait on a barrier is bounded (common.cuh); on timeout the warp
//    flags SA_ERR_TIMEOUT, drains its copies in flight and leaves.
#include "common.cuh"
#include "tc_work.cuh"

namespace sa {

namespace {

// Tuning constants (measured on GB300: 16-token tiles, two stages per warp and
// 2R lanes per token were fastest for the decode batch).
constexpr int kTile = 16;                     // tokens per stage
constexpr int kRowBytes = kHeadDim * 2;       // one K or V row: 256 bytes
constexpr int kKVBytes = kTile * kRowBytes;   // K (or V) rows of one tile, contiguous in a page
constexpr int kStageBytes = 2 * kKVBytes;     // K tile, then V tile
// Quantised pages (KB-bit codes, KB = 8 or 4): a stage holds the tile's K
// codes, V codes, K scales and V scales, in that order.
template <int KB>
struct QTile {
    static constexpr int kCodeRow = kHeadDim * KB / 8;         // bytes of one row's codes
    static constexpr int kCodeBytes = kTile * kCodeRow;        // 2 KiB (int8), 1 KiB (int4)
    static constexpr int kScaleBytes = kTile * 4;              // 64 bytes
    static constexpr int kVCodes = kCodeBytes, kKScales = 2 * kCodeBytes, kVScales = kKScales + kScaleBytes;
    static constexpr int kBytes = kVScales + kScaleBytes;
};
static_assert(QTile<8>::kBytes <= kStageBytes && QTile<4>::kBytes <= kStageBytes, "quantised tiles use the bf16 stage");
constexpr int kStages = 2;                    // pipeline depth per warp
constexpr int kRing = kStages + 2;            // piece descriptors in flight (>= kStages + 1)
constexpr int kPieceInts = 16;

template <int R>
struct Geo {
    static constexpr int L = 2 * R < 32 ? 2 * R : 32;                // lanes per token
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
    int tc;  // attended on the tensor cores (runs are then per segment: tc_work.cuh)
};

constexpr int kQkBatch = 32;  // score values a lane reduces in one batch of steps

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

// The same dims of row t of a tile of int8 codes (128-byte rows), as pairs of
// floats (pair k holds this lane's dims of bf16 word k); the codes' scale is
// applied by the caller, per token.
// Codes are converted exactly without the (slow) integer-to-float unit: u =
// code + 128 (the word xor 0x80808080) put in the low byte of the binary32
// 2^23 is 2^23 + u, and one paired subtraction of 2^23 + 128 leaves the code.
__device__ __forceinline__ float2 codes_pair(uint32_t w, int hi) {
    const uint32_t u = w ^ 0x80808080u;
    const float a = __uint_as_float(__byte_perm(u, 0x4B000000u, hi ? 0x7442u : 0x7440u));
    const float b = __uint_as_float(__byte_perm(u, 0x4B000000u, hi ? 0x7443u : 0x7441u));
    return ffma2(make_float2(a, b), make_float2(1.f, 1.f), make_float2(-8388736.f, -8388736.f));
}

template <int L>
__device__ __forceinline__ void load_tile_row_q8(const uint8_t *tile, int t, int j, float2 (&f)[64 / L]) {
    const uint8_t *row = tile + t * kHeadDim;
    if constexpr (L == 8) {
        const uint2 a = *reinterpret_cast<const uint2 *>(row + j * 8);
        const uint2 b = *reinterpret_cast<const uint2 *>(row + 64 + j * 8);
        f[0] = codes_pair(a.x, 0); f[1] = codes_pair(a.x, 1); f[2] = codes_pair(a.y, 0); f[3] = codes_pair(a.y, 1);
        f[4] = codes_pair(b.x, 0); f[5] = codes_pair(b.x, 1); f[6] = codes_pair(b.y, 0); f[7] = codes_pair(b.y, 1);
    } else if constexpr (L == 16) {
        const uint2 a = *reinterpret_cast<const uint2 *>(row + j * 8);
        f[0] = codes_pair(a.x, 0); f[1] = codes_pair(a.x, 1); f[2] = codes_pair(a.y, 0); f[3] = codes_pair(a.y, 1);
    } else {
        const uint32_t a = *reinterpret_cast<const uint32_t *>(row + j * 4);
        f[0] = codes_pair(a, 0); f[1] = codes_pair(a, 1);
    }
}

// The same dims of row t of a tile of int4 codes (64-byte rows; value 2c is
// the low nibble of byte c, stored as code + 8), as pairs of floats. The
// nibbles of a word are split into bytes (low nibbles, high nibbles) and
// converted like int8 codes: byte n in the low byte of 2^23 is 2^23 + n, and
// one paired subtraction of 2^23 + 8 leaves the code, exactly.
__device__ __forceinline__ void nibbles_pairs(uint32_t w, int npairs, float2 *f) {
    const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if (k < npairs) {
            const float a = __uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7440u + k));
            const float b = __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7440u + k));
            f[k] = ffma2(make_float2(a, b), make_float2(1.f, 1.f), make_float2(-8388616.f, -8388616.f));
        }
    }
}

template <int L>
__device__ __forceinline__ void load_tile_row_q4(const uint8_t *tile, int t, int j, float2 (&f)[64 / L]) {
    const uint8_t *row = tile + t * (kHeadDim / 2);
    if constexpr (L == 8) {  // dims 8j..8j+7 and 64+8j..64+8j+7: bytes 4j.. and 32+4j..
        nibbles_pairs(*reinterpret_cast<const uint32_t *>(row + j * 4), 4, f);
        nibbles_pairs(*reinterpret_cast<const uint32_t *>(row + 32 + j * 4), 4, f + 4);
    } else if constexpr (L == 16) {  // dims 8j..8j+7: bytes 4j..4j+3
        nibbles_pairs(*reinterpret_cast<const uint32_t *>(row + j * 4), 4, f);
    } else {  // dims 4j..4j+3: bytes 2j, 2j+1
        nibbles_pairs(*reinterpret_cast<const uint16_t *>(row + j * 2), 2, f);
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

// Per-sequence shape of the work; tiles = 0 when the sequence has none. The
// packed query rows of all sequences are checked against total_q once, by the
// caller of this function, so no per-sequence query offset is needed here.

template <int R>
__device__ __forceinline__ SeqInfo seq_info_from(const SplitParams &P, int T, int n, int skip_pages,
                                                 int run_slots, bool flag);

template <int R>
__device__ __forceinline__ SeqInfo seq_info(const SplitParams &P, int b, bool flag) {
    return seq_info_from<R>(P, P.seq_lens[b], P.q_lens[b], P.skip_pages ? P.skip_pages[b] : 0,
                            P.run_slots ? P.run_slots[b] : 0, flag);
}

template <int R>
__device__ __forceinline__ SeqInfo seq_info_from(const SplitParams &P, int T, int n, int skip_pages,
                                                 int run_slots, bool flag) {
    SeqInfo s;
    s.T = T;
    s.n = n;
    s.tiles = 0;
    s.nrb = 0;
    s.skip_tok = 0;
    s.runs = 0;
    s.tc = 0;
    if (s.n <= 0) return s;
    const int npages = (s.T + kPageSize - 1) / kPageSize;
    if (s.n > s.T || s.n > P.max_q_len || npages > P.max_pages) {
        if (flag) flag_error(P.err, kErrBitQlen);
        return s;
    }
    int skip = skip_pages;
    int runs = run_slots;
    s.tc = 0;
    if (P.tc_min_rows > 0 && P.G * s.n >= P.tc_min_rows) {  // attended on the tensor cores
        skip = npages;
        runs = 0;
        s.tc = 1;
    }
    s.runs = runs;
    s.skip_tok = skip * kPageSize;
    const int keys = s.T - s.skip_tok;
    s.tiles = keys > 0 ? (keys + kTile - 1) / kTile : 0;  // tensor-core partials only: merged by the combine pass
    s.nrb = (P.G * s.n + R - 1) / R;
    return s;
}

// The cut of the tile sequence [0, total) into one contiguous range per warp:
// every warp gets C or C + 1 tiles (the first `rem` get C + 1) when that keeps
// C >= C_min; otherwise ranges of C_min tiles and the last warps stay idle.
// Work offsets are counted in balancing units in 32 bits: the host rejects
// shapes whose largest possible total reaches 2^31.
struct Ranges {
    int C, rem;  // warp w gets C + 1 units if w < rem, else C
    __device__ __forceinline__ int begin(int w) const { return w * C + min(w, rem); }
    __device__ __forceinline__ int range_of(int t) const {
        const int big = rem * (C + 1);
        return t < big ? t / (C + 1) : rem + (t - big) / C;
    }
};

// Every warp gets C or C + 1 units when that keeps C >= C_min; otherwise
// ranges of C_min units and the last warps stay idle.
__device__ __forceinline__ Ranges make_ranges(int total, int W, int C_min) {
    const int even = total / W;
    if (even >= C_min) return Ranges{even, total - even * W};
    return Ranges{C_min, 0};
}

// The work of a segment in balancing units: kUnitsPerTile per tile plus
// kSegmentCost for the segment's start (closing the previous piece, loading
// and converting new queries), so that a warp whose range crosses into a new
// segment gets fewer tiles. Tile t of a segment that starts at unit u sits at
// unit u + kSegmentCost + kUnitsPerTile * t and belongs to the warp whose range
// holds that unit.
constexpr int kUnitsPerTile = 4;
constexpr int kSegmentCost = 8;

__device__ __forceinline__ int segment_units(const SeqInfo &s) {
    return s.tiles > 0 ? kSegmentCost + kUnitsPerTile * s.tiles : 0;
}

__device__ __forceinline__ int seq_work(const SplitParams &P, const SeqInfo &s) {
    return segment_units(s) * P.Hkv * s.nrb;
}

// Merging a row's partials (the tensor-core runs' slots, then the pieces'
// slots) with exact max-shifted rescaling.

__device__ __forceinline__ const float *ws_slot_row(const SplitParams &P, const Piece &U, int k, int64_t row,
                                                    const float *base, int width) {
    const int slot = k < U.runs ? k : P.slot_base + (k - U.runs);
    return base + (static_cast<int64_t>(slot) * P.n_rows_total + row) * width;
}

// 16 head dims (sub*16 ..) of an output row: o / Lsum rounded to bf16.
__device__ __forceinline__ void store_row(const SplitParams &P, int64_t row, int sub, const float4 (&o)[4], float Lsum) {
    const float inv = Lsum > 0.f ? __frcp_rn(Lsum) : 0.f;
    uint4 *dst = reinterpret_cast<uint4 *>(P.out + row * kHeadDim + sub * 16);
    dst[0] = make_uint4(pack_bf16x2(o[0].x * inv, o[0].y * inv), pack_bf16x2(o[0].z * inv, o[0].w * inv),
                        pack_bf16x2(o[1].x * inv, o[1].y * inv), pack_bf16x2(o[1].z * inv, o[1].w * inv));
    dst[1] = make_uint4(pack_bf16x2(o[2].x * inv, o[2].y * inv), pack_bf16x2(o[2].z * inv, o[2].w * inv),
                        pack_bf16x2(o[3].x * inv, o[3].y * inv), pack_bf16x2(o[3].z * inv, o[3].w * inv));
}

// Rows r4*4 .. r4*4+3 of a segment: eight lanes per row, 16 head dims each.
// Up to four partials are read in one round trip (every (max, sum) and
// accumulator in flight together); more take two (the maxima, then the
// accumulators).
__device__ __forceinline__ void merge_rows(const SplitParams &P, const Piece &U, int R, int r4, int lane, bool store) {
    const int nslots = U.runs + U.pieces;
    const int sub = lane & 7;
    const int r = r4 * 4 + (lane >> 3);
    if (r >= U.nvr) return;
    const int64_t row = out_row(P, U, U.rb * R + r);
    float M = -INFINITY, Lsum = 0.f;
    float4 o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) o[q] = make_float4(0, 0, 0, 0);
    if (nslots <= 4) {
        float2 ml[4];
        float4 av[4][4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            ml[k] = make_float2(-INFINITY, 0.f);
            if (k < nslots) {
                ml[k] = __ldcg(reinterpret_cast<const float2 *>(ws_slot_row(P, U, k, row, P.ws_ml, 2)));
                const float4 *a = reinterpret_cast<const float4 *>(ws_slot_row(P, U, k, row, P.ws_acc, kHeadDim) + sub * 16);
#pragma unroll
                for (int q = 0; q < 4; ++q) av[k][q] = __ldcg(a + q);
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (ml[k].y > 0.f) M = fmaxf(M, ml[k].x);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (ml[k].y > 0.f) {
                const float w = exp2f(ml[k].x - M);
                Lsum += ml[k].y * w;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    o[q].x += av[k][q].x * w;
                    o[q].y += av[k][q].y * w;
                    o[q].z += av[k][q].z * w;
                    o[q].w += av[k][q].w * w;
                }
            }
        }
    } else {
        // the maxima first (all loads in flight), then the accumulators
        for (int k = 0; k < nslots; ++k) {
            const float2 ml = __ldcg(reinterpret_cast<const float2 *>(ws_slot_row(P, U, k, row, P.ws_ml, 2)));
            if (ml.y > 0.f) M = fmaxf(M, ml.x);
        }
        for (int k = 0; k < nslots; ++k) {
            const float2 ml = __ldcg(reinterpret_cast<const float2 *>(ws_slot_row(P, U, k, row, P.ws_ml, 2)));
            if (ml.y > 0.f) {
                const float w = exp2f(ml.x - M);
                Lsum += ml.y * w;
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
    }
    if (store) store_row(P, row, sub, o, Lsum);
}

__device__ __forceinline__ SeqInfo shfl_seq_info(SeqInfo si, int src) {
    si.T = __shfl_sync(0xffffffffu, si.T, src);
    si.n = __shfl_sync(0xffffffffu, si.n, src);
    si.skip_tok = __shfl_sync(0xffffffffu, si.skip_tok, src);
    si.tiles = __shfl_sync(0xffffffffu, si.tiles, src);
    si.nrb = __shfl_sync(0xffffffffu, si.nrb, src);
    si.runs = __shfl_sync(0xffffffffu, si.runs, src);
    si.tc = __shfl_sync(0xffffffffu, si.tc, src);
    return si;
}

// ---- the work scan shared by the split and combine kernels
// Lane i looks after sequences i, i + 32, ...; each round of 32 sequences is
// reduced with warp-wide integer reductions, and the next round's lengths are
// loaded before the current round is reduced. The code is kept small on
// purpose: it runs once per warp, so its instructions are fetched cold.
struct WorkScan {
    int total;      // all work, in tiles
    int q_total;    // all query tokens
    int max_tiles;  // longest segment, in tiles
};

template <int R>
__device__ __forceinline__ SeqInfo seq_of(const SplitParams &P, int b, bool flag) {
    if (b >= P.B) return SeqInfo{0, 0, 0, 0, 0, 0, 0};
    return seq_info<R>(P, b, flag);
}

// A sequence's raw lengths (no work when b is past the batch).
struct SeqRaw {
    int T, n, sk, rs;
};

__device__ __forceinline__ SeqRaw load_raw(const SplitParams &P, int b) {
    if (b >= P.B) return SeqRaw{0, 0, 0, 0};
    return SeqRaw{P.seq_lens[b], P.q_lens[b], P.skip_pages ? P.skip_pages[b] : 0, P.run_slots ? P.run_slots[b] : 0};
}

template <int R>
__device__ __forceinline__ void scan_work(const SplitParams &P, int lane, bool flag, WorkScan &sc) {
    sc.total = 0;
    sc.q_total = 0;
    sc.max_tiles = 0;
    SeqRaw nxt = load_raw(P, lane);
#pragma unroll 1
    for (int base = 0; base < P.B; base += 32) {
        const SeqRaw cur = nxt;
        if (base + 32 < P.B) nxt = load_raw(P, base + 32 + lane);  // in flight while this round is reduced
        const SeqInfo si = seq_info_from<R>(P, cur.T, cur.n, cur.sk, cur.rs, flag);
        sc.total += __reduce_add_sync(0xffffffffu, static_cast<unsigned>(seq_work(P, si)));
        sc.q_total += __reduce_add_sync(0xffffffffu, static_cast<unsigned>(max(0, si.n)));
        sc.max_tiles = max(sc.max_tiles, static_cast<int>(__reduce_max_sync(0xffffffffu, static_cast<unsigned>(si.tiles))));
    }
}

// The cut of the work into W warp ranges. A segment of u units spans at most
// ceil(u / C) + 1 ranges: C is at least ceil(longest / (slots - 1)) so that no
// segment has more pieces than the workspace has partial slots.
__device__ __forceinline__ Ranges split_ranges(const SplitParams &P, const WorkScan &sc, int W) {
    const int mu = kSegmentCost + kUnitsPerTile * sc.max_tiles;
    const int C_min = P.piece_slots > 1 ? (mu + P.piece_slots - 2) / (P.piece_slots - 1) : mu;
    return make_ranges(sc.total, W, max(C_min, 1));
}

// Pieces (warp ranges) that a segment starting at unit u0 with `tiles` tiles is cut into.
__device__ __forceinline__ void segment_ranges(const Ranges &rg, int u0, int tiles, int &first, int &last) {
    first = rg.range_of(u0 + kSegmentCost);
    last = rg.range_of(u0 + kSegmentCost + kUnitsPerTile * (tiles - 1));
}

// The sequence whose work holds tile g (by_work) or sequence bt: its index,
// work offset, query offset and shape, the same on every lane. A second pass
// over the lengths, which the scan left in L1.
template <int R>
__device__ __forceinline__ void locate_seq(const SplitParams &P, int lane, bool by_work, int g, int bt,
                                           int &b_out, int &pos, int &qs, SeqInfo &si_out) {
    int w_base = 0, q_base = 0;
#pragma unroll 1
    for (int base = 0; base < P.B; base += 32) {
        const int b = base + lane;
        const SeqInfo si = seq_of<R>(P, b, false);
        const int w = seq_work(P, si), qn = max(0, si.n);
        int wi = w, qi = qn;  // inclusive prefix sums over the lanes
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int a = __shfl_up_sync(0xffffffffu, wi, o), c = __shfl_up_sync(0xffffffffu, qi, o);
            if (lane >= o) {
                wi += a;
                qi += c;
            }
        }
        const int wx = w_base + wi - w, qx = q_base + qi - qn;
        const unsigned hit = __ballot_sync(0xffffffffu, by_work ? (w > 0 && wx <= g && g < wx + w) : b == bt);
        if (hit) {
            const int src = __ffs(hit) - 1;
            b_out = base + src;
            pos = __shfl_sync(0xffffffffu, wx, src);
            qs = __shfl_sync(0xffffffffu, qx, src);
            si_out = shfl_seq_info(si, src);
            return;
        }
        w_base += __shfl_sync(0xffffffffu, wi, 31);
        q_base += __shfl_sync(0xffffffffu, qi, 31);
    }
    b_out = P.B;  // not found (only when g is past all work)
}


// KB: 16 for bf16 pages, 8 for int8 pages, 4 for int4 pages.
template <int R, int KB>
__global__ void __launch_bounds__(32, 1) split_attn_kernel(const SplitParams P) {
    using Gm = Geo<R>;
    using Lay = Layout<R>;
    constexpr bool Q = KB < 16;             // quantised pages
    using QT = QTile<Q ? KB : 8>;           // their stage layout (unused for bf16 pages)
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

    // The combine kernel may be scheduled now: it waits for this grid before
    // it reads the partials. This kernel itself may have been started while
    // the kernel before it still runs. After kv_append, everything up to the
    // grid dependency wait below reads only lengths and block tables, which
    // kv_append does not write; queries and pages are read after the wait.
    // After a tensor-core kernel of this call (which started once the pages
    // were complete and writes only partials), pages are read at once, and
    // CTA 0 alone waits for that kernel before it exits: this grid then
    // completes after its predecessor (the combine pass sees the tensor-core
    // partials), while every other CTA leaves as soon as its range is done,
    // so that the SMs the tensor-core kernel leaves free keep taking new CTAs.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const bool exit_wait = !P.pages_ready || blockIdx.x == 0;

    // ---- 1. total work and this warp's range [g_begin, g_end) of tiles
    WorkScan sc;
    scan_work<R>(P, lane, true, sc);
    if (sc.q_total > P.total_q) {  // q_lens disagree with dims.total_q: reject the whole call
        if (lane == 0) flag_error(P.err, kErrBitQlen);
        grid_dependency_wait();
        return;
    }
    const Ranges rg = split_ranges(P, sc, gridDim.x);
    const int g_begin = rg.begin(blockIdx.x);
    const int g_end = min(sc.total, rg.begin(blockIdx.x + 1));
    __syncwarp();
    if (g_begin >= g_end) {
        if (exit_wait) grid_dependency_wait();
        return;
    }

    // ---- 2. locate the first tile (the first tile unit at or after g_begin)
    // and read its page id and the next page's
    int b0 = 0, q0 = 0, ws0 = 0;
    SeqInfo si0{};
    locate_seq<R>(P, lane, true, g_begin, 0, b0, ws0, q0, si0);
    const int seg_units0 = segment_units(si0);
    const int iseg0 = (g_begin - ws0) / seg_units0;
    const int in_seg = (g_begin - ws0) - iseg0 * seg_units0;
    const int tile0 = in_seg <= kSegmentCost ? 0 : (in_seg - kSegmentCost + kUnitsPerTile - 1) / kUnitsPerTile;
    const bool primed = tile0 < si0.tiles;  // else the first tile is in the next segment
    const int t0_first = si0.skip_tok + tile0 * kTile;
    const int j0 = t0_first / kPageSize;
    const int64_t bt0 = static_cast<int64_t>(b0) * P.max_pages;
    const int pid0 = primed && t0_first < si0.T ? P.block_table[bt0 + j0] : -1;
    const int pid1 = primed && j0 + 1 < (si0.T + kPageSize - 1) / kPageSize ? P.block_table[bt0 + j0 + 1] : -1;

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

    // ---- issue cursor: walks this warp's tiles ahead of the consumer; ig is
    // the unit of the next tile
    int ib = b0, iq = q0;
    int iws = ws0;
    SeqInfo isi = si0;
    int iseg = iseg0, itile = tile0;
    int ikvh = iseg / isi.nrb, irb = iseg % isi.nrb;
    int ig = ws0 + iseg * seg_units0 + kSegmentCost + kUnitsPerTile * tile0;
    bool first_piece = true;
    uint32_t issued = 0, consumed = 0, pieces_pushed = 0;
    // Page ids and lengths the issue cursor needs, each read well before its
    // first use so that no block-table or length load stalls the issue of a
    // tile: the current page's id and the next page's; the current sequence's
    // first page (every KV head's segment starts there); the next sequence's
    // lengths and, without a plan, its first page.
    int pg_b = primed ? b0 : -1, pg_j = j0, pg_id = pid0, pg_next = pid1;  // primed after locating
    int f_b = b0, f_j = si0.skip_tok / kPageSize;
    int f_pid = primed && j0 == f_j ? pid0 : P.block_table[static_cast<int64_t>(b0) * P.max_pages + f_j];
    const bool plain = P.skip_pages == nullptr && P.run_slots == nullptr;  // sequences start at page 0
    int nx_b = -1, nx_T = 0, nx_n = 0, nx_sk = 0, nx_rs = 0, nx_pid = -1;
    auto prefetch_next = [&](int b) {
        nx_b = b + 1 < P.B ? b + 1 : -1;
        if (nx_b < 0) return;
        nx_T = P.seq_lens[nx_b];
        nx_n = P.q_lens[nx_b];
        nx_sk = P.skip_pages ? P.skip_pages[nx_b] : 0;
        nx_rs = P.run_slots ? P.run_slots[nx_b] : 0;
        nx_pid = plain ? P.block_table[static_cast<int64_t>(nx_b) * P.max_pages] : -1;
    };
    prefetch_next(b0);
    auto page_id = [&](int b, int jp, int npages) -> int {
        if (b == pg_b && jp == pg_j) return pg_id;
        const int64_t base = static_cast<int64_t>(b) * P.max_pages;
        pg_id = (b == pg_b && jp == pg_j + 1) ? pg_next : (b == f_b && jp == f_j) ? f_pid : P.block_table[base + jp];
        pg_b = b;
        pg_j = jp;
        pg_next = jp + 1 < npages ? P.block_table[base + jp + 1] : -1;
        return pg_id;
    };
    auto issue_next = [&]() -> bool {
        if (ig >= g_end) return false;
        if (itile == isi.tiles) {  // next segment
            itile = 0;
            ig += kSegmentCost;
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
                    isi = ib == nx_b ? seq_info_from<R>(P, nx_T, nx_n, nx_sk, nx_rs, false) : seq_info<R>(P, ib, false);
                } while (seq_work(P, isi) == 0);
                f_b = ib;
                f_j = isi.skip_tok / kPageSize;
                f_pid = (ib == nx_b && plain && f_j == 0) ? nx_pid : P.block_table[static_cast<int64_t>(ib) * P.max_pages + f_j];
                prefetch_next(ib);
            }
            if (ig >= g_end) return false;
        }
        const int kvh = ikvh, rb = irb;
        if (first_piece || itile == 0) {
            // a new piece: describe it for the consumer and fetch its query rows
            first_piece = false;
            int first, last;
            segment_ranges(rg, iws + iseg * segment_units(isi), isi.tiles, first, last);
            const int nvr = min(R, P.G * isi.n - rb * R);
            const int qs = pieces_pushed % S;
            if (lane == 0) {
                int32_t *d = ring + (pieces_pushed % kRing) * kPieceInts;
                d[0] = ib; d[1] = kvh; d[2] = rb; d[3] = isi.T; d[4] = isi.n; d[5] = iq;
                d[6] = isi.skip_tok + itile * kTile;
                d[7] = min(isi.tiles - itile, (g_end - ig + kUnitsPerTile - 1) / kUnitsPerTile);
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
        // (t0 < T for every tile of a segment: tiles = ceil(keys / kTile))
        const int pid = page_id(ib, t0 / kPageSize, (isi.T + kPageSize - 1) / kPageSize);
        const bool ok = static_cast<unsigned>(pid) < static_cast<unsigned>(P.num_pages);
        if (!ok && lane == 0) flag_error(P.err, kErrBitPageOOB);
        if (lane < (Q ? 4 : 2)) {
            if (ok) {
                // The tile's K rows and V rows are each one contiguous run in the
                // page: lane 0 copies the K rows, lane 1 the V rows, in one
                // instruction (the copy instruction's issue is slow; two lanes
                // take the time of one). Quantised pages: lanes 2 and 3 copy the
                // rows' K and V scales (also contiguous) in the same instruction.
                const int64_t row = static_cast<int64_t>(pid * P.Hkv + kvh) * kPageSize + (t0 % kPageSize);
                if (lane == 0) {
                    stage_ok[s] = 1;
                    mbar_arrive_expect_tx(&full[s], Q ? QT::kBytes : kStageBytes);
                }
                if constexpr (Q) {
                    const void *src = lane == 0 ? static_cast<const void *>(P.k_codes + row * QT::kCodeRow)
                                    : lane == 1 ? static_cast<const void *>(P.v_codes + row * QT::kCodeRow)
                                    : lane == 2 ? static_cast<const void *>(P.k_scales + row)
                                                : static_cast<const void *>(P.v_scales + row);
                    const int off = lane == 0 ? 0 : lane == 1 ? QT::kVCodes : lane == 2 ? QT::kKScales : QT::kVScales;
                    bulk_load_hint(smem + s * kStageBytes + off, src, lane < 2 ? QT::kCodeBytes : QT::kScaleBytes,
                                   &full[s], policy);
                } else {
                    bulk_load_hint(smem + s * kStageBytes + lane * kKVBytes, (lane ? P.v_pages : P.k_pages) + row * kHeadDim,
                                   kKVBytes, &full[s], policy);
                }
            } else if (lane == 0) {
                stage_ok[s] = 0;
                mbar_arrive(&full[s]);  // nothing to load: the consumer skips this tile
            }
        }
        ++issued;
        ++itile;
        ig += kUnitsPerTile;
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
        if (P.pages_ready) grid_dependency_wait();
        for (uint32_t c = consumed; c < issued; ++c) (void)mbar_wait(&full[c % S], (c / S) & 1);
        for (uint32_t c = pieces_done; c < pieces_pushed; ++c) (void)mbar_wait(&qfull[c % S], (c / S) & 1);
    };

    // the pages written by the previous kernel are complete (when a tensor-core
    // kernel of this call ran first, it started after them: no wait needed here)
    if (!P.pages_ready) grid_dependency_wait();
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
                constexpr int NB0 = (kQkBatch / R) < NS ? (kQkBatch / R) : NS;
                constexpr int NB = NB0 > 0 ? NB0 : 1;  // steps per batch
#pragma unroll
                for (int b0 = 0; b0 < NS; b0 += NB) {
                    float v[NB][R];
#pragma unroll
                    for (int bi = 0; bi < NB; ++bi) {
                        const int t = (b0 + bi) * TG + tg;
                        uint32_t kw[NW];
                        float2 kq[NW];
                        if constexpr (KB == 8) load_tile_row_q8<L>(st, t, j, kq);
                        else if constexpr (KB == 4) load_tile_row_q4<L>(st, t, j, kq);
                        else load_tile_row<L>(st, t, j, kw);
                        float2 a2[R];
#pragma unroll
                        for (int r = 0; r < R; ++r) a2[r] = make_float2(0.f, 0.f);
#pragma unroll
                        for (int k = 0; k < NW; ++k) {
                            const float2 kf = Q ? kq[k] : unpack_bf16x2(kw[k]);
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
                        // quantised pages: the dot was over codes; the key row's scale completes it
                        const float ks = Q ? reinterpret_cast<const float *>(st + QT::kKScales)[t] : 1.f;
                        sv[b0 + bi] = t0 + t <= lim ? v[bi][0] * ks : -INFINITY;
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
                    // quantised pages: p times the value row's scale, so that P V runs on codes
                    if (row_writer)
                        pbuf[step * TG + tg][rj] = Q ? p * reinterpret_cast<const float *>(st + QT::kVScales)[step * TG + tg] : p;
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
                        float2 vq[NW];
                        if constexpr (KB == 8) load_tile_row_q8<L>(st + QT::kVCodes, t, j, vq);
                        else if constexpr (KB == 4) load_tile_row_q4<L>(st + QT::kVCodes, t, j, vq);
                        else load_tile_row<L>(st + kKVBytes, t, j, vw);
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
                            const float2 vf = Q ? vq[k] : unpack_bf16x2(vw[k]);
#pragma unroll
                            for (int r = 0; r < R; ++r) acc[r][k] = ffma2(make_float2(pr[r], pr[r]), vf, acc[r][k]);
                        }
                    }
                }
            }
            __syncwarp();   // stage and p buffer are reused by later tiles
            ++consumed;
        }

        // ---- finish the piece. The token groups' accumulators are summed in
        // shared memory, in the stage of the piece's last tile (free until the
        // next top-up), as [TG][R][128] fp32; then each lane owns 4R head dims
        // of one row and writes them out (bf16) or as a partial (fp32).
#pragma unroll
        for (int o = L; o < 32; o <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
        if (tg == 0 && row_writer) {
            rowx[rj] = m;
            rowx[R + rj] = lsum;
        }
        float *red = reinterpret_cast<float *>(smem + ((consumed - 1) % S) * kStageBytes);
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int k = 0; k < NW; k += 2)
                *reinterpret_cast<float4 *>(red + (tg * R + r) * kHeadDim + lane_dim_of_word<L>(j, k)) =
                    make_float4(acc[r][k].x, acc[r][k].y, acc[r][k + 1].x, acc[r][k + 1].y);
        __syncwarp();
        {
            constexpr int DPL = 4 * R;              // head dims per lane
            constexpr int LPR = kHeadDim / DPL;     // lanes per row
            const int r = lane / LPR, d0 = (lane % LPR) * DPL;
            if (r < U.nvr) {
                float4 o[DPL / 4];
#pragma unroll
                for (int v = 0; v < DPL / 4; ++v) {
                    o[v] = *reinterpret_cast<const float4 *>(red + r * kHeadDim + d0 + 4 * v);
#pragma unroll
                    for (int g = 1; g < TG; ++g) {
                        const float4 a = *reinterpret_cast<const float4 *>(red + (g * R + r) * kHeadDim + d0 + 4 * v);
                        o[v].x += a.x;
                        o[v].y += a.y;
                        o[v].z += a.z;
                        o[v].w += a.w;
                    }
                }
                const int64_t row = out_row(P, U, U.rb * R + r);
                if (direct) {
                    const float inv = __frcp_rn(rowx[R + r]);
                    uint4 *dst = reinterpret_cast<uint4 *>(P.out + row * kHeadDim + d0);
#pragma unroll
                    for (int v = 0; v < DPL / 8; ++v)
                        dst[v] = make_uint4(pack_bf16x2(o[2 * v].x * inv, o[2 * v].y * inv),
                                            pack_bf16x2(o[2 * v].z * inv, o[2 * v].w * inv),
                                            pack_bf16x2(o[2 * v + 1].x * inv, o[2 * v + 1].y * inv),
                                            pack_bf16x2(o[2 * v + 1].z * inv, o[2 * v + 1].w * inv));
                } else {
                    const int64_t wi = static_cast<int64_t>(P.slot_base + U.piece) * P.n_rows_total + row;
                    float4 *dst = reinterpret_cast<float4 *>(P.ws_acc + wi * kHeadDim + d0);
#pragma unroll
                    for (int v = 0; v < DPL / 4; ++v) dst[v] = o[v];
                    if (d0 == 0) *reinterpret_cast<float2 *>(P.ws_ml + wi * 2) = make_float2(rowx[r], rowx[R + r]);
                }
            }
        }
        __syncwarp();
    }
    if (P.pages_ready && blockIdx.x == 0) grid_dependency_wait();  // see exit_wait above
}

// Pieces the tensor-core sequence mode cut segment (bt, kvh, mt) into: a scan
// over the sequences gives the tile sequence's total, its longest segment and
// the segment's first unit, and the same cut as the tensor-core kernel's.
template <int R>
__device__ int tc_pieces(const SplitParams &P, int lane, int bt, int kvh, int mt) {
    int total = 0, max_tiles = 0, u0 = 0;
    TcSeq wb{0, 0, 0};
    bool uniform = P.B > 0;  // as the tensor-core kernel decides its waves
    const int T0 = P.B > 0 ? P.seq_lens[0] : 0, n0 = P.B > 0 ? P.q_lens[0] : 0;
#pragma unroll 1
    for (int base = 0; base < P.B; base += 32) {
        const int b = base + lane;
        const int T = b < P.B ? P.seq_lens[b] : 0, n = b < P.B ? P.q_lens[b] : 0;
        const TcSeq w = tc_seq(T, n, P.G, P.Hkv, P.max_q_len, P.max_pages, P.tc_min_rows);
        uniform = uniform && __all_sync(0xffffffffu, b >= P.B || (T == T0 && n == n0 && w.units > 0));
        int ui = w.units;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int a = __shfl_up_sync(0xffffffffu, ui, o);
            if (lane >= o) ui += a;
        }
        const int src = bt - base;
        if (src >= 0 && src < 32) {
            u0 = total + __shfl_sync(0xffffffffu, ui - w.units, src);
            wb.tiles = __shfl_sync(0xffffffffu, w.tiles, src);
            wb.mtiles = __shfl_sync(0xffffffffu, w.mtiles, src);
        }
        total += __shfl_sync(0xffffffffu, ui, 31);
        max_tiles = max(max_tiles, static_cast<int>(__reduce_max_sync(0xffffffffu, static_cast<unsigned>(w.tiles))));
    }
    if (wb.tiles == 0) return 0;
    const TcWaves waves = make_tc_waves(uniform, P.B, tc_seq(T0, n0, P.G, P.Hkv, P.max_q_len, P.max_pages, P.tc_min_rows),
                                        P.Hkv, P.tc_grid, P.G * n0);
    const int s0 = u0 + (kvh * wb.mtiles + mt) * wb.tiles;
    if (s0 < waves.base) return 0;  // a whole segment of a wave: written by the tensor-core kernel
    const TcRanges rg = make_tc_ranges(total - waves.base, P.tc_grid, max_tiles);
    return rg.range_of(s0 - waves.base + wb.tiles - 1) - rg.range_of(s0 - waves.base) + 1;
}

// ---- the combine pass: one warp per (sequence, KV head, row block, group of
// four rows) merges the partials of a segment that was cut into pieces or
// has tensor-core partials. It repeats the split kernel's scan (before the
// grid dependency wait, so this overlaps the split kernel) to find the pieces.
// One warp per CTA and at most 128 registers, so that a combine CTA fits beside
// the eight resident split CTAs of an SM and can be scheduled early.
constexpr int kCombineWarps = 1;
constexpr int kCombineMinCtas = 16;

template <int R>
__global__ void __launch_bounds__(kCombineWarps * 32, kCombineMinCtas) combine_kernel(const SplitParams P) {
    const int lane = threadIdx.x & 31;
    constexpr int RG = R / 4;
    const int64_t unit = static_cast<int64_t>(blockIdx.x) * kCombineWarps + threadIdx.x / 32;
    const int64_t per_seq = static_cast<int64_t>(P.Hkv) * P.n_row_blocks * RG;
    const int bt = static_cast<int>(unit / per_seq);
    if (bt >= P.B) return;
    int rem = static_cast<int>(unit % per_seq);
    const int kvh = rem / (P.n_row_blocks * RG);
    rem %= P.n_row_blocks * RG;
    const int rb = rem / RG, r4 = rem % RG;

    WorkScan sc;
    scan_work<R>(P, lane, false, sc);
    if (sc.q_total > P.total_q) return;  // flagged by the split kernel
    int b = 0, qs = 0, pos = 0;
    SeqInfo si{};
    locate_seq<R>(P, lane, false, 0, bt, b, pos, qs, si);
    if (si.n <= 0 || rb >= si.nrb) return;
    const int nvr = min(R, P.G * si.n - rb * R);
    if (r4 * 4 >= nvr) return;
    int pieces = 0;
    if (si.tiles > 0) {
        const Ranges rg = split_ranges(P, sc, P.split_ctas);
        int first, last;
        segment_ranges(rg, pos + (kvh * si.nrb + rb) * segment_units(si), si.tiles, first, last);
        pieces = last - first + 1;
    }
    int runs = si.runs;
    if (si.tc) runs = tc_pieces<R>(P, lane, bt, kvh, (rb * R) / kTcRowTile);
    if (runs == 0 && pieces <= 1) return;  // written directly by the split kernel
    Piece U{};
    U.b = bt;
    U.kvh = kvh;
    U.rb = rb;
    U.qstart = qs;
    U.pieces = pieces;
    U.runs = runs;
    U.nvr = nvr;
    // Pass 0 runs the merge on whatever the workspace holds now and stores
    // nothing: it brings the merge's instructions and address translations on
    // chip while the split kernel finishes. Pass 1, after the grid dependency
    // wait (the split kernel's partials are complete), is the merge.
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
        if (pass == 1) grid_dependency_wait();
        merge_rows(P, U, R, r4, lane, pass == 1);
    }
}

template <int R>
constexpr size_t smem_bytes() { return Layout<R>::kBytes + 1024; }

template <int R, int KB>
cudaError_t prepare() {
    static cudaError_t err = cudaFuncSetAttribute(split_attn_kernel<R, KB>,
                                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  static_cast<int>(smem_bytes<R>()));
    return err;
}

// Launch as a programmatic dependent of whatever precedes it on the stream:
// the kernel may start once its predecessor has signalled (kv_append does at
// once; any other kernel at its end) and waits for the predecessor's
// completion itself (griddepcontrol.wait) before reading its results.
template <typename Kernel>
cudaError_t launch_dependent(Kernel kernel, int grid, int threads, size_t smem, cudaStream_t stream,
                             const SplitParams &p) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <int R, int KB>
cudaError_t launch_r(const SplitParams &p, cudaStream_t stream) {
    cudaError_t e = prepare<R, KB>();
    if (e != cudaSuccess) return e;
    e = launch_dependent(split_attn_kernel<R, KB>, p.split_ctas, 32, smem_bytes<R>(), stream, p);
    if (e != cudaSuccess) return e;
    // the combine pass: its scan runs while the split kernel finishes
    const int64_t units = static_cast<int64_t>(p.B) * p.Hkv * p.n_row_blocks * (R / 4);
    return launch_dependent(combine_kernel<R>, static_cast<int>((units + kCombineWarps - 1) / kCombineWarps),
                            kCombineWarps * 32, 0, stream, p);
}

template <int R, int KB>
cudaError_t occupancy_r(int *ctas_per_sm) {
    cudaError_t e = prepare<R, KB>();
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, split_attn_kernel<R, KB>, 32,
                                                         smem_bytes<R>());
}

}  // namespace

int split_tile_tokens() { return kTile; }
int split_units_per_tile() { return kUnitsPerTile; }
int split_segment_cost() { return kSegmentCost; }

#define SA_SPLIT_CASES(F, ...)                                                                      \
    switch (R * 100 + KB) {                                                                          \
        case 416: return F<4, 16>(__VA_ARGS__);                                                       \
        case 816: return F<8, 16>(__VA_ARGS__);                                                       \
        case 1616: return F<16, 16>(__VA_ARGS__);                                                     \
        case 408: return F<4, 8>(__VA_ARGS__);                                                        \
        case 808: return F<8, 8>(__VA_ARGS__);                                                        \
        case 1608: return F<16, 8>(__VA_ARGS__);                                                      \
        case 404: return F<4, 4>(__VA_ARGS__);                                                        \
        case 804: return F<8, 4>(__VA_ARGS__);                                                        \
        case 1604: return F<16, 4>(__VA_ARGS__);                                                      \
        default: return cudaErrorInvalidValue;                                                       \
    }

cudaError_t split_occupancy(int R, int code_bits, int *ctas_per_sm) {
    const int KB = code_bits;
    SA_SPLIT_CASES(occupancy_r, ctas_per_sm)
}

cudaError_t launch_split_attn(const SplitParams &p, cudaStream_t stream) {
    const int R = p.rows_per_block, KB = p.k_codes != nullptr ? p.code_bits : 16;
    SA_SPLIT_CASES(launch_r, p, stream)
}
#undef SA_SPLIT_CASES

}  // namespace sa
