// attn_stream.cu -- page-streamed attention with one persistent CTA per SM:
// decode (q_len = 1) and short causal multi-query blocks (fewer than 16 query
// rows per KV head), bf16 pages.
//
// What it computes: for each sequence b, new query token i and query head h,
// softmax(scale * q . K_b^T) V_b over the keys at positions
// 0 .. seq_len - q_len + i, with K_b/V_b gathered through the block table
// (ExLlamaV2 "Dynamic Generator" page, "Continuous batching"; causal rows as
// in the Hugging Face "Assisted Generation" page, "How Assisted Generation
// works"). The softmax is evaluated online; partial (max, sum, accumulator)
// states are merged exactly with max-shifted rescaling.
//
// Design (sm_103a):
//  * Segment = (sequence, KV head, block of R <= 16 query rows): the G query
//    heads of the KV head times the sequence's new tokens, so every K/V byte
//    read serves all of them. The segments' 16-token sub-tiles, plus a small
//    cost per segment start, form one sequence of work units that is cut into
//    one equal contiguous range per CTA (one CTA per SM).
//  * Warp 0 produces: it walks the CTA's range and streams the tokens of one
//    KV head up to the next multiple of 64 per stage (so a stage lies in one
//    page) into a ring of six 32 KiB stages with 2-D TMA copies (128-byte
//    swizzle; at most three boxes of 64, 32 or 16 rows per half of K or V,
//    all issued by one instruction, since every box costs the TMA unit tens
//    of cycles to issue), and bulk-copies each piece's query rows. Six stages
//    keep about 160 KiB per SM in flight.
//  * Warps 4-7 consume: warp c takes tokens 16c .. 16c + 15 of every stage, a
//    16-token sub-tile. Each sub-tile is two tensor-core contractions of
//    one warp (mma.sync m16n8k16, bf16 in, fp32 accumulate): S = Q K^T with
//    the segment's query rows as M (padded to 16), eight tokens per N and the
//    head dimension as K, then O^T += V^T P^T with the head dimension as M, so
//    that the probabilities are the B operand straight from the S accumulators
//    and the R <= 8 query rows fill N = 8 without padding. K and V fragments come from
//    the swizzled stage with ldmatrix (transposed for V), free of bank
//    conflicts. Each warp keeps its own online-softmax state (lazy rescaling:
//    the reference maximum only moves when a tile beats it by 2^8).
//  * Warp 1 merges: at the end of a piece each consumer warp writes its
//    state over its own rows of the stage and hands the piece over through a
//    four-deep ring; the merge warp combines the four states, writes bf16
//    output (or an fp32 partial when the segment is cut between CTAs) and
//    releases the stage, so the consumers never wait for global memory.
//  * A CTA first streams the head of the segment it shares with the next CTA,
//    then the tail of the one it shares with the previous CTA, then its whole
//    segments, so that every CTA ends on segments it writes directly. Warp 2
//    counts the partials: the last CTA to finish a piece of a cut segment (one
//    atomic counter per cut, reset by that CTA) merges all of the segment's
//    partials; no CTA waits for another, and neither the consumers nor the
//    merge warp wait for these round trips to L2.
//  * Every wait is bounded (common.cuh). On timeout a warp flags
//    SA_ERR_TIMEOUT and leaves; the producer first waits (bounded) for its
//    copies in flight.
#include <cuda_fp16.h>

#include <type_traits>

#include "common.cuh"

namespace sa {

namespace {

constexpr int kStageTok = 64;                    // tokens per stage of bf16 pages
constexpr int kSub = 16;                         // tokens per sub-tile (and per smallest TMA box)
constexpr int kRoleWarps = 4;                    // warp 0 produces, 1 merges, 2 counts, 3 idle
constexpr int kHalf = kStageTok * 128;           // bf16 pages: 64 columns x 64 rows, 8 KiB
constexpr int kBoxBytes = kSub * 128;            // bf16 pages: one 16-row x 64-column box, 2 KiB
// The work is cut between CTAs at whole stages of a segment (64-token
// tiles): under a saturated memory system every stage in flight takes about
// one memory latency whatever its size, so a CTA's time follows its count of
// stages, and a cut inside a stage would add a partly filled one on each side.
constexpr int kCutTok = kStageTok;               // tokens per cut tile
constexpr int kUnitsPerTile = 16;                // balancing units of a cut tile
constexpr int kSegCost = 12;                     // units of a segment start (its queries, its
                                                 // merge)
constexpr int kMinUnits = 2 * kUnitsPerTile;     // smallest range: two full stages (a small batch
                                                 // is cut into fewer pieces, whose merge is a
                                                 // chain of L2 round trips)
constexpr int kPieceInts = 16;
constexpr int kQRow = kHeadDim + 8;              // query row stride in shared memory (bf16):
                                                 // 272 bytes, so that eight rows fall on
                                                 // different banks
constexpr int kQSlots = 4;                       // pieces whose queries are loaded ahead
constexpr int kMergeSlots = 4;
constexpr int kMslotInts = 8;
constexpr int kSmemLimit = 232448;               // dynamic shared memory of one CTA (227 KiB)

// stage descriptor flags
constexpr int kFirst = 1;  // first stage of a piece
constexpr int kLast = 2;   // last stage of a piece
constexpr int kEnd = 4;    // no more stages
constexpr int kSkip = 8;   // page id out of range: nothing was loaded

// A stage of one page format; KB = bits of a cached value: 16 (bf16 pages),
// 8 (int8 codes) or 4 (int4 codes, two per byte). Every stage costs the
// producer about the same few copies to issue, so stages of codes hold more
// tokens: about 32 KiB each.
//  * bf16: 64 tokens; K as two 64-column halves of 64 rows x 128 bytes
//    (128-byte swizzle), then V alike: 32 KiB.
//  * int8: 128 tokens; K codes, 128 rows x 128 bytes (128-byte swizzle), V
//    codes alike, then 128 K scales and 128 V scales (fp32): 33 KiB.
//  * int4: 256 tokens (a page); K codes, 256 rows x 64 bytes (64-byte
//    swizzle), V codes alike, then the scales: 34 KiB.
template <int KB>
struct Fmt {
    static constexpr bool kQuant = KB != 16;
    static constexpr int kStageTok = KB == 16 ? 64 : KB == 8 ? 128 : 256;  // tokens per stage
    // consumer warps (from warp 4 on): over codes two per scheduler, so that
    // one's code conversions and products hide the other's latencies
    static constexpr int kConsumers = kQuant ? 8 : 4;
    static constexpr int kThreads = 32 * (kRoleWarps + kConsumers);
    static constexpr int kWarpTok = kStageTok / kConsumers;  // tokens of a stage per consumer warp
    static constexpr int kRowBytes = KB * kHeadDim / 8;      // one cached row: 256, 128 or 64 bytes
    static constexpr int kRegion = kStageTok * kRowBytes;    // K (or V) rows of a stage
    static constexpr int kScaleOff = 2 * kRegion;            // K scales, then V scales
    static constexpr int kScaleBytes = kStageTok * 4;        // one stage's scales of K (or V)
    static constexpr int kStageBytes = 2 * kRegion + (kQuant ? 2 * kScaleBytes : 0);
    static_assert(kStageBytes % 1024 == 0, "stages keep the swizzle atoms aligned");
    static_assert(!kQuant || kScaleOff + 2 * kScaleBytes == kStageBytes, "the scales close a quantised stage");
    static_assert(kPageSize % kStageTok == 0, "a stage lies in one page");
    static_assert(kWarpTok % kSub == 0 && kStageTok / kSub < (1 << kStreamBoxKinds), "boxes of a stage");
};

// Shared memory of one CTA. Over quantised pages the consumers hand their
// piece states to the merge warp in a buffer of their own (over bf16 pages
// they write them over the stage they just used, which is large enough), and
// the ring holds as many stages as fit.
template <int R, int KB>
struct Lay {
    using F = Fmt<KB>;
    static constexpr int kStateBytes = F::kQuant ? F::kConsumers * R * kHeadDim * 4 : 0;
    static constexpr int kFixed = kQSlots * 16 * kQRow * 2 + kStateBytes + F::kConsumers * 16 * 8 +
                                  kQSlots * kPieceInts * 4 + 2 * kMergeSlots * kMslotInts * 4 +
                                  (2 * kQSlots + 4 * kMergeSlots + 1) * 8 + 1024;
    static constexpr int kPerStage = F::kStageBytes + 16 + 16 + (F::kQuant ? 0 : F::kConsumers * 16 * 8);
    static constexpr int kFit = (kSmemLimit - kFixed) / kPerStage;
    static constexpr int kStages = F::kQuant ? (kFit < 24 ? kFit : 24) : 6;  // ring depth
    static constexpr int kQ = kStages * F::kStageBytes;              // bf16 [kQSlots][16][kQRow]
    static constexpr int kState = kQ + kQSlots * 16 * kQRow * 2;     // fp32 [warp][R][128] (quantised)
    static constexpr int kMl = kState + kStateBytes;                 // float2 [stage or 1][warp][16]
    static constexpr int kPiece = kMl + (F::kQuant ? 1 : kStages) * F::kConsumers * 16 * 8;  // int32 [kQSlots][16]
    static constexpr int kDesc = kPiece + kQSlots * kPieceInts * 4;  // int32 [kStages][4]
    static constexpr int kMslot = kDesc + kStages * 16;              // int32 [4][8]
    static constexpr int kXslot = kMslot + kMergeSlots * kMslotInts * 4;  // int32 [4][8]
    static constexpr int kBar = kXslot + kMergeSlots * kMslotInts * 4;
    // full, empty [kStages]; qfull, qempty [kQSlots]; mfull, mempty, xfull,
    // xempty [kMergeSlots]; sempty (quantised: the state buffer is free)
    static constexpr int kNumBars = 2 * kStages + 2 * kQSlots + 4 * kMergeSlots + 1;
    static constexpr int kBytes = kBar + kNumBars * 8;
    static_assert(kBytes + 1024 <= kSmemLimit, "shared memory of one CTA");
};

// Shape of one sequence's work; tiles = 0 when it has none.
struct Seq {
    int T, n, tiles, nrb;
};

template <int R>
__device__ __forceinline__ Seq seq_from(const StreamParams &P, int T, int n, bool flag) {
    Seq s{T, n, 0, 0};
    if (n <= 0) return s;
    const int npages = (T + kPageSize - 1) / kPageSize;
    if (n > T || n > P.max_q_len || npages > P.max_pages) {
        if (flag) flag_error(P.err, kErrBitQlen);
        return s;
    }
    s.tiles = (T + kCutTok - 1) / kCutTok;
    s.nrb = (P.G * n + R - 1) / R;
    return s;
}

template <int R>
__device__ __forceinline__ Seq seq_at(const StreamParams &P, int b) {
    if (b >= P.B) return Seq{0, 0, 0, 0};
    return seq_from<R>(P, P.seq_lens[b], P.q_lens[b], false);
}

__device__ __forceinline__ int seg_units(const Seq &s) {
    return s.tiles > 0 ? kSegCost + kUnitsPerTile * s.tiles : 0;
}

__device__ __forceinline__ int seq_units(const StreamParams &P, const Seq &s) {
    return seg_units(s) * P.Hkv * s.nrb;
}

// The cut of the units [0, total) into one contiguous range per CTA: C or
// C + 1 units each (the first `rem` get C + 1), or ranges of kMinUnits units
// (two stages) when there is less work than that, the last CTAs then staying
// idle, so that a piece is never so short that its merge costs more than its
// stream. A range of at least kUnitsPerTile units inside a segment holds a
// tile start, so every CTA between a cut segment's first and last holds a
// piece.
struct Ranges {
    int C, rem;
    __device__ __forceinline__ int begin(int c) const { return c * C + min(c, rem); }
    __device__ __forceinline__ int range_of(int u) const {
        const int big = rem * (C + 1);
        return u < big ? u / (C + 1) : rem + (u - big) / C;
    }
};

__device__ __forceinline__ Ranges make_ranges(int total, int n) {
    const int even = total / n;
    if (even >= kMinUnits) return Ranges{even, total - even * n};
    return Ranges{kMinUnits, 0};
}

__device__ __forceinline__ int ceil_units(int x) { return x <= 0 ? 0 : (x + kUnitsPerTile - 1) / kUnitsPerTile; }

// Warp-wide pass over the lengths: total units and total query tokens. For
// batches of up to 512 sequences it also pulls the first line of every
// block-table row into L1, so that the windows read after the cut is known
// do not wait for DRAM.
template <int R>
__device__ void scan_work(const StreamParams &P, int lane, int &total, int &q_total) {
    total = 0;
    q_total = 0;
    if (P.B <= 512)
        for (int b = lane; b < P.B; b += 32)
            asm volatile("prefetch.global.L1 [%0];" ::"l"(P.block_table + static_cast<int64_t>(b) * P.max_pages));
    int T = lane < P.B ? P.seq_lens[lane] : 0, n = lane < P.B ? P.q_lens[lane] : 0;
#pragma unroll 1
    for (int base = 0; base < P.B; base += 32) {
        const int cT = T, cn = n;
        if (base + 32 < P.B) {  // the next round's lengths are in flight while this one is reduced
            const int b = base + 32 + lane;
            T = b < P.B ? P.seq_lens[b] : 0;
            n = b < P.B ? P.q_lens[b] : 0;
        }
        const Seq s = seq_from<R>(P, cT, cn, true);
        total += static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(seq_units(P, s))));
        q_total += static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(max(0, cn))));
    }
}

// Where a unit falls: the sequence whose units hold it, that sequence's unit
// and query-row offsets and its shape (b = B past the work).
struct Loc {
    int b, ws, qs;
    Seq s;
};

// One pass over the lengths locating units g0 and g1 (g0 <= g1), the same on
// every lane.
template <int R>
__device__ void locate2(const StreamParams &P, int lane, int g0, int g1, Loc &l0, Loc &l1) {
    l0 = Loc{P.B, 0, 0, Seq{0, 0, 0, 0}};
    l1 = l0;
    bool f0 = false, f1 = false;
    int w_base = 0, q_base = 0;
#pragma unroll 1
    for (int base = 0; base < P.B && !f1; base += 32) {
        const int b = base + lane;
        const Seq s = seq_at<R>(P, b);
        const int w = seq_units(P, s), qn = b < P.B ? max(0, s.n) : 0;
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
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const int g = which ? g1 : g0;
            const unsigned hit = __ballot_sync(0xffffffffu, w > 0 && wx <= g && g < wx + w);
            if (hit && !(which ? f1 : f0)) {
                const int src = __ffs(hit) - 1;
                Loc l;
                l.b = base + src;
                l.ws = __shfl_sync(0xffffffffu, wx, src);
                l.qs = __shfl_sync(0xffffffffu, qx, src);
                l.s.T = __shfl_sync(0xffffffffu, s.T, src);
                l.s.n = __shfl_sync(0xffffffffu, s.n, src);
                l.s.tiles = __shfl_sync(0xffffffffu, s.tiles, src);
                l.s.nrb = __shfl_sync(0xffffffffu, s.nrb, src);
                if (which) {
                    l1 = l;
                    f1 = true;
                } else {
                    l0 = l;
                    f0 = true;
                }
            }
        }
        w_base += __shfl_sync(0xffffffffu, wi, 31);
        q_base += __shfl_sync(0xffffffffu, qi, 31);
    }
}

// Bounded wait by a whole warp: true on every lane when the phase completed.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

__device__ __forceinline__ void mbar_arrive_n(uint64_t *bar, uint32_t n) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(n) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// D += A B for one m16n8k16 tile: A 16x16 bf16 (four registers), B 16x8 bf16
// (two registers), D 16x8 fp32.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte address of 16-byte chunk j of row r inside a swizzled 64-column half.
__device__ __forceinline__ uint32_t sw_addr(uint32_t half, int r, int j) {
    return half + r * 128 + (((j ^ r) & 7) << 4);
}

// Byte address of 16-byte chunk j of row r of 64-byte rows with the 64-byte
// swizzle (int4 codes).
__device__ __forceinline__ uint32_t sw64_addr(uint32_t base, int r, int j) {
    return base + r * 64 + (((j ^ (r >> 1)) & 3) << 4);
}

// Bytes of the scales of a stage's n rows: whole 16-byte chunks (the rows
// past n in the chunk lie in the same page and are never used).
__device__ __forceinline__ uint32_t scale_bytes(int n) { return static_cast<uint32_t>((n + 3) / 4 * 16); }

// D += A B for one m16n8k16 tile in fp16 (fp32 accumulate).
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Codes to exact fp16 values. An integer u in [0, 1023] placed in the
// mantissa of 1024 (bits 0x6400 | u) is the fp16 number 1024 + u, so one
// fp16 subtraction leaves u minus the offset exactly.
//  * int8: w holds four codes (two's complement); the sign flip makes them
//    code + 128; lo/hi pick bytes (0, 2) and (1, 3) of w as two fp16 pairs.
__device__ __forceinline__ void i8x4_pairs(uint32_t w, uint32_t sel_lo, uint32_t sel_hi, uint32_t &lo, uint32_t &hi) {
    w ^= 0x80808080u;
    lo = hsub2(prmt(w, 0x64646464u, sel_lo), 0x64806480u);  // - (1024 + 128)
    hi = hsub2(prmt(w, 0x64646464u, sel_hi), 0x64806480u);
}
//  * int4: nibble i of w (code + 8) and nibble i + 4 become one fp16 pair
//    p[i], for i = 0..3. Nibbles 1 and 3 are masked in place (bits 4..7 of a
//    half: 1024 + 16 u), which one fp16 FMA by 1/16 minus 72 brings to u - 8.
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}
__device__ __forceinline__ void i4x8_pairs(uint32_t w, uint32_t (&p)[4]) {
    const uint32_t w8 = w >> 8;
    p[0] = hsub2((w & 0x000F000Fu) | 0x64006400u, 0x64086408u);                // - (1024 + 8)
    p[1] = hfma2((w & 0x00F000F0u) | 0x64006400u, 0x2C002C00u, 0xD480D480u);   // / 16 - 72
    p[2] = hsub2((w8 & 0x000F000Fu) | 0x64006400u, 0x64086408u);
    p[3] = hfma2((w8 & 0x00F000F0u) | 0x64006400u, 0x2C002C00u, 0xD480D480u);
}

__device__ __forceinline__ uint32_t half2_bits(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Consumer warp c's state inside a stage: row r of O (512 bytes) over the
// warp's own 16 rows of the four halves (2 KiB each), four O rows per half,
// word w of row r stored at w ^ 4 (r % 8) (so that the eight rows a store
// instruction touches fall on different banks); its (max, sum) pairs in the
// stage's slot of the pair array.
__device__ __forceinline__ float *state_row(uint8_t *stage, int c, int r) {
    return reinterpret_cast<float *>(stage + (r >> 2) * kHalf + c * (kSub * 128) + (r & 3) * 512);
}
__device__ __forceinline__ float2 *state_ml(float2 *ml, int st, int c, int consumers) {
    return ml + (st * consumers + c) * 16;
}

// Query row fragments (fp16) for the products with codes: the row times the
// softmax scale and a power of two that puts its largest magnitude in [2^13,
// 2^14) (within fp16 range, at full fp16 precision). The head dimensions are
// ordered as the code fragments deliver them: int8, k-step s pairs dims (16 s
// + 4 cq, + 1) and (+ 2, + 3); int4, k-steps 2 c and 2 c + 1 pair dims 32 c +
// 8 cq + (0, 4), (1, 5) and (2, 6), (3, 7). Row sel 0 fills a0/a2, 1 fills
// a1/a3. Returns the factor that undoes the power of two on the scores.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int KB>
__device__ __forceinline__ float quant_q_row(const uint16_t *qrow, int cq, float qscale, uint32_t (&qa)[8][4],
                                             int sel) {
    float amax = 0.f;
    if constexpr (KB == 8) {
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const uint2 w = *reinterpret_cast<const uint2 *>(qrow + 16 * s + 4 * cq);
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf_lo(w.x)), fabsf(bf_hi(w.x))),
                                     fmaxf(fabsf(bf_lo(w.y)), fabsf(bf_hi(w.y)))));
        }
    } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint4 w = *reinterpret_cast<const uint4 *>(qrow + 32 * c + 8 * cq);
            amax = fmaxf(amax, fmaxf(fmaxf(fmaxf(fabsf(bf_lo(w.x)), fabsf(bf_hi(w.x))),
                                           fmaxf(fabsf(bf_lo(w.y)), fabsf(bf_hi(w.y)))),
                                     fmaxf(fmaxf(fabsf(bf_lo(w.z)), fabsf(bf_hi(w.z))),
                                           fmaxf(fabsf(bf_lo(w.w)), fabsf(bf_hi(w.w))))));
        }
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const float m = amax * fabsf(qscale);
    int ex = m > 0.f ? ((__float_as_int(m) >> 23) & 0xff) - 127 : 0;
    ex = min(max(ex, -100), 127);
    const float up = qscale * __int_as_float((127 + 13 - ex) << 23);
    if constexpr (KB == 8) {
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const uint2 w = *reinterpret_cast<const uint2 *>(qrow + 16 * s + 4 * cq);
            qa[s][sel] = half2_bits(bf_lo(w.x) * up, bf_hi(w.x) * up);
            qa[s][2 + sel] = half2_bits(bf_lo(w.y) * up, bf_hi(w.y) * up);
        }
    } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint4 w = *reinterpret_cast<const uint4 *>(qrow + 32 * c + 8 * cq);
            // dims 0..7 of the lane's eight: w.x = (0, 1), w.y = (2, 3), w.z = (4, 5), w.w = (6, 7)
            qa[2 * c][sel] = half2_bits(bf_lo(w.x) * up, bf_lo(w.z) * up);
            qa[2 * c][2 + sel] = half2_bits(bf_hi(w.x) * up, bf_hi(w.z) * up);
            qa[2 * c + 1][sel] = half2_bits(bf_lo(w.y) * up, bf_lo(w.w) * up);
            qa[2 * c + 1][2 + sel] = half2_bits(bf_hi(w.y) * up, bf_hi(w.w) * up);
        }
    }
    return __int_as_float((127 + ex - 13) << 23);
}

// Head dimension of O^T row g (hi = 0) or g + 8 (hi = 1) of 16-dim block m,
// as the products deliver them.
template <int KB>
__device__ __forceinline__ int o_dim(int m, int g, int hi) {
    if constexpr (KB == 16) return 16 * m + g + 8 * hi;
    else if constexpr (KB == 8) return 16 * m + 2 * g + hi;
    else return 32 * (m >> 1) + 4 * g + 2 * (m & 1) + hi;
}

template <int R>
__device__ __forceinline__ int64_t part_row(int sl, int r) {
    return static_cast<int64_t>(sl) * R + r;
}

template <int R, int KB>
__global__ void __launch_bounds__(Fmt<KB>::kThreads, 1)
    stream_attn_kernel(const StreamParams P, const __grid_constant__ StreamMaps maps) {
    using L = Lay<R, KB>;
    using F = Fmt<KB>;
    constexpr int kStages = L::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint16_t *qbuf = reinterpret_cast<uint16_t *>(smem + L::kQ);
    float *sbuf = reinterpret_cast<float *>(smem + L::kState);  // quantised: the consumers' piece states
    int32_t *ring = reinterpret_cast<int32_t *>(smem + L::kPiece);
    float2 *mlbuf = reinterpret_cast<float2 *>(smem + L::kMl);
    int32_t *desc = reinterpret_cast<int32_t *>(smem + L::kDesc);
    int32_t *mslot = reinterpret_cast<int32_t *>(smem + L::kMslot);
    int32_t *xslot = reinterpret_cast<int32_t *>(smem + L::kXslot);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kBar);
    uint64_t *empty = full + kStages;
    uint64_t *qfull = empty + kStages;
    uint64_t *qempty = qfull + kQSlots;
    uint64_t *mfull = qempty + kQSlots;
    uint64_t *mempty = mfull + kMergeSlots;
    uint64_t *xfull = mempty + kMergeSlots;
    uint64_t *xempty = xfull + kMergeSlots;
    uint64_t *sempty = xempty + kMergeSlots;
    const int cta = blockIdx.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], F::kConsumers);
        }
        for (int s = 0; s < kQSlots; ++s) {
            mbar_init(&qfull[s], 1);
            mbar_init(&qempty[s], F::kConsumers);
        }
        for (int s = 0; s < kMergeSlots; ++s) {
            mbar_init(&mfull[s], F::kConsumers);
            mbar_init(&mempty[s], 1);
            mbar_init(&xfull[s], 1);
            mbar_init(&xempty[s], 1);
        }
        mbar_init(sempty, 1);
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ================================================================ producer
        if (lane < 2 * kStreamBoxKinds)
            prefetch_tensormap(lane < kStreamBoxKinds ? &maps.k[lane] : &maps.v[lane - kStreamBoxKinds]);
        int total = 0, q_total = 0;
        scan_work<R>(P, lane, total, q_total);
        uint32_t k = 0;   // stages issued
        uint32_t pc = 0;  // pieces issued
        uint32_t qi = 0;  // pieces whose query rows were requested
        auto finish = [&]() {  // the end marker, after the last stage
            const int s = k % kStages;
            if (!warp_wait(&empty[s], ((k / kStages) & 1) ^ 1)) return false;
            if (lane == 0) {
                desc[s * 4 + 2] = kEnd;
                mbar_arrive(&full[s]);
            }
            return true;
        };
        auto drain = [&]() {  // timeout: wait (bounded) for the copies still in flight
            if (lane == 0) flag_error(P.err, kErrBitTimeout);
            for (uint32_t c = k > kStages ? k - kStages : 0; c < k; ++c)
                (void)mbar_wait(&full[c % kStages], (c / kStages) & 1);
            for (uint32_t c = qi > kQSlots ? qi - kQSlots : 0; c < qi; ++c)
                (void)mbar_wait(&qfull[c % kQSlots], (c / kQSlots) & 1);
        };
        if (q_total > P.total_q) {  // q_lens disagree with dims.total_q: reject the whole call
            if (lane == 0) flag_error(P.err, kErrBitQlen);
            if (!finish()) drain();
            return;
        }
        const Ranges rg = make_ranges(total, P.n_ctas);
        const int gb = min(total, rg.begin(cta));
        const int ge = min(total, rg.begin(cta + 1));
        Loc L0{P.B, 0, 0, Seq{0, 0, 0, 0}}, L1 = L0;
        if (gb < ge) locate2<R>(P, lane, gb, ge - 1, L0, L1);
        const int iseg0 = L0.b < P.B ? (gb - L0.ws) / seg_units(L0.s) : 0;
        const int iseg1 = L1.b < P.B ? (ge - 1 - L1.ws) / seg_units(L1.s) : 0;

        // Block-table entries: two cached windows of 32 consecutive entries of
        // one sequence (lane i holds entry 32w + i); entry A is the one in use.
        int ab = -1, aw = 0, ap = -1, bb = -1, bw = 0, bp = -1;
        auto load_win = [&](int b, int w) -> int {
            const int jj = (w << 5) + lane;
            return (b >= 0 && b < P.B && jj < P.max_pages)
                       ? P.block_table[static_cast<int64_t>(b) * P.max_pages + jj] : -1;
        };
        auto pid_of = [&](int b, int jp) -> int {
            const int w = jp >> 5;
            if (b != ab || w != aw) {
                const int tb = ab, tw = aw, tp = ap;
                if (b == bb && w == bw) {
                    ab = bb; aw = bw; ap = bp;
                } else {
                    ab = b; aw = w; ap = load_win(b, w);
                }
                bb = tb; bw = tw; bp = tp;
            }
            return __shfl_sync(0xffffffffu, ap, jp & 31);
        };
        auto prefetch = [&](int b, int w) {
            if ((b == ab && w == aw) || (b == bb && w == bw)) return;
            bb = b; bw = w; bp = load_win(b, w);
        };
        if (gb < ge) {  // the first windows this CTA needs, in flight before the dependency wait
            const int u1 = L1.ws + iseg1 * seg_units(L1.s);
            const int t1 = ceil_units(gb - u1 - kSegCost) * kCutTok;
            ab = L1.b; aw = (t1 / kPageSize) >> 5; ap = load_win(ab, aw);
            const int u0 = L0.ws + iseg0 * seg_units(L0.s);
            const int t0 = ceil_units(gb - u0 - kSegCost) * kCutTok;
            prefetch(L0.b, (t0 / kPageSize) >> 5);
        }
        const uint64_t policy = P.evict_first ? l2_policy_evict_first() : l2_policy_evict_normal();
        // queries and pages may be written by the kernel before this one
        grid_dependency_wait();

        int last_b = -1;
        bool keep_window = false;  // the next piece's window is already held
        // One piece: tokens [tok_lo, tok_hi) of segment (b, kvh, rb); its
        // partial goes to `slot` and counts at counter f when pieces > 1.
        auto issue_piece = [&](int b, int kvh, int rb, const Seq &s, int qs, int tok_lo, int tok_hi, int pieces,
                               int slot, int f) -> bool {
            // next sequence's first window, while this one streams (after this
            // piece's first stage is issued: the load may first wait for the
            // one before it into the same registers)
            bool want_window = b != last_b && !keep_window;
            keep_window = false;
            last_b = b;
            const int nvr = min(R, P.G * s.n - rb * R);
            // the piece's descriptor now, its query rows after its first stage
            const int qslot = pc % kQSlots;
            if (!warp_wait(&qempty[qslot], ((pc / kQSlots) & 1) ^ 1)) return false;
            if (lane == 0) {
                int32_t *d = ring + qslot * kPieceInts;
                d[0] = b; d[1] = kvh; d[2] = rb; d[3] = s.T; d[4] = s.n; d[5] = qs; d[6] = nvr;
                d[7] = pieces; d[8] = slot; d[9] = f;
            }
            __syncwarp();
            bool want_q = true;
            auto issue_q = [&]() {
                if (lane == 0) mbar_arrive_expect_tx(&qfull[qslot], nvr * 256);
                __syncwarp();
                if (lane < nvr) {  // query row r = rb R + lane: token r / G, head kvh G + r % G
                    const int r = rb * R + lane;
                    const uint16_t *src =
                        P.q + (static_cast<int64_t>(qs + r / P.G) * P.Hq + kvh * P.G + r % P.G) * kHeadDim;
                    bulk_load(qbuf + (qslot * 16 + lane) * kQRow, src, 256, &qfull[qslot]);
                }
                want_q = false;
                ++qi;
            };
            ++pc;
            // the stages: tokens up to the next multiple of 64, so a stage lies in
            // one page; its rows go in at most three boxes per half of K or V
            // (64, 32 and 16 rows: the binary digits of its 16-row count)
            for (int t = tok_lo; t < tok_hi;) {
                const int e = min(tok_hi, (t / F::kStageTok + 1) * F::kStageTok);
                const int st = k % kStages;
                const int pid = pid_of(b, t / kPageSize);
                if (!warp_wait(&empty[st], ((k / kStages) & 1) ^ 1)) return false;
                const bool ok = static_cast<unsigned>(pid) < static_cast<unsigned>(P.num_pages);
                const int n16 = (e - t + kSub - 1) / kSub;  // 16-row chunks per half
                if (lane == 0) {
                    desc[st * 4 + 0] = t;
                    desc[st * 4 + 1] = e - t;
                    desc[st * 4 + 2] = (t == tok_lo ? kFirst : 0) | (e == tok_hi ? kLast : 0) | (ok ? 0 : kSkip);
                    if (ok) {
                        if constexpr (F::kQuant)  // codes of K and V, and their scales
                            mbar_arrive_expect_tx(&full[st], n16 * kSub * 2 * F::kRowBytes + 2 * scale_bytes(e - t));
                        else
                            mbar_arrive_expect_tx(&full[st], n16 * 4 * kBoxBytes);
                    } else {
                        flag_error(P.err, kErrBitPageOOB);
                        mbar_arrive(&full[st]);
                    }
                }
                __syncwarp();
                // lane: box (lane & 7) of half-tensor (lane >> 3): K low and high
                // 64 columns, then V low and high, all in one instruction
                int sel = -1, off = 0;
                {
                    int at = 0, idx = 0;
#pragma unroll
                    for (int m = kStreamBoxKinds - 1; m >= 0; --m) {
                        if (n16 & (1 << m)) {
                            if (idx == (lane & 7)) {
                                sel = m;
                                off = at;
                            }
                            at += 1 << m;
                            ++idx;
                        }
                    }
                }
                if constexpr (F::kQuant) {
                    // lanes 0-2: boxes of K codes, 8-10: of V codes; lanes 16, 17:
                    // the K and V scales of the stage's rows (one bulk copy each)
                    const int row = (pid * P.Hkv + kvh) * kPageSize + (t % kPageSize);
                    if (ok && sel >= 0 && lane < 16) {
                        const int qh = lane >> 3;
                        tma_load_2d(smem + st * F::kStageBytes + qh * F::kRegion + off * kSub * F::kRowBytes,
                                    qh == 0 ? &maps.k[sel] : &maps.v[sel], &full[st], 0, row + off * kSub, policy);
                    }
                    if (ok && (lane == 16 || lane == 17))
                        bulk_load(smem + st * F::kStageBytes + F::kScaleOff + (lane - 16) * F::kScaleBytes,
                                  (lane == 16 ? P.k_scales : P.v_scales) + row, scale_bytes(e - t), &full[st]);
                } else if (ok && sel >= 0) {
                    const int qh = lane >> 3;  // 0, 1: K halves; 2, 3: V halves
                    const int row = (pid * P.Hkv + kvh) * kPageSize + (t % kPageSize) + off * kSub;
                    tma_load_2d(smem + st * F::kStageBytes + qh * kHalf + off * kBoxBytes,
                                qh < 2 ? &maps.k[sel] : &maps.v[sel], &full[st], 64 * (qh & 1), row, policy);
                }
                ++k;
                t = e;
                if (want_q) issue_q();
                if (want_window) {
                    prefetch(b + 1, 0);
                    want_window = false;
                }
            }
            if (want_q) issue_q();  // (a piece has at least one stage)
            return true;
        };
        // One piece of the static range: the part of segment iseg of sequence
        // b (units from ws, query rows from qs) inside [gb, ge).
        auto emit = [&](int b, int iseg, const Seq &s, int ws, int qs) -> bool {
            const int u0 = ws + iseg * seg_units(s);
            const int t_lo = min(s.tiles, ceil_units(gb - u0 - kSegCost));
            const int t_hi = min(s.tiles, ceil_units(ge - u0 - kSegCost));
            if (t_lo >= t_hi) return true;
            const int f = rg.range_of(u0 + kSegCost);
            const int pieces = rg.range_of(u0 + kSegCost + kUnitsPerTile * (s.tiles - 1)) - f + 1;
            const bool head = t_lo == 0 && t_hi < s.tiles;
            return issue_piece(b, iseg / s.nrb, iseg % s.nrb, s, qs, t_lo * kCutTok, min(s.T, t_hi * kCutTok), pieces,
                               2 * cta + (head ? 1 : 0), f);
        };

        bool ok = true;
        if (gb < ge) {
            // 1. the head of the segment shared with the next CTA
            bool rotated = false;
            if (L1.b < P.B && !(L1.b == L0.b && iseg1 == iseg0)) {
                const int u1 = L1.ws + iseg1 * seg_units(L1.s);
                const int t_lo = ceil_units(gb - u1 - kSegCost), t_hi = min(L1.s.tiles, ceil_units(ge - u1 - kSegCost));
                if (t_lo == 0 && t_hi > 0 && t_hi < L1.s.tiles) {
                    rotated = true;
                    keep_window = true;  // the window of L0's sequence, fetched above, comes next
                    ok = emit(L1.b, iseg1, L1.s, L1.ws, L1.qs);
                }
            }
            // 2. everything else, in order
            int b = L0.b, iseg = iseg0, ws = L0.ws, qs = L0.qs;
            Seq s = L0.s;
#pragma unroll 1
            while (ok && b < P.B) {
                if (ws + iseg * seg_units(s) >= ge) break;
                if (!(rotated && b == L1.b && iseg == iseg1)) ok = emit(b, iseg, s, ws, qs);
                if (++iseg == P.Hkv * s.nrb) {
                    iseg = 0;
                    do {
                        ws += seq_units(P, s);
                        qs += max(0, s.n);
                        if (++b >= P.B) break;
                        s = seq_at<R>(P, b);
                    } while (seq_units(P, s) == 0);
                }
            }
        }
        if (!ok || !finish()) drain();
        return;
    }

    if (warp == 1) {
        // ================================================================ merge warp
        // outputs are written after the kernel before this one has completed
        grid_dependency_wait();
        uint32_t xp = 0;  // partials handed to the counting warp
        auto hand_over = [&](int nvr, int qs, int kvh, int rb, int pieces, int f) -> bool {
            const int xs = xp % kMergeSlots;
            if (!warp_wait(&xempty[xs], ((xp / kMergeSlots) & 1) ^ 1)) return false;
            if (lane == 0) {
                int32_t *x = xslot + xs * kMslotInts;
                x[0] = nvr; x[1] = qs; x[2] = kvh; x[3] = rb; x[4] = pieces; x[5] = f;
            }
            __syncwarp();  // the partial writes of every lane precede the hand-over
            if (lane == 0) mbar_arrive(&xfull[xs]);
            ++xp;
            return true;
        };
#pragma unroll 1
        for (uint32_t hp = 0;; ++hp) {
            const int ms = hp % kMergeSlots;
            if (!warp_wait(&mfull[ms], (hp / kMergeSlots) & 1)) {
                if (lane == 0) flag_error(P.err, kErrBitTimeout);
                return;
            }
            const int32_t *m = mslot + ms * kMslotInts;
            const int st = m[0], nvr = m[1], qs = m[2], kvh = m[3], rb = m[4], pieces = m[5], slot = m[6], f = m[7];
            __syncwarp();
            if (lane == 0) mbar_arrive(&mempty[ms]);
            if (st < 0) {  // the consumers are done: so is the counting warp, after the partials before
                if (!hand_over(-1, 0, 0, 0, 0, 0) && lane == 0) flag_error(P.err, kErrBitTimeout);
                return;
            }
            uint8_t *stage = smem + st * F::kStageBytes;
            const bool direct = pieces == 1;
            // each lane owns head dims 4 lane .. 4 lane + 3 of every row; the
            // rows' shared-memory loads are all independent
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (r < nvr) {
                    float2 x[F::kConsumers];
                    float M = -INFINITY;
#pragma unroll
                    for (int c = 0; c < F::kConsumers; ++c) {
                        x[c] = state_ml(mlbuf, F::kQuant ? 0 : st, c, F::kConsumers)[r];
                        if (x[c].y > 0.f) M = fmaxf(M, x[c].x);
                    }
                    float Ls = 0.f;
                    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int c = 0; c < F::kConsumers; ++c) {
                        const float wt = x[c].y > 0.f ? exp2f(x[c].x - M) : 0.f;
                        Ls += x[c].y * wt;
                        const float *srow = F::kQuant ? sbuf + (c * R + r) * kHeadDim : state_row(stage, c, r);
                        const float4 a = reinterpret_cast<const float4 *>(srow)[lane ^ (r & 7)];
                        o.x += a.x * wt;
                        o.y += a.y * wt;
                        o.z += a.z * wt;
                        o.w += a.w * wt;
                    }
                    const int rr = rb * R + r;
                    const int64_t orow = static_cast<int64_t>(qs + rr / P.G) * P.Hq + kvh * P.G + rr % P.G;
                    if (direct) {
                        const float inv = Ls > 0.f ? __frcp_rn(Ls) : 0.f;
                        reinterpret_cast<uint2 *>(P.out + orow * kHeadDim)[lane] =
                            make_uint2(pack_bf16x2(o.x * inv, o.y * inv), pack_bf16x2(o.z * inv, o.w * inv));
                    } else {
                        reinterpret_cast<float4 *>(P.part_acc + part_row<R>(slot, r) * kHeadDim)[lane] = o;
                        if (lane == 0) reinterpret_cast<float2 *>(P.part_ml)[part_row<R>(slot, r)] = make_float2(M, Ls);
                    }
                }
            }
            if constexpr (F::kQuant) {
                // the states are read: the consumers may write the next ones
                __syncwarp();
                if (lane == 0) mbar_arrive(sempty);
            } else {
                // the states are read: the stage may be refilled (the next
                // writes to it are the TMA's)
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive_n(&empty[st], F::kConsumers);
            }
            if (!direct && !hand_over(nvr, qs, kvh, rb, pieces, f)) {
                if (lane == 0) flag_error(P.err, kErrBitTimeout);
                return;
            }
        }
    }

    if (warp == 2) {
        // ============================================================= counting warp
        // Counts the partials of cut segments; the last piece of a segment to
        // finish merges all of them. Its loads go to L2 under a full HBM
        // stream, so they are issued together: every piece's (max, sum) pairs
        // at once, then each piece's accumulator rows at once.
        grid_dependency_wait();
#pragma unroll 1
        for (uint32_t xp = 0;; ++xp) {
            const int xs = xp % kMergeSlots;
            if (!warp_wait(&xfull[xs], (xp / kMergeSlots) & 1)) {
                if (lane == 0) flag_error(P.err, kErrBitTimeout);
                return;
            }
            const int32_t *x = xslot + xs * kMslotInts;
            const int nvr = x[0], qs = x[1], kvh = x[2], rb = x[3], pieces = x[4], f = x[5];
            __syncwarp();
            if (lane == 0) mbar_arrive(&xempty[xs]);
            if (nvr < 0) return;
            // The release orders the merge warp's partial writes (which this
            // warp synchronised with) before the count; the acquire lets the
            // merge below see the other CTAs' partials.
            int old = 0;
            if (lane == 0)
                asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(P.counters + f) : "memory");
            old = __shfl_sync(0xffffffffu, old, 0);
            if (old != pieces - 1) continue;
            // the head in its first CTA's second slot, the rest in their CTAs' first slots
            auto piece_slot = [&](int kk) { return kk == 0 ? 2 * f + 1 : 2 * (f + kk); };
            constexpr int RG = 4;  // rows merged together
#pragma unroll 1
            for (int r0 = 0; r0 < nvr; r0 += RG) {
                float M[RG], Ls[RG];
                float4 o[RG];
#pragma unroll
                for (int i = 0; i < RG; ++i) {
                    M[i] = -INFINITY;
                    Ls[i] = 0.f;
                    o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
                // lane kk holds piece k0 + kk's (max, sum) pairs; those of the
                // first 32 pieces stay in registers for the weights below
                float2 v0[RG];
                for (int k0 = 0; k0 < pieces; k0 += 32) {
                    const int kk = k0 + lane;
#pragma unroll
                    for (int i = 0; i < RG; ++i) {
                        float2 v = make_float2(0.f, 0.f);
                        if (kk < pieces && r0 + i < nvr)
                            v = __ldcg(reinterpret_cast<const float2 *>(P.part_ml) + part_row<R>(piece_slot(kk), r0 + i));
                        if (k0 == 0) v0[i] = v;
                        if (v.y > 0.f) M[i] = fmaxf(M[i], v.x);
                    }
                }
#pragma unroll
                for (int i = 0; i < RG; ++i)
#pragma unroll
                    for (int sh = 16; sh >= 1; sh >>= 1) M[i] = fmaxf(M[i], __shfl_xor_sync(0xffffffffu, M[i], sh));
                for (int k0 = 0; k0 < pieces; k0 += 32) {
                    const int kk = k0 + lane;
                    float wt[RG];
#pragma unroll
                    for (int i = 0; i < RG; ++i) {
                        wt[i] = 0.f;
                        float lw = 0.f;
                        if (kk < pieces && r0 + i < nvr) {
                            const float2 v = k0 == 0 ? v0[i]
                                                     : __ldcg(reinterpret_cast<const float2 *>(P.part_ml) +
                                                              part_row<R>(piece_slot(kk), r0 + i));
                            if (v.y > 0.f) {
                                wt[i] = exp2f(v.x - M[i]);
                                lw = v.y * wt[i];
                            }
                        }
#pragma unroll
                        for (int sh = 16; sh >= 1; sh >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, sh);
                        Ls[i] += lw;
                    }
                    const int cnt = min(32, pieces - k0);
                    // pieces whose rows are loaded together (over codes the
                    // kernel runs 384 threads and has fewer registers to spare)
                    constexpr int PJ = F::kQuant ? 4 : 8;
                    for (int j0 = 0; j0 < cnt; j0 += PJ) {
                        float4 a[PJ][RG];
                        float w[PJ][RG];
#pragma unroll
                        for (int jj = 0; jj < PJ; ++jj)
#pragma unroll
                            for (int i = 0; i < RG; ++i) {
                                const int j = min(j0 + jj, 31);
                                w[jj][i] = j0 + jj < cnt ? __shfl_sync(0xffffffffu, wt[i], j) : 0.f;
                                a[jj][i] = (r0 + i < nvr && w[jj][i] != 0.f)
                                               ? __ldcg(reinterpret_cast<const float4 *>(
                                                            P.part_acc + part_row<R>(piece_slot(k0 + j), r0 + i) * kHeadDim) + lane)
                                               : make_float4(0.f, 0.f, 0.f, 0.f);
                            }
#pragma unroll
                        for (int jj = 0; jj < PJ; ++jj)
#pragma unroll
                            for (int i = 0; i < RG; ++i) {
                                o[i].x += a[jj][i].x * w[jj][i];
                                o[i].y += a[jj][i].y * w[jj][i];
                                o[i].z += a[jj][i].z * w[jj][i];
                                o[i].w += a[jj][i].w * w[jj][i];
                            }
                    }
                }
#pragma unroll
                for (int i = 0; i < RG; ++i) {
                    if (r0 + i < nvr) {
                        const int rr = rb * R + r0 + i;
                        const int64_t orow = static_cast<int64_t>(qs + rr / P.G) * P.Hq + kvh * P.G + rr % P.G;
                        const float inv = Ls[i] > 0.f ? __frcp_rn(Ls[i]) : 0.f;
                        reinterpret_cast<uint2 *>(P.out + orow * kHeadDim)[lane] =
                            make_uint2(pack_bf16x2(o[i].x * inv, o[i].y * inv), pack_bf16x2(o[i].z * inv, o[i].w * inv));
                    }
                }
            }
            if (lane == 0) P.counters[f] = 0;  // ready for the next call
        }
    }
    if (warp < kRoleWarps) return;  // warp 3 has no role

    // ==================================================================== consumers
    const int cw = warp - 4;
    const int g = lane >> 2, cq = lane & 3;  // mma fragment row group and column pair
    // Lane address parts for ldmatrix: matrix index and row within it
    const int lm = lane >> 3, lr = lane & 7;
    const uint32_t smem_base = smem_u32(smem);

    constexpr int NR = R == 16 ? 2 : 1;  // eight-row tiles of the query rows
    uint32_t qa[8][4];   // Q as the A operand, one 16-dim K-step per entry (rows g, g + 8)
    // O transposed: ot[m][nr] is the 16-dim x 8-row tile (dims 16 m .., rows
    // 8 nr ..); lane (g, cq) holds dims 16 m + g (+ 8) of rows 8 nr + 2 cq (+ 1)
    float ot[8][NR][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows g and g + 8
    float qf0 = 1.f, qf1 = 1.f;  // quantised pages: factors that undo the query rows' powers of two
    int lim0 = -1, lim1 = -1;
    int pT = 0, pn = 0, prb = 0, pnvr = 0, pqs = 0, pkvh = 0, ppieces = 1, pslot = 0, pf = 0;
    const float qscale = P.qscale;
    // One step of this warp: NS 16-token sub-tiles (stage st_u, first row
    // tb_u, keys t0_u + tb_u .., of which the first nv_u are valid), as one
    // tile of 16 NS keys with one online-softmax update. Over quantised pages
    // a warp's 32 or 64 tokens of a stage go two sub-tiles at a time, so that
    // their products and conversions overlap (one consumer warp per
    // scheduler leaves nothing else to hide their latency).
    auto consume = [&](auto ns_tag, int stA, int stB, int tbA, int tbB, int t0A, int t0B, int nvA, int nvB) {
        constexpr int NS = decltype(ns_tag)::value;
        constexpr int NT = 2 * NS;  // eight-key tiles
        const int st_u[2] = {stA, stB}, tb_u[2] = {tbA, tbB}, t0_u[2] = {t0A, t0B}, nv_u[2] = {nvA, nvB};
        // ---- S = Q K^T over the 16 NS keys (2 NS N tiles of 8), even and odd
        // K-steps in two chains of accumulators (half the dependent latency),
        // added at the end
        float sacc[NT][4], sodd[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) sacc[nt][e] = sodd[nt][e] = 0.f;
        // quantised pages: matrix j of a four-matrix load is tokens 8 (j & 1)
        // .. + 7 of 16-byte column (j >> 1) of the pair being read
#pragma unroll
        for (int u = 0; u < NS; ++u) {
            const int tb = tb_u[u];
            const int qrow = tb + 8 * (lm & 1) + lr;
            (void)qrow;
            uint8_t *stage = smem + st_u[u] * F::kStageBytes;
            const uint32_t kh0 = smem_base + st_u[u] * F::kStageBytes, kh1 = kh0 + kHalf;
            (void)kh1;
            if (!F::kQuant && nv_u[u] < kSub) {
                // rows past the valid tokens hold whatever the page held: zero
                // their V so that 0 x (stale) cannot be NaN (codes are
                // integers, and their probabilities are zeroed before the V
                // scales multiply them)
                for (int i = lane; i < (kSub - nv_u[u]) * 16; i += 32) {
                    const int rr = tb + nv_u[u] + i / 16, ch = i % 16;
                    *reinterpret_cast<uint4 *>(stage + 2 * kHalf + (ch >> 3) * kHalf + rr * 128 + (ch & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                __syncwarp();
            }
            if constexpr (KB == 8) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {  // k-steps 2 i, 2 i + 1 (one column each)
                    uint32_t r[4];
                    ldsm_x4(sw_addr(kh0, qrow, 2 * i + (lm >> 1)), r[0], r[1], r[2], r[3]);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t b0, b1;
                        i8x4_pairs(r[j], 0x4140u, 0x4342u, b0, b1);
                        mma_f16((j >> 1) ? sodd[2 * u + (j & 1)] : sacc[2 * u + (j & 1)], qa[2 * i + (j >> 1)], b0, b1);
                    }
                }
            } else if constexpr (KB == 4) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {  // columns 2 i, 2 i + 1: k-steps 4 i .. 4 i + 3
                    uint32_t r[4];
                    ldsm_x4(sw64_addr(kh0, qrow, 2 * i + (lm >> 1)), r[0], r[1], r[2], r[3]);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int c = 2 * i + (j >> 1);
                        uint32_t x[4];
                        i4x8_pairs(r[j], x);
                        mma_f16(sacc[2 * u + (j & 1)], qa[2 * c], x[0], x[1]);
                        mma_f16(sodd[2 * u + (j & 1)], qa[2 * c + 1], x[2], x[3]);
                    }
                }
            } else {
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint32_t half = s < 4 ? kh0 : kh1;
                    const int row = tb + 8 * (lm >> 1) + lr;
                    uint32_t b00, b01, b10, b11;
                    ldsm_x4(sw_addr(half, row, 2 * (s & 3) + (lm & 1)), b00, b01, b10, b11);
                    mma_bf16((s & 1) ? sodd[2 * u] : sacc[2 * u], qa[s], b00, b01);
                    mma_bf16((s & 1) ? sodd[2 * u + 1] : sacc[2 * u + 1], qa[s], b10, b11);
                }
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) sacc[nt][e] += sodd[nt][e];
        // quantised pages: the scales of this lane's keys (tb + 8 n + 2 cq, + 1),
        // K's at the stage's scale area, V's after them
        float2 ks[NT], vs[NT];
        (void)ks;
        (void)vs;
        if constexpr (F::kQuant) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float *scl = reinterpret_cast<const float *>(smem + st_u[nt >> 1] * F::kStageBytes + F::kScaleOff);
                const int key = tb_u[nt >> 1] + 8 * (nt & 1) + 2 * cq;
                ks[nt] = *reinterpret_cast<const float2 *>(scl + key);
                vs[nt] = *reinterpret_cast<const float2 *>(scl + F::kStageTok + key);
            }
        }
        // ---- online softmax on rows g (and g + 8), log2 units
        float x[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int kl = 8 * (nt & 1) + 2 * cq + (e & 1);  // key within the sub-tile
                const int lim = e < 2 ? lim0 : lim1;
                float sc = qscale;
                if constexpr (F::kQuant) sc = ((e & 1) ? ks[nt].y : ks[nt].x) * (e < 2 ? qf0 : qf1);
                x[nt][e] = (kl < nv_u[nt >> 1] && t0_u[nt >> 1] + tb_u[nt >> 1] + kl <= lim) ? sacc[nt][e] * sc : -INFINITY;
            }
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mx0 = fmaxf(mx0, fmaxf(x[nt][0], x[nt][1]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        if constexpr (R == 16) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mx1 = fmaxf(mx1, fmaxf(x[nt][2], x[nt][3]));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        }
        // the reference max only moves when the tile max beats it by 2^8
        const bool grow0 = mx0 > m0 + 8.f, grow1 = mx1 > m1 + 8.f;
        if (__any_sync(0xffffffffu, grow0 || grow1)) {
            const float a0 = grow0 ? exp2f(m0 - mx0) : 1.f;  // 0 when m was -inf
            const float a1 = grow1 ? exp2f(m1 - mx1) : 1.f;
            if (grow0) m0 = mx0;
            if (grow1) m1 = mx1;
            l0 *= a0;
            l1 *= a1;
            // this lane's O rows are 2 cq and 2 cq + 1 (of each row tile),
            // whose factors the lanes of row groups 2 cq and 2 cq + 1 hold
            const float r0a = __shfl_sync(0xffffffffu, a0, 8 * cq), r1a = __shfl_sync(0xffffffffu, a0, 8 * cq + 4);
            const float r0b = __shfl_sync(0xffffffffu, a1, 8 * cq), r1b = __shfl_sync(0xffffffffu, a1, 8 * cq + 4);
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                ot[m][0][0] *= r0a;
                ot[m][0][1] *= r1a;
                ot[m][0][2] *= r0a;
                ot[m][0][3] *= r1a;
                if constexpr (NR == 2) {
                    ot[m][1][0] *= r0b;
                    ot[m][1][1] *= r1b;
                    ot[m][1][2] *= r0b;
                    ot[m][1][3] *= r1b;
                }
            }
        }
        const float mu0 = m0 == -INFINITY ? 0.f : m0, mu1 = m1 == -INFINITY ? 0.f : m1;
        (void)mu1;
        float p[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            p[nt][0] = exp2f(x[nt][0] - mu0);
            p[nt][1] = exp2f(x[nt][1] - mu0);
            l0 += p[nt][0] + p[nt][1];
            if constexpr (R == 16) {
                p[nt][2] = exp2f(x[nt][2] - mu1);
                p[nt][3] = exp2f(x[nt][3] - mu1);
                l1 += p[nt][2] + p[nt][3];
            } else {
                p[nt][2] = p[nt][3] = 0.f;
            }
        }
        // O^T += V^T P^T: P is the B operand (16 keys x 8 rows) straight from
        // the S accumulators, per sub-tile; V^T the A operand (16 dims x 16
        // keys) by transposing loads
        uint32_t pb[NS][NR][2];
#pragma unroll
        for (int u = 0; u < NS; ++u) {
            if constexpr (F::kQuant) {
                // P times the V scales (fp16); a zero probability stays zero
                // whatever the scale of its row
                float pv[2][4];
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 v = vs[2 * u + n];
                        pv[n][e] = p[2 * u + n][e] > 0.f ? p[2 * u + n][e] * ((e & 1) ? v.y : v.x) : 0.f;
                    }
                pb[u][0][0] = half2_bits(pv[0][0], pv[0][1]);
                pb[u][0][1] = half2_bits(pv[1][0], pv[1][1]);
                if constexpr (NR == 2) {
                    pb[u][1][0] = half2_bits(pv[0][2], pv[0][3]);
                    pb[u][1][1] = half2_bits(pv[1][2], pv[1][3]);
                }
            } else {
                pb[u][0][0] = pack_bf16x2(p[2 * u][0], p[2 * u][1]);
                pb[u][0][1] = pack_bf16x2(p[2 * u + 1][0], p[2 * u + 1][1]);
                if constexpr (NR == 2) {
                    pb[u][1][0] = pack_bf16x2(p[2 * u][2], p[2 * u][3]);
                    pb[u][1][1] = pack_bf16x2(p[2 * u + 1][2], p[2 * u + 1][3]);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < NS; ++u) {
            const uint32_t kh0 = smem_base + st_u[u] * F::kStageBytes;
            const int qrow = tb_u[u] + 8 * (lm & 1) + lr;
            (void)qrow;
            if constexpr (KB == 8) {
                // V codes by transposing loads: matrix j holds tokens 8 (j & 1) ..
                // of 16-dim block 2 i + (j >> 1); a lane's word is two tokens x
                // dims (2 g, 2 g + 1), so O^T row g is dim 2 g, row g + 8 dim 2 g + 1
                const uint32_t vq = kh0 + F::kRegion;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint32_t r[4];
                    ldsm_x4_t(sw_addr(vq, qrow, 2 * i + (lm >> 1)), r[0], r[1], r[2], r[3]);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t va[4];
                        i8x4_pairs(r[2 * h], 0x4240u, 0x4341u, va[0], va[1]);
                        i8x4_pairs(r[2 * h + 1], 0x4240u, 0x4341u, va[2], va[3]);
#pragma unroll
                        for (int nr = 0; nr < NR; ++nr) mma_f16(ot[2 * i + h][nr], va, pb[u][nr][0], pb[u][nr][1]);
                    }
                }
            } else if constexpr (KB == 4) {
                // int4: a lane's word is two tokens x dims 4 g .. 4 g + 3 of a
                // 32-dim column; block 2 c takes dims 4 g, 4 g + 1, block 2 c + 1
                // dims 4 g + 2, 4 g + 3
                const uint32_t vq = kh0 + F::kRegion;
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    uint32_t r[4];
                    ldsm_x4_t(sw64_addr(vq, qrow, 2 * i + (lm >> 1)), r[0], r[1], r[2], r[3]);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int c = 2 * i + h;
                        uint32_t xa[4], xb[4];
                        i4x8_pairs(r[2 * h], xa);
                        i4x8_pairs(r[2 * h + 1], xb);
                        const uint32_t va[4] = {xa[0], xa[1], xb[0], xb[1]};
                        const uint32_t vb[4] = {xa[2], xa[3], xb[2], xb[3]};
#pragma unroll
                        for (int nr = 0; nr < NR; ++nr) {
                            mma_f16(ot[2 * c][nr], va, pb[u][nr][0], pb[u][nr][1]);
                            mma_f16(ot[2 * c + 1][nr], vb, pb[u][nr][0], pb[u][nr][1]);
                        }
                    }
                }
            } else {
                const uint32_t vh0 = kh0 + 2 * kHalf, vh1 = kh0 + 3 * kHalf;
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const uint32_t half = m < 4 ? vh0 : vh1;
                    const int row = tb_u[u] + 8 * (lm >> 1) + lr;
                    uint32_t va[4];
                    ldsm_x4_t(sw_addr(half, row, 2 * (m & 3) + (lm & 1)), va[0], va[1], va[2], va[3]);
#pragma unroll
                    for (int nr = 0; nr < NR; ++nr) mma_bf16(ot[m][nr], va, pb[u][nr][0], pb[u][nr][1]);
                }
            }
        }
    };
    uint32_t k = 0, pc = 0;
#pragma unroll 1
    while (true) {
        const int st = k % kStages;
        if (!warp_wait(&full[st], (k / kStages) & 1)) {
            if (lane == 0) flag_error(P.err, kErrBitTimeout);
            return;
        }
        const int t0 = desc[st * 4 + 0], ntok = desc[st * 4 + 1], flags = desc[st * 4 + 2];
        if (flags & kEnd) {
            // hand the end over to the merge warp
            const int ms = pc % kMergeSlots;
            if (!warp_wait(&mempty[ms], ((pc / kMergeSlots) & 1) ^ 1)) {
                if (lane == 0) flag_error(P.err, kErrBitTimeout);
                return;
            }
            if (cw == 0 && lane == 0) mslot[ms * kMslotInts] = -1;
            __syncwarp();
            if (lane == 0) mbar_arrive(&mfull[ms]);
            return;
        }
        if (flags & kFirst) {
            // a new piece: its descriptor, then its queries as A fragments
            const int qslot = pc % kQSlots;
            const int32_t *d = ring + qslot * kPieceInts;
            pkvh = d[1]; prb = d[2]; pT = d[3]; pn = d[4]; pqs = d[5]; pnvr = d[6];
            ppieces = d[7]; pslot = d[8]; pf = d[9];
            if (!warp_wait(&qfull[qslot], (pc / kQSlots) & 1)) {
                if (lane == 0) flag_error(P.err, kErrBitTimeout);
                return;
            }
            // rows past nvr hold stale data; their scores are masked
            if constexpr (F::kQuant) {
                const uint16_t *qrows = qbuf + qslot * 16 * kQRow;
                qf0 = quant_q_row<KB>(qrows + g * kQRow, cq, qscale, qa, 0);
                if constexpr (R == 16) {
                    qf1 = quant_q_row<KB>(qrows + (g + 8) * kQRow, cq, qscale, qa, 1);
                } else {
#pragma unroll
                    for (int s = 0; s < 8; ++s) qa[s][1] = qa[s][3] = 0u;
                }
            } else {
                const uint32_t *qw = reinterpret_cast<const uint32_t *>(qbuf + qslot * 16 * kQRow);
                constexpr int kQW = kQRow / 2;  // words per query row
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    qa[s][0] = qw[g * kQW + 8 * s + cq];
                    qa[s][2] = qw[g * kQW + 8 * s + 4 + cq];
                    if constexpr (R == 16) {
                        qa[s][1] = qw[(g + 8) * kQW + 8 * s + cq];
                        qa[s][3] = qw[(g + 8) * kQW + 8 * s + 4 + cq];
                    } else {
                        qa[s][1] = 0u;
                        qa[s][3] = 0u;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&qempty[qslot]);
#pragma unroll
            for (int m = 0; m < 8; ++m)
#pragma unroll
                for (int nr = 0; nr < NR; ++nr) ot[m][nr][0] = ot[m][nr][1] = ot[m][nr][2] = ot[m][nr][3] = 0.f;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
            lim0 = g < pnvr ? pT - pn + (prb * R + g) / P.G : -1;  // last key of each row
            lim1 = (R == 16 && g + 8 < pnvr) ? pT - pn + (prb * R + g + 8) / P.G : -1;
        }
        // this warp's sub-tiles of the stage: rows cw W .. cw W + W - 1, one at a
        // time (the two consumer warps of a scheduler overlap each other)
        constexpr int kNS = 1;
        const int nvw = (flags & kSkip) ? 0 : ntok - cw * F::kWarpTok;  // its valid tokens
#pragma unroll 1
        for (int j = 0; j < F::kWarpTok && j < nvw; j += kNS * kSub) {
            const int tb = cw * F::kWarpTok + j;
            const int nvA = min(kSub, nvw - j);
            if constexpr (kNS == 2)
                consume(std::integral_constant<int, 2>{}, st, st, tb, tb + kSub, t0, t0, nvA, max(0, min(kSub, nvw - j - kSub)));
            else
                consume(std::integral_constant<int, 1>{}, st, st, tb, tb, t0, t0, nvA, 0);
        }
        uint8_t *stage = smem + st * F::kStageBytes;
        if (flags & kLast) {
            // ---- end of the piece: hand the state to the merge warp
            l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
            l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
            const int ms = pc % kMergeSlots;
            if (!warp_wait(&mempty[ms], ((pc / kMergeSlots) & 1) ^ 1)) {
                if (lane == 0) flag_error(P.err, kErrBitTimeout);
                return;
            }
            // quantised pages: the state buffer, once the merge warp has read
            // the previous piece's states from it
            if (F::kQuant && !warp_wait(sempty, (pc & 1) ^ 1)) {
                if (lane == 0) flag_error(P.err, kErrBitTimeout);
                return;
            }
            __syncwarp();  // every lane of this warp is done reading its rows of the stage
#pragma unroll
            for (int nr = 0; nr < NR; ++nr)
#pragma unroll
                for (int e2 = 0; e2 < 2; ++e2) {
                    const int row = 8 * nr + 2 * cq + e2;
                    if (row < pnvr) {
                        float *dst = F::kQuant ? sbuf + (cw * R + row) * kHeadDim : state_row(stage, cw, row);
#pragma unroll
                        for (int m = 0; m < 8; ++m) {
                            dst[o_dim<KB>(m, g, 0) ^ (4 * (row & 7))] = ot[m][nr][e2];
                            dst[o_dim<KB>(m, g, 1) ^ (4 * (row & 7))] = ot[m][nr][2 + e2];
                        }
                    }
                }
            float2 *mlw = state_ml(mlbuf, F::kQuant ? 0 : st, cw, F::kConsumers);
            if (g < pnvr && cq == 0) mlw[g] = make_float2(m0, l0);
            if (R == 16 && g + 8 < pnvr && cq == 0) mlw[g + 8] = make_float2(m1, l1);
            // the state was written by this (generic) proxy; the next writes to
            // the stage, after the merge warp releases it, are the TMA's
            if constexpr (!F::kQuant) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            if (cw == 0 && lane == 0) {
                int32_t *m = mslot + ms * kMslotInts;
                m[0] = st; m[1] = pnvr; m[2] = pqs; m[3] = pkvh; m[4] = prb; m[5] = ppieces; m[6] = pslot; m[7] = pf;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&mfull[ms]);
            if (F::kQuant && lane == 0) mbar_arrive(&empty[st]);  // the stage itself is free now
            ++pc;
        } else {
            // zeroed V rows were written by this (generic) proxy; the next
            // writes to the stage are the TMA's
            if (!F::kQuant && nvw > 0 && nvw < kSub) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
        }
        ++k;
    }
}

template <int R, int KB>
constexpr size_t smem_bytes() { return Lay<R, KB>::kBytes + 1024; }

template <int R, int KB>
cudaError_t launch_r(const StreamParams &p, const StreamMaps &maps, cudaStream_t stream) {
    static const cudaError_t attr = cudaFuncSetAttribute(
        stream_attn_kernel<R, KB>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_bytes<R, KB>()));
    if (attr != cudaSuccess) return attr;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(p.n_ctas));
    cfg.blockDim = dim3(Fmt<KB>::kThreads);
    cfg.dynamicSmemBytes = smem_bytes<R, KB>();
    cfg.stream = stream;
    // a programmatic dependent of the kernel before it: the work scan and the
    // first block-table reads overlap that kernel's end (sa_kv_append allows
    // it); queries and pages are read, and outputs written, after the
    // dependency wait
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, stream_attn_kernel<R, KB>, p, maps);
}

}  // namespace

int stream_units_per_tile() { return kUnitsPerTile; }
int stream_segment_cost() { return kSegCost; }
int stream_tile_tokens() { return kCutTok; }
int stream_box_rows() { return kSub; }

template <int KB>
cudaError_t launch_kb(const StreamParams &p, const StreamMaps &maps, cudaStream_t stream) {
    switch (p.R) {
        case 4: return launch_r<4, KB>(p, maps, stream);
        case 8: return launch_r<8, KB>(p, maps, stream);
        case 16: return launch_r<16, KB>(p, maps, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_stream_attn(const StreamParams &p, const StreamMaps &maps, cudaStream_t stream) {
    switch (p.code_bits) {
        case 16: return launch_kb<16>(p, maps, stream);
        case 8: return launch_kb<8>(p, maps, stream);
        case 4: return launch_kb<4>(p, maps, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sa
