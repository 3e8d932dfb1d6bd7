// prefix_tc.cu -- shared-prefix attention on the tcgen05 tensor cores.
//
// ExLlamaV2 "Dynamic Generator" page, "Deduplication": many sequences index
// the same physical pages for a common prefix. Attention over such a run of
// pages is one dense contraction: the query rows of every member sequence
// (G heads x its new tokens, all for one KV head) against the run's keys and
// values. This kernel streams each shared 64-token K/V tile from HBM once per
// 128-row tile of queries (row tiles of one run share their tiles through L2)
// and computes
//     S = Q K^T          (tcgen05.mma, bf16 x bf16 -> fp32 in tensor memory)
//     P = exp2(S*scale*log2e - m)  online, one thread per row, bf16 to smem
//     O += P V           (tcgen05.mma, fp32 accumulator in tensor memory)
// and stores, per row, an fp32 partial (O, m, l) that the combine kernel merges
// with the rest of the sequence's keys.
//
// CTA = 11 warps: warps 0-7 softmax and epilogue, two per tensor-memory lane
// quadrant (warp w reads lanes [32 (w % 4), +32), the same scheduler's lanes
// for both), which take alternate K/V tiles of a piece, each with its own
// running max and O buffer, merged at the piece's end; warp 8 the TMA
// producer, warp 9 allocates tensor memory and issues Q K^T, warp 10 issues
// P V (one thread each). K/V tiles of 64 keys
// (32 KiB) stream through five stages, so four loads are in flight while a
// tile is consumed; S (tensor memory, four buffers) and P (shared memory, two,
// one per half) are multi-buffered, so Q K^T runs up to three tiles ahead and
// P V of one half's tile runs on the tensor cores while the other half's
// softmax runs on the CUDA cores. With at most 32 query rows (q_len = k+1
// verification of one sequence) every row is held four times and each copy's
// softmax (warps 0-3) takes a quarter of a tile's keys. Operands sit in shared
// memory in the 128-byte-swizzled K-major layout the TMA writes (Q, K and P)
// or the MN-major one (V), described to the tensor core by shared-memory
// matrix descriptors. Every wait is bounded; on timeout the CTA flags
// SA_ERR_TIMEOUT, drains what it issued and frees its tensor memory.
#include <cuda_bf16.h>

#include <type_traits>

#include "common.cuh"
#include "plan.h"
#include "tc_work.cuh"

namespace sa {

namespace {

constexpr int kM = 128;                       // rows per tile (tensor-memory lanes)
constexpr int kN = 64;                        // keys per K/V tile
constexpr int kRowBlk = kM * 128;             // one 64-wide bf16 column block of 128 rows: 16 KiB
constexpr int kKVBlk = kN * 128;              // one 64-wide bf16 column block of a K or V tile: 8 KiB
constexpr int kQBytes = 2 * kRowBlk;          // Q [128 rows][128 d]
constexpr int kPBytes = kRowBlk;              // P [128 rows][64 keys], double-buffered
constexpr int kKVStage = 4 * kKVBlk;          // K (2 blocks) + V (2 blocks) = 32 KiB
constexpr int kStagesTC = 5;                  // K/V stages
constexpr int kSBufs = 4;                     // S buffers: Q K^T runs up to three tiles ahead of the softmax
constexpr int kTmemCols = 512;                // S buffers: columns 0 .. 4*64-1, two O buffers: the next 2*128
static_assert(kSBufs * 64 + 2 * 128 <= kTmemCols, "tensor-memory columns");
// softmax / epilogue warps (4 or 8), then the TMA producer, the Q K^T issuer
// (which also holds the tensor memory) and the P V issuer
constexpr int tc_threads(int soft_warps) { return (soft_warps + 3) * 32; }

constexpr int kOffQ = 0;
constexpr int kOffP = kOffQ + kQBytes;
constexpr int kOffKV = kOffP + 2 * kPBytes;
constexpr int kOffBar = kOffKV + kStagesTC * kKVStage;
constexpr int kOffML = kOffBar + 320;             // epilogue of four copies: (max, sum) of the 128 lanes
constexpr int kOffStart = kOffML + kM * 2 * 4;    // sequence mode: where this CTA's range starts
constexpr int kSmemBytes = kOffStart + 128 + 1024;  // + alignment slack

static_assert(kN == kTcKeyTile && kM == kTcRowTile, "tile shapes shared with the combine pass");
static_assert(kSmemBytes <= 227 * 1024, "shared memory of one CTA");
// barriers: K/V full and empty, Q, S full and free, P full and free, O free,
// all MMAs done, the tensor-memory address and abort flag, four exchanges, P V
// done, Q loaded by TMA, Q read by the piece's Q K^T
static_assert((2 * kStagesTC + 1 + 2 * kSBufs + 2 + 2 + 2 + 1 + 2 + 4 + 1 + 2) * 8 <= kOffML - kOffBar, "barrier space");
static_assert(kOffML + 2 * kM * 4 <= kOffStart, "the (max, sum) pairs of the copies' epilogue fit their space");

// ------------------------------------------------------------ tcgen05 helpers
// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor for kind::f16: fp32 accumulate, bf16 A and B, A
// K-major, B K-major or MN-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_bf16(bool b_mn_major, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn_major ? (1u << 16) : 0u) |
           (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(kM >> 4) << 24);
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

// Paired fp32 fused multiply-add: (a.x * b.x + c.x, a.y * b.y + c.y), one instruction.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    unsigned long long ra = *reinterpret_cast<unsigned long long *>(&a);
    unsigned long long rb = *reinterpret_cast<unsigned long long *>(&b);
    unsigned long long rc = *reinterpret_cast<unsigned long long *>(&c);
    unsigned long long rd;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
    return *reinterpret_cast<float2 *>(&rd);
}

// max(a, b, c) in one instruction (exact, like two fmaxf).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// 2^x by the special-function unit's approximation, results below the
// smallest normal flushed to zero (a probability that small adds nothing
// to a row sum of at least 1).
__device__ __forceinline__ float ex2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

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

// N consecutive 32-bit columns (16, 32 or 64) of this thread's lane, one wait.
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float *v) {
    uint32_t r[N];
    if constexpr (N == 16) {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
            : "r"(taddr));
    } else {
#pragma unroll
        for (int h = 0; h < N / 32; ++h)
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                : "=r"(r[32 * h + 0]), "=r"(r[32 * h + 1]), "=r"(r[32 * h + 2]), "=r"(r[32 * h + 3]),
                  "=r"(r[32 * h + 4]), "=r"(r[32 * h + 5]), "=r"(r[32 * h + 6]), "=r"(r[32 * h + 7]),
                  "=r"(r[32 * h + 8]), "=r"(r[32 * h + 9]), "=r"(r[32 * h + 10]), "=r"(r[32 * h + 11]),
                  "=r"(r[32 * h + 12]), "=r"(r[32 * h + 13]), "=r"(r[32 * h + 14]), "=r"(r[32 * h + 15]),
                  "=r"(r[32 * h + 16]), "=r"(r[32 * h + 17]), "=r"(r[32 * h + 18]), "=r"(r[32 * h + 19]),
                  "=r"(r[32 * h + 20]), "=r"(r[32 * h + 21]), "=r"(r[32 * h + 22]), "=r"(r[32 * h + 23]),
                  "=r"(r[32 * h + 24]), "=r"(r[32 * h + 25]), "=r"(r[32 * h + 26]), "=r"(r[32 * h + 27]),
                  "=r"(r[32 * h + 28]), "=r"(r[32 * h + 29]), "=r"(r[32 * h + 30]), "=r"(r[32 * h + 31])
                : "r"(taddr + 32 * h));
    }
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = __uint_as_float(r[i]);
}

// 3-D tiled TMA load (coordinates innermost first) completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar, int32_t x, int32_t y,
                                            int32_t z, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

struct PrefixParams {
    const uint16_t *q;
    const int32_t *block_table;
    // plan mode: work items and rows from a shared-run plan (one item per CTA)
    const int32_t *run_desc;
    const int32_t *run_rows;
    const int32_t *tiles;
    // sequence mode: the cut of the tile sequence (tc_work.cuh), one range per CTA
    const int32_t *seq_lens;
    const int32_t *q_lens;
    int32_t seq_mode, B, max_q_len, total_q, min_rows;
    float *ws_acc;
    float *ws_ml;
    uint16_t *out;  // sequence mode: output of the segments attended whole (waves)
    int32_t *err;
    int32_t Hq, Hkv, G, max_pages, num_pages;
    int64_t n_rows_total;
    float qscale;  // scale * log2(e)
    int32_t q_tma;  // sequence mode: pieces held once per row load Q by TMA (3-D map: d, head, token)
};

// A piece: the tiles of one segment that this CTA attends.
struct TcPiece {
    int member;                       // block-table row whose pages are read
    int g;                            // KV head
    int row0, row_count, rows_begin;  // rows [row0, min(row0 + 128, row_count)) of the segment
    int pc_lo;                        // page of tile 0
    int t_lo, t_hi;                   // 64-key tiles [t_lo, t_hi) counted from page pc_lo
    int key_end;                      // keys at or past this position are not in the cache
    int seq_n, qstart;                // sequence mode: new tokens, packed row of the first
    int slot;                         // sequence mode: partial slot; plan mode: page chunk
    int whole;                        // sequence mode: a whole segment of a wave (output written here)
    int qbox;                         // plan mode: first token of the rows' query box, or -1
};

// Start of this CTA's range in sequence mode, found by warp 0 and shared:
// its waves of whole segments, then its range of the cut (units counted from
// the start of the work; the cut's own units from waves.base).
struct TcStart {
    int has_work, b, qstart, seg, tile, unit, end;
    TcRanges rg;
    TcWaves waves;
};

// The walk over the pieces of this CTA's range (sequence mode); every role
// runs its own copy and they see the same pieces.
struct TcCursor {
    int b, qstart, seg, tile, unit, end, T, n;
    TcSeq w;
    TcRanges rg;
    TcWaves waves;
    int wave;

    __device__ __forceinline__ void load(const PrefixParams &P) {
        T = P.seq_lens[b];
        n = P.q_lens[b];
        w = tc_seq(T, n, P.G, P.Hkv, P.max_q_len, P.max_pages, P.min_rows);
    }
    __device__ __forceinline__ void init(const PrefixParams &P, const TcStart &s) {
        b = s.b;
        qstart = s.qstart;
        seg = s.seg;
        tile = s.tile;
        unit = s.unit;
        end = s.end;
        rg = s.rg;
        waves = s.waves;
        wave = 0;
        if (unit < end) load(P);
    }
    __device__ __forceinline__ bool next(const PrefixParams &P, TcPiece &pc) {
        if (wave < waves.waves) {  // whole segment wave * grid + this CTA, its only piece
            const int sg = wave * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x);
            const int bb = sg / waves.seg_per_seq, ss = sg % waves.seg_per_seq;
            const int Tb = P.seq_lens[bb], nb = P.q_lens[bb];
            const TcSeq wb = tc_seq(Tb, nb, P.G, P.Hkv, P.max_q_len, P.max_pages, P.min_rows);
            pc.member = bb;
            pc.g = ss / wb.mtiles;
            pc.row0 = (ss % wb.mtiles) * kTcRowTile;
            pc.row_count = P.G * nb;
            pc.rows_begin = 0;
            pc.pc_lo = 0;
            pc.t_lo = 0;
            pc.t_hi = wb.tiles;
            pc.key_end = Tb;
            pc.seq_n = nb;
            pc.qstart = bb * nb;  // every sequence has nb new tokens
            pc.slot = 0;
            pc.whole = 1;
            pc.qbox = -1;
            ++wave;
            return true;
        }
        if (unit >= end) return false;
        const int mt = seg % w.mtiles;
        pc.member = b;
        pc.g = seg / w.mtiles;
        pc.row0 = mt * kTcRowTile;
        pc.row_count = P.G * n;
        pc.rows_begin = 0;
        pc.pc_lo = 0;
        pc.t_lo = tile;
        pc.t_hi = min(w.tiles, tile + (end - unit));
        pc.key_end = T;
        pc.seq_n = n;
        pc.qstart = qstart;
        pc.slot = static_cast<int>(blockIdx.x) - rg.range_of(unit - tile - waves.base);
        pc.whole = 0;
        pc.qbox = -1;
        unit += pc.t_hi - tile;
        tile = pc.t_hi;
        if (tile == w.tiles && unit < end) {  // the next segment (of the next tensor-core sequence)
            tile = 0;
            if (++seg == P.Hkv * w.mtiles) {
                seg = 0;
                do {
                    qstart += max(0, n);
                    ++b;
                    load(P);
                } while (w.units == 0 && b + 1 < P.B);
            }
        }
        return true;
    }
};

// Epilogue of a piece held four times (sequence mode, at most 32 rows; run
// by the four warps of half 0, thread t on tensor-memory lane t, with o_lane
// its lane's O address): in two halves of 64 columns staged in the P
// buffers (idle until the next piece's softmax), every lane stages its half
// row, then thread t merges 16 columns of row t % 32 over the copies and
// writes the row's fp32 partial.
__device__ __forceinline__ void merge_copies(uint8_t *smem, int t, int rpc, const TcPiece &pc, uint32_t o_lane,
                                          float m_ref, float lsum, float *ws_acc, float *ws_ml,
                                          int64_t n_rows_total, int Hq, int G) {
    float *ost = reinterpret_cast<float *>(smem + kOffP);  // [128 lanes][64], 16-byte chunks xor-swizzled
    float *mls = reinterpret_cast<float *>(smem + kOffML);
    mls[2 * t] = m_ref;
    mls[2 * t + 1] = lsum;
    const int rl = t % rpc, q4 = t / rpc;
    const int rr = pc.row0 + rl;
    float M = -INFINITY, L = 0.f, wgt[4];
    int64_t wi = 0;
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            float o[32];
            tmem_ld32(o_lane + h * 64 + c * 32, o);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                *reinterpret_cast<float4 *>(ost + t * 64 + (((c * 8 + k) ^ (t & 7)) * 4)) =
                    make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");  // the four warps of half 0 only
        if (rr < pc.row_count) {
            if (h == 0) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (mls[2 * (c * rpc + rl) + 1] > 0.f) M = fmaxf(M, mls[2 * (c * rpc + rl)]);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float lc = mls[2 * (c * rpc + rl) + 1];
                    wgt[c] = lc > 0.f ? exp2f(mls[2 * (c * rpc + rl)] - M) : 0.f;
                    L += lc * wgt[c];
                }
                const int64_t tk = pc.qstart + rr / G;
                wi = static_cast<int64_t>(pc.slot) * n_rows_total + tk * Hq + pc.g * G + rr % G;
                if (q4 == 0) *reinterpret_cast<float2 *>(ws_ml + wi * 2) = make_float2(M, L);
            }
            float4 o[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) o[k] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (wgt[c] > 0.f) {
                    const int ln = c * rpc + rl;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float4 v = *reinterpret_cast<const float4 *>(ost + ln * 64 + (((q4 * 4 + k) ^ (ln & 7)) * 4));
                        o[k].x += v.x * wgt[c];
                        o[k].y += v.y * wgt[c];
                        o[k].z += v.z * wgt[c];
                        o[k].w += v.w * wgt[c];
                    }
                }
            }
            float4 *dst = reinterpret_cast<float4 *>(ws_acc + wi * kHeadDim + h * 64 + q4 * 16);
#pragma unroll
            for (int k = 0; k < 4; ++k) dst[k] = o[k];
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");  // staging read before it is rewritten
    }
}

// The same, out of line: with eight softmax warps (168 registers a thread)
// its registers would otherwise weigh on the softmax loop.
__device__ __noinline__ void merge_copies_call(uint8_t *smem, int t, int rpc, const TcPiece &pc, uint32_t o_lane,
                                               float m_ref, float lsum, float *ws_acc, float *ws_ml,
                                               int64_t n_rows_total, int Hq, int G) {
    merge_copies(smem, t, rpc, pc, o_lane, m_ref, lsum, ws_acc, ws_ml, n_rows_total, Hq, G);
}

template <int kSoftWarps>
__global__ void __launch_bounds__(tc_threads(kSoftWarps), 1)
    prefix_tc_kernel(const PrefixParams P, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmq) {
    constexpr int kSoft = kSoftWarps * 32;
    constexpr int kWarpTMA = kSoftWarps, kWarpQK = kSoftWarps + 1;
    // with eight softmax warps the two of a lane quadrant take alternate tiles
    // of a piece held once per row, each into its own O buffer; with four, O is
    // double-buffered by piece (an epilogue overlaps the next piece's P V)
    constexpr bool kTwo = kSoftWarps == 8;
    static_assert(kSoftWarps == 4 || kSoftWarps == 8, "one or two softmax warps per lane quadrant");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint64_t *kv_full = bars;                   // [kStagesTC] K/V tile landed
    uint64_t *kv_empty = bars + kStagesTC;      // [kStagesTC] K/V stage free again
    uint64_t *q_full = bars + 2 * kStagesTC;    // Q rows of a piece written
    uint64_t *s_full = q_full + 1;              // [kSBufs] S buffer holds Q K^T of a tile
    uint64_t *p_full = s_full + kSBufs;         // [2] P buffer written (and its S buffer read)
    uint64_t *p_free = p_full + 2;              // [2] P V of that buffer finished (O up to date with it)
    uint64_t *o_free = p_free + 2;              // [2] piece p's epilogue read the O buffers: o_free[p & 1]
    uint64_t *s_free = o_free + 2;              // [kSBufs] S buffer read by the softmax
    uint64_t *mma_done = s_free + kSBufs;       // every MMA of both issuers finished
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(mma_done + 1);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(mma_done + 2);
    uint64_t *xbar = mma_done + 3;              // [4] both halves of a lane quadrant posted (max, sum)
    uint64_t *pv_done = mma_done + 7;           // every P V of a piece finished (one phase per piece)
    uint64_t *q_tma = mma_done + 8;             // Q rows of a piece landed by TMA (one phase per such piece)
    uint64_t *q_free = mma_done + 9;            // every Q K^T of a piece finished (one phase per piece)
    TcStart *start = reinterpret_cast<TcStart *>(smem + kOffStart);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    // the split kernel that follows reads nothing this kernel writes (the
    // combine pass reads the partials after both grids), so it may start on
    // SMs this grid leaves free
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // ---- the work: plan mode, this CTA's item; sequence mode, this CTA's range
    TcPiece plan_piece{};
    if (!P.seq_mode) {  // (run, KV head, 128-row tile, page chunk) from the plan
        const int32_t *it = P.tiles + static_cast<int64_t>(blockIdx.x) * kTileInts;
        const int32_t *rd = P.run_desc + static_cast<int64_t>(it[0]) * kRunDescInts;
        plan_piece.member = rd[5];
        plan_piece.g = it[1];
        plan_piece.row0 = it[2];
        plan_piece.row_count = rd[3];
        plan_piece.rows_begin = rd[2];
        plan_piece.pc_lo = it[3];
        plan_piece.t_lo = 0;
        plan_piece.t_hi = ((it[4] - it[3]) * kPageSize + kN - 1) / kN;
        plan_piece.key_end = 0x7fffffff;
        plan_piece.slot = it[5];
        plan_piece.qbox = it[6];
    } else if (warp == 0) {
        // lane-per-sequence scan: the total work, the longest segment, the queries
        int total = 0, max_tiles = 0, q_total = 0;
        bool uniform = P.B > 0;  // every sequence: the same length and query count, and work
        const int T0 = P.B > 0 ? P.seq_lens[0] : 0, n0 = P.B > 0 ? P.q_lens[0] : 0;
#pragma unroll 1
        for (int base = 0; base < P.B; base += 32) {
            const int b = base + lane;
            const int T = b < P.B ? P.seq_lens[b] : 0, n = b < P.B ? P.q_lens[b] : 0;
            const TcSeq w = tc_seq(T, n, P.G, P.Hkv, P.max_q_len, P.max_pages, P.min_rows);
            total += __reduce_add_sync(0xffffffffu, static_cast<unsigned>(w.units));
            max_tiles = max(max_tiles, static_cast<int>(__reduce_max_sync(0xffffffffu, static_cast<unsigned>(w.tiles))));
            q_total += __reduce_add_sync(0xffffffffu, static_cast<unsigned>(max(0, n)));
            uniform = uniform && __all_sync(0xffffffffu, b >= P.B || (T == T0 && n == n0 && w.units > 0));
        }
        const TcWaves waves = make_tc_waves(uniform, P.B, tc_seq(T0, n0, P.G, P.Hkv, P.max_q_len, P.max_pages, P.min_rows),
                                            P.Hkv, gridDim.x, P.G * n0);
        const int total_cut = total - waves.base;  // the cut's units, after the waves
        const TcRanges rg = make_tc_ranges(total_cut, gridDim.x, max_tiles);
        const int c_begin = waves.base + rg.begin(blockIdx.x);
        const int c_end = waves.base + min(total_cut, rg.begin(blockIdx.x + 1));
        const bool valid_q = q_total <= P.total_q;  // else the split kernel flags the lengths
        int has = valid_q && c_begin < c_end;
        int fb = 0, fq = 0, fu = 0;
        if (has && waves.waves > 0) {  // uniform sequences: the start by arithmetic
            const int su = waves.seg_per_seq * tc_seq(T0, n0, P.G, P.Hkv, P.max_q_len, P.max_pages, P.min_rows).tiles;
            fb = c_begin / su;
            fu = fb * su;
            fq = fb * n0;
        } else if (has) {  // the sequence whose units hold c_begin
            int u_base = 0, q_base = 0;
            has = 0;
#pragma unroll 1
            for (int base = 0; base < P.B && !has; base += 32) {
                const int b = base + lane;
                const int T = b < P.B ? P.seq_lens[b] : 0, n = b < P.B ? P.q_lens[b] : 0;
                const int u = tc_seq(T, n, P.G, P.Hkv, P.max_q_len, P.max_pages, P.min_rows).units;
                const int qn = max(0, n);
                int ui = u, qi = qn;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int a = __shfl_up_sync(0xffffffffu, ui, o), c = __shfl_up_sync(0xffffffffu, qi, o);
                    if (lane >= o) {
                        ui += a;
                        qi += c;
                    }
                }
                const int ux = u_base + ui - u, qx = q_base + qi - qn;
                const unsigned hit = __ballot_sync(0xffffffffu, u > 0 && ux <= c_begin && c_begin < ux + u);
                if (hit) {
                    const int src = __ffs(hit) - 1;
                    fb = base + src;
                    fu = __shfl_sync(0xffffffffu, ux, src);
                    fq = __shfl_sync(0xffffffffu, qx, src);
                    has = 1;
                }
                u_base += __shfl_sync(0xffffffffu, ui, 31);
                q_base += __shfl_sync(0xffffffffu, qi, 31);
            }
        }
        if (lane == 0) {
            start->has_work = has || (valid_q && waves.waves > 0);
            start->rg = rg;
            start->waves = waves;
            start->unit = start->end = 0;  // no range of the cut unless set below
            if (has) {
                const TcSeq w = tc_seq(P.seq_lens[fb], P.q_lens[fb], P.G, P.Hkv, P.max_q_len, P.max_pages, P.min_rows);
                const int off = c_begin - fu;
                start->b = fb;
                start->qstart = fq;
                start->seg = off / w.tiles;
                start->tile = off % w.tiles;
                start->unit = c_begin;
                start->end = c_end;
            }
        }
    }
    if (P.seq_mode) {
        __syncthreads();
        if (!start->has_work) return;  // uniform over the CTA: nothing allocated yet
    }
    auto first_piece = [&](TcCursor &cur, TcPiece &pc) -> bool {
        if (!P.seq_mode) {
            pc = plan_piece;
            return true;
        }
        cur.init(P, *start);
        return cur.next(P, pc);
    };
    auto next_piece = [&](TcCursor &cur, TcPiece &pc) -> bool { return P.seq_mode && cur.next(P, pc); };
    // a sequence-mode piece held once per row (more than 32 rows), or a plan
    // item whose rows are consecutive tokens with their G heads, takes its Q
    // rows as one box of the 3-D map (tokens x G heads x d): the Q K^T issuer
    // loads it; other pieces' rows are copied by the softmax warps
    auto q_by_tma = [&](const TcPiece &pc) -> bool {
        return P.q_tma && (P.seq_mode ? pc.row_count - pc.row0 > kM / 4 : pc.qbox >= 0);
    };

    if (tid == 0) {
        for (int s = 0; s < kStagesTC; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        mbar_init(q_full, kSoft);
        for (int b = 0; b < kSBufs; ++b) mbar_init(&s_full[b], 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&p_full[b], kM);  // the 128 lanes of the half attending the tile
            mbar_init(&p_free[b], 1);
            mbar_init(&o_free[b], kSoft);
        }
        for (int b = 0; b < kSBufs; ++b) mbar_init(&s_free[b], kM);
        mbar_init(mma_done, 2);
        for (int q = 0; q < 4; ++q) mbar_init(&xbar[q], 64);
        mbar_init(pv_done, 1);
        mbar_init(q_tma, 1);
        mbar_init(q_free, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kWarpQK) {  // tensor memory for S and O
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
    const uint32_t tmem_o0 = tmem + kSBufs * kN;  // S buffers at columns 0, kN, 2 kN, 3 kN; O buffers A and B after them

    const uint32_t sQ = smem_u32(smem + kOffQ), sP = smem_u32(smem + kOffP), sKV = smem_u32(smem + kOffKV);

    if (warp < kSoftWarps) {
        // ================= softmax / epilogue warps. Warp w reads tensor-memory
        // lanes [32 (w % 4), +32) (lane t holds row slot t). In pieces with one
        // copy per row the two warps of a lane quadrant (the same scheduler)
        // take alternate tiles: half h = w / 4 attends the piece's tiles
        // t_lo + h, t_lo + h + 2, ... with its own running max and sum, into
        // its own O buffer, so that one warp's exponentials overlap the other's
        // waits; the two halves merge at the end of the piece. With at most 32
        // rows in a piece, every row is held by four lanes, one in each warp
        // of half 0 (the Q tile holds four copies of the rows), and copy c
        // takes keys [16c, 16c + 16) of every tile; half 1 then has no rows.
        // The P rows of a copy are zero outside its keys, so P V sums each
        // copy's keys into its own lanes of O, with its own running max; the
        // epilogue merges the four copies.
        const int t = (warp & 3) * 32 + lane;
        const int hf = warp >> 2;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        bool ok = true;
        uint64_t *xb = &xbar[warp & 3];  // the two halves posted their (max, sum) at a piece's end
        uint32_t xe = 0;                  // such exchanges so far
        // P buffer b = i & 1 is free again once P V of tile i - 2 has run;
        // that P V is the ((i - 2) >> 1)-th commit on p_free[b]
        auto wait_pv = [&](int j) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(&p_free[j & 1], (j >> 1) & 1));
        };
        // the rows of a piece that lane t holds
        struct RowMap {
            int rf, rpc, cp, r;
            bool valid, warp_valid;
            int32_t token, hl, limit, slot;
        };
        auto row_of = [&](const TcPiece &pc, int rr, int32_t &token, int32_t &hl, int32_t &limit, int32_t &slot) {
            if (!P.seq_mode) {
                const int32_t *rrow = P.run_rows + static_cast<int64_t>(pc.rows_begin + rr) * 4;
                token = rrow[0];
                hl = rrow[1];
                limit = rrow[2];
                slot = rrow[3] + pc.slot;
            } else {
                token = pc.qstart + rr / P.G;
                hl = rr % P.G;
                limit = pc.key_end - pc.seq_n + rr / P.G;
                slot = pc.slot;
            }
        };
        auto map_rows = [&](const TcPiece &pc) -> RowMap {
            RowMap m{};
            m.rf = (P.seq_mode && pc.row_count - pc.row0 <= kM / 4) ? 4 : 1;  // copies per row
            m.rpc = kM / m.rf;                                               // rows per copy
            m.cp = t / m.rpc;
            m.r = pc.row0 + t % m.rpc;
            m.valid = m.r < pc.row_count && (m.rf == 1 || hf == 0);
            m.warp_valid = __any_sync(0xffffffffu, m.valid);  // warps without rows skip the softmax
            m.token = 0;
            m.hl = 0;
            m.limit = -1;
            m.slot = 0;
            if (m.valid) row_of(pc, m.r, m.token, m.hl, m.limit, m.slot);
            return m;
        };
        // the piece's Q rows -> shared memory, 128-byte swizzled K-major (two
        // 64-column blocks), one copy per row group; every Q K^T of the
        // previous piece has completed. The softmax threads copy the rows
        // together with 16-byte asynchronous copies (16 threads per row:
        // thread s takes column chunk s % 16 of rows s / 16 + 16k, for every
        // copy of the row), all of a thread's copies in flight at once, then
        // wait for them. Lanes past the piece's rows keep whatever they hold:
        // their S, P and O lanes are never read for output.
        auto write_q = [&](const TcPiece &pc, const RowMap &m) {
            const int nrow = min(m.rpc, pc.row_count - pc.row0);
            const int c = tid & 15;
            for (int rr = tid >> 4; rr < nrow; rr += kSoft / 16) {
                int32_t tk, hh, lim, sl;
                row_of(pc, pc.row0 + rr, tk, hh, lim, sl);
                const uint16_t *src = P.q + (static_cast<int64_t>(tk) * P.Hq + pc.g * P.G + hh) * kHeadDim + c * 8;
                for (int cp = 0; cp < m.rf; ++cp)
                    cp_async16(smem + kOffQ + (c >> 3) * kRowBlk + sw128_offset(cp * m.rpc + rr, c & 7), src);
            }
            asm volatile("cp.async.wait_all;" ::: "memory");
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(q_full);
        };
        // Pieces held four times need their P rows at zero outside each copy's
        // keys: half 0 clears both buffers before such a piece, when every
        // P V of the previous piece has completed (with one copy per row, a
        // valid row writes all its keys and an invalid one feeds only O lanes
        // that are never read).
        auto zero_p = [&]() {
            if (hf != 0) return;
#pragma unroll
            for (int c = 0; c < kN / 8; ++c) {
                *reinterpret_cast<uint4 *>(smem + kOffP + sw128_offset(t, c)) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4 *>(smem + kOffP + kPBytes + sw128_offset(t, c)) = make_uint4(0, 0, 0, 0);
            }
        };
        int i = 0;  // tile index over all pieces of this CTA
        int p = 0;  // piece index
        const bool pos_scale = P.qscale > 0.f;
        const float qs = pos_scale ? P.qscale : 1.f;  // the scale applied in the exponent
        TcCursor cur;
        TcPiece pc;
        bool more = first_piece(cur, pc);
        RowMap rm = map_rows(pc);
        if (rm.rf == 4) zero_p();
        if (!q_by_tma(pc)) write_q(pc, rm);
        while (more && ok) {
            // the next piece, found now: its lengths load while this piece's tiles run
            TcPiece nx{};
            const bool has_next = next_piece(cur, nx);
            float m_ref = -INFINITY, lsum = 0.f;
            bool began = false;  // this lane's O buffer holds a tile of the piece
            auto softmax_tiles = [&](auto kpc_tag) {
                constexpr int KPC = decltype(kpc_tag)::value;  // keys of a tile this lane takes
                constexpr bool ONE = KPC == kN;                 // one copy per row
                constexpr bool ALT = ONE && kTwo;               // ... and the halves alternate tiles
                const int koff = ONE ? 0 : rm.cp * KPC;
                const uint32_t tmem_o = kTwo ? tmem_o0 + (ALT ? hf * kHeadDim : 0) : tmem_o0 + (p & 1) * kHeadDim;
                if (!ONE && hf == 1) {  // four copies: half 0 attends every tile
                    i += pc.t_hi - pc.t_lo;
                    return;
                }
                for (int tt = pc.t_lo; tt < pc.t_hi && ok; ++tt, ++i) {
                    if (ALT && ((tt - pc.t_lo) & 1) != hf) continue;  // the other half's tile
                    ok = __all_sync(0xffffffffu, mbar_wait(&s_full[i % kSBufs], (i / kSBufs) & 1));
                    if (!ok) break;
                    tc_fence_after();
                    const int pos0 = pc.pc_lo * kPageSize + tt * kN;
                    uint8_t *pbuf = smem + kOffP + (i & 1) * kPBytes;
                    uint8_t *vstage = smem + kOffKV + (i % kStagesTC) * kKVStage + 2 * kKVBlk;
                    // keys past the end may hold stale data: their V rows are zeroed
                    const bool zero_v = t < kN && pos0 + t >= pc.key_end;
                    if (!rm.warp_valid) {
                        tc_fence_before();
                        mbar_arrive(&s_free[i % kSBufs]);
                        // arrivals on p_full[i & 1] must not run ahead of the phase that
                        // tile i - 2 completes there: wait, like the rows with data do,
                        // until P V of tile i - 2 (which follows that phase) is done
                        if (i >= 2) {
                            ok = wait_pv(i - 2);
                            if (!ok) break;
                        }
                        if (zero_v) {
#pragma unroll
                            for (int c = 0; c < 8; ++c) {
                                *reinterpret_cast<uint4 *>(vstage + t * 128 + c * 16) = make_uint4(0, 0, 0, 0);
                                *reinterpret_cast<uint4 *>(vstage + kKVBlk + t * 128 + c * 16) = make_uint4(0, 0, 0, 0);
                            }
                        }
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        tc_fence_before();
                        mbar_arrive(&p_full[i & 1]);
                        continue;
                    }
                    float x[KPC];
                    tmem_ld_cols<KPC>(tmem + (i % kSBufs) * kN + koff + lane_base, x);
                    tc_fence_before();
                    mbar_arrive(&s_free[i % kSBufs]);  // Q K^T of tile i + kSBufs may overwrite it
                    // Scores stay unscaled: with a positive scale the row max of the
                    // raw scores, scaled once, is the max of the scaled scores, and
                    // the scale enters each probability's exponent through one paired
                    // FMA. Any other scale multiplies the scores first (qs = 1).
                    if (!pos_scale) {
#pragma unroll
                        for (int k = 0; k < KPC; ++k) x[k] *= P.qscale;
                    }
                    if (pos0 + kN - 1 > rm.limit) {  // a diagonal tile: keys past the row's limit are masked
#pragma unroll
                        for (int k = 0; k < KPC; ++k)
                            if (pos0 + koff + k > rm.limit) x[k] = -INFINITY;
                    }
                    // row max as a tree of three-input maxima (independent partial
                    // maxima, short dependency chains)
                    float mx[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) mx[k] = x[k];
#pragma unroll
                    for (int k = 8; k < KPC; k += 16)
#pragma unroll
                        for (int c = 0; c < 8; ++c) mx[c] = fmax3(mx[c], x[k + c], k + 8 + c < KPC ? x[k + 8 + c] : x[k + c]);
                    const float tmax = qs * fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], fmax3(mx[4], mx[5], mx[6]), mx[7]));
                    // move the reference max only when it grows by more than 2^8, so
                    // that tensor-memory O is rarely rescaled (p stays below 256)
                    const bool grow = tmax > m_ref + 8.f;
                    const float m_new = grow ? tmax : m_ref;
                    const float alpha = grow ? exp2f(m_ref - m_new) : 1.f;  // 0 when m_ref was -inf
                    const float m_use = m_new == -INFINITY ? 0.f : m_new;
                    // probabilities, packed to bf16 pairs while the tensor cores run P V
                    uint32_t pw[KPC / 2];
                    float2 ps[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) ps[k] = make_float2(0.f, 0.f);
#pragma unroll
                    for (int k = 0; k < KPC / 2; ++k) {
                        const float2 e = fma2(make_float2(x[2 * k], x[2 * k + 1]), make_float2(qs, qs),
                                              make_float2(-m_use, -m_use));
                        const float2 ab = make_float2(ex2_ftz(e.x), ex2_ftz(e.y));
                        ps[k & 3] = fma2(ab, make_float2(1.f, 1.f), ps[k & 3]);
                        pw[k] = pack_bf16x2(ab.x, ab.y);
                    }
                    const float psum = ((ps[0].x + ps[0].y) + (ps[1].x + ps[1].y)) + ((ps[2].x + ps[2].y) + (ps[3].x + ps[3].y));
                    // P V of tile i - 2 must be done before its P buffer is rewritten;
                    // with alternate tiles it is also the last P V into this half's O
                    if (i >= 2) {
                        ok = wait_pv(i - 2);
                        if (!ok) break;
                    }
                    if (began && __any_sync(0xffffffffu, grow)) {  // O must hold every earlier P V into it
                        if (!ALT) {
                            ok = wait_pv(i - 1);
                            if (!ok) break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int c = 0; c < kHeadDim / 32; ++c) {
                            float o[32];
                            tmem_ld32(tmem_o + lane_base + c * 32, o);
#pragma unroll
                            for (int k = 0; k < 32; ++k) o[k] *= alpha;
                            tmem_st32(tmem_o + lane_base + c * 32, o);
                        }
                    }
                    began = true;
                    lsum = lsum * alpha + psum;
                    m_ref = m_new;
                    // this lane's keys of P row t -> shared memory (bf16, 128-byte swizzled K-major)
#pragma unroll
                    for (int c = 0; c < KPC / 8; ++c)
                        *reinterpret_cast<uint4 *>(pbuf + sw128_offset(t, koff / 8 + c)) =
                            make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
                    if (zero_v) {
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            *reinterpret_cast<uint4 *>(vstage + t * 128 + c * 16) = make_uint4(0, 0, 0, 0);
                            *reinterpret_cast<uint4 *>(vstage + kKVBlk + t * 128 + c * 16) = make_uint4(0, 0, 0, 0);
                        }
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    tc_fence_before();
                    mbar_arrive(&p_full[i & 1]);
                }
            };
            if (rm.rf == 4) softmax_tiles(std::integral_constant<int, kN / 4>{});
            else softmax_tiles(std::integral_constant<int, kN>{});
            // every P V of the piece: a per-piece barrier, since a half may have
            // skipped the piece's last tiles (a parity wait on p_free is only
            // sound one phase ahead of what this thread has seen complete)
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(pv_done, p & 1));
            // One copy per row: the halves trade (max, sum) through the P buffers,
            // idle now. Half h's next tile goes to buffer (i + h) & 1: each posts
            // into the buffer its partner writes next and reads from its own, so
            // that neither post is overwritten before it is read.
            float m_o = -INFINITY, l_o = 0.f;  // the other half's
            if (kTwo && ok && rm.rf == 1 && rm.warp_valid) {
                reinterpret_cast<float2 *>(smem + kOffP + ((i + 1 + hf) & 1) * kPBytes)[t] = make_float2(m_ref, lsum);
                mbar_arrive(xb);
                ok = __all_sync(0xffffffffu, mbar_wait(xb, xe & 1));
                ++xe;
                const float2 v = reinterpret_cast<const float2 *>(smem + kOffP + ((i + hf) & 1) * kPBytes)[t];
                m_o = v.x;
                l_o = v.y;
            }
            if (!ok) {
                *abort_flag = 1;
                if (lane == 0) flag_error(P.err, kErrBitTimeout);
                break;
            }
            tc_fence_after();
            // the next piece's queries first, so that its Q K^T runs during this epilogue
            RowMap rn{};
            if (has_next) {
                rn = map_rows(nx);
                if (!q_by_tma(nx)) write_q(nx, rn);
            }
            if (rm.rf == 1) {
                if (rm.warp_valid) {
                    // the row's two halves (max, sum, O) merged; this half writes
                    // columns [64 hf, 64 hf + 64). A half's O holds data only once
                    // it attended a tile (its sum may still be 0 if every key of
                    // its tiles is masked for the row; its O is then 0).
                    const float mA = (kTwo && hf == 1) ? m_o : m_ref, lA = (kTwo && hf == 1) ? l_o : lsum;
                    const float mB = !kTwo ? -INFINITY : hf == 0 ? m_o : m_ref;
                    const float lB = !kTwo ? 0.f : hf == 0 ? l_o : lsum;
                    const float M = fmaxf(lA > 0.f ? mA : -INFINITY, lB > 0.f ? mB : -INFINITY);
                    const float wA = lA > 0.f ? exp2f(mA - M) : 0.f;
                    const float wB = lB > 0.f ? exp2f(mB - M) : 0.f;
                    const float L = lA * wA + lB * wB;
                    const int64_t orow = static_cast<int64_t>(rm.token) * P.Hq + pc.g * P.G + rm.hl;
                    const float inv = L > 0.f ? __frcp_rn(L) : 0.f;
                    const int64_t wi = static_cast<int64_t>(rm.slot) * P.n_rows_total + orow;
                    const uint32_t o_a = kTwo ? tmem_o0 : tmem_o0 + (p & 1) * kHeadDim;
#pragma unroll
                    // 16 columns at a time with two O buffers (fewer live registers
                    // under the 168-register cap), 32 with one
                    constexpr int CW = kTwo ? 16 : 32;
#pragma unroll 1
                    for (int c = 0; c < (kTwo ? kHeadDim / 2 : kHeadDim) / CW; ++c) {
                        const int col = (kTwo ? hf * (kHeadDim / 2) : 0) + c * CW;
                        float oa[CW];
                        tmem_ld_cols<CW>(o_a + lane_base + col, oa);
                        if constexpr (kTwo) {
                            float ob[CW];
                            tmem_ld_cols<CW>(tmem_o0 + kHeadDim + lane_base + col, ob);
#pragma unroll
                            for (int k = 0; k < CW; ++k) oa[k] = wB > 0.f ? fmaf(ob[k], wB, oa[k] * wA) : oa[k] * wA;
                        } else {
#pragma unroll
                            for (int k = 0; k < CW; ++k) oa[k] *= wA;
                        }
                        if (rm.valid && pc.whole) {  // a whole segment: this row's bf16 output
                            uint4 *dst = reinterpret_cast<uint4 *>(P.out + orow * kHeadDim + col);
#pragma unroll
                            for (int k = 0; k < CW / 8; ++k)
                                dst[k] = make_uint4(pack_bf16x2(oa[8 * k] * inv, oa[8 * k + 1] * inv),
                                                    pack_bf16x2(oa[8 * k + 2] * inv, oa[8 * k + 3] * inv),
                                                    pack_bf16x2(oa[8 * k + 4] * inv, oa[8 * k + 5] * inv),
                                                    pack_bf16x2(oa[8 * k + 6] * inv, oa[8 * k + 7] * inv));
                        } else if (rm.valid) {  // fp32 partial (O, m, l) of this row
                            float4 *dst = reinterpret_cast<float4 *>(P.ws_acc + wi * kHeadDim + col);
#pragma unroll
                            for (int k = 0; k < CW / 4; ++k) dst[k] = make_float4(oa[4 * k], oa[4 * k + 1], oa[4 * k + 2], oa[4 * k + 3]);
                        }
                    }
                    if (rm.valid && !pc.whole && hf == 0) *reinterpret_cast<float2 *>(P.ws_ml + wi * 2) = make_float2(M, L);
                }
            } else if (hf == 0) {
                if constexpr (kTwo)
                    merge_copies_call(smem, t, rm.rpc, pc, tmem_o0 + lane_base, m_ref, lsum, P.ws_acc, P.ws_ml,
                                      P.n_rows_total, P.Hq, P.G);
                else
                    merge_copies(smem, t, rm.rpc, pc, tmem_o0 + (p & 1) * kHeadDim + lane_base, m_ref, lsum, P.ws_acc,
                                 P.ws_ml, P.n_rows_total, P.Hq, P.G);
            }
            tc_fence_before();
            mbar_arrive(&o_free[p & 1]);  // this piece's O buffers may be overwritten
            if (kTwo && ((rm.rf == 4 && hf == 1) || (has_next && rn.rf == 4 && hf == 0))) {
                // half 1 waits for half 0's staged epilogue (it uses the P buffers
                // and the (max, sum) space) before the next piece; half 0 clears both
                // P buffers for a piece held four times once half 1 has read its post
                ok = __all_sync(0xffffffffu, mbar_wait(&o_free[p & 1], (p >> 1) & 1));
                if (!ok) {
                    *abort_flag = 1;
                    if (lane == 0) flag_error(P.err, kErrBitTimeout);
                    break;
                }
            }
            if (!has_next) break;
            if (rn.rf == 4) zero_p();
            pc = nx;
            rm = rn;
            ++p;
        }
    } else if (warp == kWarpTMA) {
        // ================= TMA producer
        if (lane == 0) {
            // plan mode: the row tiles of a chunk re-read its tiles; waves: the
            // CTAs of a wave re-read each other's tiles; otherwise a tile is read
            // by one CTA
            const uint64_t policy = !P.seq_mode             ? l2_policy_evict_last()
                                    : start->waves.waves > 0 ? l2_policy_evict_normal()
                                                             : l2_policy_evict_first();
            int i = 0;
            bool ok = true;
            TcCursor cur;
            TcPiece pc;
            for (bool more = first_piece(cur, pc); more && ok; more = next_piece(cur, pc)) {
                if (P.seq_mode && i > 0) {
                    // the softmax warps load this piece's query rows when the previous
                    // piece ends; bring them into L2 now, while that piece still runs
                    const int k_hi = min(pc.seq_n, (pc.row0 + kM + P.G - 1) / P.G);
                    for (int k = pc.row0 / P.G; k < k_hi; ++k)
                        bulk_prefetch_l2(P.q + (static_cast<int64_t>(pc.qstart + k) * P.Hq + pc.g * P.G) * kHeadDim,
                                         P.G * kHeadDim * 2);
                }
                for (int tt = pc.t_lo; tt < pc.t_hi; ++tt, ++i) {
                    const int s = i % kStagesTC;
                    if (i >= kStagesTC && !mbar_wait(&kv_empty[s], ((i / kStagesTC) - 1) & 1)) {
                        *abort_flag = 1;
                        flag_error(P.err, kErrBitTimeout);
                        ok = false;
                        break;
                    }
                    if (*abort_flag) {
                        ok = false;
                        break;
                    }
                    const int page = pc.pc_lo + tt / (kPageSize / kN);
                    const int pid = P.block_table[static_cast<int64_t>(pc.member) * P.max_pages + page];
                    // (the last tile may reach past the sequence's keys; the rows past
                    // the end are zeroed in shared memory before P V)
                    uint8_t *dst = smem + kOffKV + s * kKVStage;
                    if (pid < 0 || pid >= P.num_pages) {
                        flag_error(P.err, kErrBitPageOOB);
                        mbar_arrive(&kv_full[s]);
                    } else {
                        const int y = (pid * P.Hkv + pc.g) * kPageSize + (tt % (kPageSize / kN)) * kN;
                        mbar_arrive_expect_tx(&kv_full[s], kKVStage);
                        tma_load_2d(dst, &tmk, &kv_full[s], 0, y, policy);
                        tma_load_2d(dst + kKVBlk, &tmk, &kv_full[s], 64, y, policy);
                        tma_load_2d(dst + 2 * kKVBlk, &tmv, &kv_full[s], 0, y, policy);
                        tma_load_2d(dst + 3 * kKVBlk, &tmv, &kv_full[s], 64, y, policy);
                    }
                }
            }
            // copies still in flight finish before the CTA can leave
            for (int k = i - kStagesTC < 0 ? 0 : i - kStagesTC; k < i; ++k)
                (void)mbar_wait(&kv_full[k % kStagesTC], (k / kStagesTC) & 1);
        }
    } else if (warp == kWarpQK) {
        // ================= Q K^T issuer (one thread): tile qk into S buffer
        // qk % kSBufs once its K has landed and the softmax has read that
        // buffer's previous tile, so Q K^T runs up to kSBufs tiles ahead of
        // the softmax within a piece (the next piece's Q is written after this
        // one ends). Descriptors are linear in the start address (its 14-bit
        // field holds address / 16; shared-memory offsets stay below 256 KiB),
        // so each is a base plus a byte offset / 16, computed once.
        if (lane == 0) {
            constexpr uint32_t kIdQK = idesc_bf16(false, kN);
            const uint64_t dQ = smem_desc(sQ, 16, 1024), dK = smem_desc(sKV, 16, 1024);
            bool ok = true;
            int qk = 0, p = 0, n_tma = 0, n_copy = 0;
            const uint64_t q_policy = l2_policy_evict_first();
            TcCursor cur;
            TcPiece pc;
            for (bool more = first_piece(cur, pc); more && ok; more = next_piece(cur, pc), ++p) {
                if (q_by_tma(pc)) {  // the rows by TMA, once every Q K^T of the previous piece has read Q
                    if (p >= 1) ok = mbar_wait(q_free, (p - 1) & 1);
                    if (!ok) break;
                    mbar_arrive_expect_tx(q_tma, kQBytes);
                    const int y = pc.g * P.G, z = P.seq_mode ? pc.qstart + pc.row0 / P.G : pc.qbox;
                    tma_load_3d(smem + kOffQ, &tmq, q_tma, 0, y, z, q_policy);
                    tma_load_3d(smem + kOffQ + kRowBlk, &tmq, q_tma, 64, y, z, q_policy);
                    ok = mbar_wait(q_tma, n_tma++ & 1);
                } else {  // the rows copied by the softmax warps
                    ok = mbar_wait(q_full, n_copy++ & 1);
                }
                if (!ok) break;
                tc_fence_after();
                for (int tt = pc.t_lo; ok && tt < pc.t_hi; ++tt, ++qk) {
                    const int s = qk % kStagesTC;
                    ok = mbar_wait(&kv_full[s], (qk / kStagesTC) & 1);
                    if (ok && qk >= kSBufs) ok = mbar_wait(&s_free[qk % kSBufs], ((qk / kSBufs) - 1) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t dKs = dK + ((s * kKVStage) >> 4);
                    const uint32_t d_s = tmem + (qk % kSBufs) * kN;
#pragma unroll
                    for (int k = 0; k < kHeadDim / 16; ++k)
                        mma_bf16(d_s, dQ + (((k >> 2) * kRowBlk + (k & 3) * 32) >> 4),
                                 dKs + (((k >> 2) * kKVBlk + (k & 3) * 32) >> 4), kIdQK, k > 0);
                    mma_commit(&s_full[qk % kSBufs]);
                }
                if (ok) mma_commit(q_free);  // the piece's last Q K^T
            }
            if (!ok) {
                *abort_flag = 1;
                flag_error(P.err, kErrBitTimeout);
            }
            mma_commit(mma_done);  // every MMA this thread issued completes before tensor memory is freed
        }
    } else {
        // ================= P V issuer (one thread): tile j once the softmax has
        // written P(j). With one copy per row, the tiles alternate between O
        // buffers A and B (the halves' own); with four copies all go to A. The
        // first tile of a piece into each buffer overwrites it, after the
        // epilogue of the previous piece has read both.
        if (lane == 0) {
            constexpr uint32_t kIdPV = idesc_bf16(true, kHeadDim);
            const uint64_t dP = smem_desc(sP, 16, 1024), dV = smem_desc(sKV + 2 * kKVBlk, kKVBlk, 1024);
            bool ok = true;
            int j = 0, p = 0;
            TcCursor cur;
            TcPiece pc;
            for (bool more = first_piece(cur, pc); more && ok; more = next_piece(cur, pc), ++p) {
                const bool alt = kTwo && !(P.seq_mode && pc.row_count - pc.row0 <= kM / 4);
                const int j0 = j;
                for (int tt = pc.t_lo; ok && tt < pc.t_hi; ++tt, ++j) {
                    // the epilogue of the piece that last used this O buffer has read it:
                    // piece p - 1 with the halves' buffers, p - 2 with buffers by piece
                    constexpr int kBack = kTwo ? 1 : 2;
                    if (j == j0 && p >= kBack) {
                        ok = mbar_wait(&o_free[(p - kBack) & 1], ((p - kBack) >> 1) & 1);
                        if (!ok) break;
                    }
                    ok = mbar_wait(&p_full[j & 1], (j >> 1) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    const int k = j - j0;
                    const uint32_t d_o = kTwo ? tmem_o0 + (alt ? (k & 1) * kHeadDim : 0) : tmem_o0 + (p & 1) * kHeadDim;
                    const bool first = alt ? k < 2 : k < 1;
                    const uint64_t dVs = dV + (((j % kStagesTC) * kKVStage) >> 4);
                    const uint64_t dPj = dP + (((j & 1) * kPBytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kN / 16; ++kk)
                        mma_bf16(d_o, dPj + ((kk * 32) >> 4), dVs + ((kk * 16 * 128) >> 4), kIdPV, !first || kk > 0);
                    mma_commit(&kv_empty[j % kStagesTC]);
                    mma_commit(&p_free[j & 1]);
                }
                if (ok) mma_commit(pv_done);  // the piece's last P V
            }
            if (!ok) {
                *abort_flag = 1;
                flag_error(P.err, kErrBitTimeout);
            }
            mma_commit(mma_done);
        }
    }
    if (warp == kWarpQK && lane == 0) (void)mbar_wait(mma_done, 0);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpQK) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// The queries [total_q][Hq][128] bf16 as a 3-D map (d, head, token): 128
// rows of one KV head that are 128 / G consecutive tokens x its G heads are
// one box per 64 columns. False (and *map untouched) when G does not divide
// 128 or the encoding fails: the rows are then copied by the softmax warps.
bool encode_q_map(const sa_dims &d, const uint16_t *q, CUtensorMap *map) {
    const int G = d.num_q_heads / d.num_kv_heads;
    if (kM % G != 0 || d.total_q <= 0) return false;
    const uint64_t dims[3] = {static_cast<uint64_t>(kHeadDim), static_cast<uint64_t>(d.num_q_heads),
                              static_cast<uint64_t>(d.total_q)};
    const uint64_t strides[2] = {static_cast<uint64_t>(kHeadDim) * 2,
                                 static_cast<uint64_t>(d.num_q_heads) * kHeadDim * 2};
    const uint32_t box[3] = {64, static_cast<uint32_t>(G), static_cast<uint32_t>(kM / G)};
    CUtensorMap m;
    if (encode_tensor_map_3d(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<uint16_t *>(q), dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return false;
    *map = m;
    return true;
}

// the shared-memory opt-in of both kernel instances, once
cudaError_t tc_attributes() {
    static const cudaError_t e = [] {
        cudaError_t r = cudaFuncSetAttribute(prefix_tc_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(prefix_tc_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        return r;
    }();
    return e;
}

}  // namespace

cudaError_t launch_prefix_tc(const sa_dims &d, const PlanDevice &pd, const uint16_t *q,
                             const CUtensorMap &tmk, const CUtensorMap &tmv, float scale,
                             float *ws_acc, float *ws_ml, int64_t rows_total, int32_t *err,
                             const int32_t *block_table, cudaStream_t stream) {
    if (const cudaError_t e = tc_attributes(); e != cudaSuccess) return e;
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
    CUtensorMap tmq = tmk;
    p.q_tma = encode_q_map(d, q, &tmq);
    // a plan's rows are held once: two softmax warps per lane quadrant
    prefix_tc_kernel<8><<<pd.num_tiles, tc_threads(8), kSmemBytes, stream>>>(p, tmk, tmv, tmq);
    return cudaGetLastError();
}

cudaError_t launch_seq_tc(const sa_dims &d, const SeqTcConfig &c, const uint16_t *q,
                          const CUtensorMap &tmk, const CUtensorMap &tmv, float scale,
                          float *ws_acc, float *ws_ml, int64_t rows_total, int32_t *err,
                          const int32_t *block_table, const int32_t *seq_lens,
                          const int32_t *q_lens, uint16_t *out, cudaStream_t stream) {
    if (const cudaError_t e = tc_attributes(); e != cudaSuccess) return e;
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
    p.ws_acc = ws_acc;
    p.ws_ml = ws_ml;
    p.out = out;
    p.err = err;
    p.Hq = d.num_q_heads;
    p.Hkv = d.num_kv_heads;
    p.G = d.num_q_heads / d.num_kv_heads;
    p.max_pages = d.max_pages_per_seq;
    p.num_pages = d.num_pages;
    p.n_rows_total = rows_total;
    p.qscale = scale * 1.4426950408889634f;
    if (d.num_seqs == 0 || c.grid <= 0) return cudaSuccess;
    CUtensorMap tmq = tmk;
    p.q_tma = encode_q_map(d, q, &tmq);
    // persistent: one CTA per SM, each walks its range of the tile sequence.
    // Pieces of at most 32 rows (every row held four times) keep half 1 idle,
    // so such batches take four softmax warps (and their registers)
    if (p.G * d.max_q_len > kM / 4)
        prefix_tc_kernel<8><<<static_cast<unsigned>(c.grid), tc_threads(8), kSmemBytes, stream>>>(p, tmk, tmv, tmq);
    else
        prefix_tc_kernel<4><<<static_cast<unsigned>(c.grid), tc_threads(4), kSmemBytes, stream>>>(p, tmk, tmv, tmq);
    return cudaGetLastError();
}

int prefix_tile_rows() { return kM; }
int prefix_key_tile() { return kN; }

}  // namespace sa
