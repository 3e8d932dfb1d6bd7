// tc_work.cuh -- the work of the tensor-core kernel's sequence mode, shared by
// that kernel (which walks it) and the combine pass (which finds the pieces
// it wrote). Sequences with at least min_rows query rows per KV head (G heads
// x new tokens, e.g. q_len = k+1 verification) are attended entirely on the
// tensor cores. A segment is (sequence, KV head, 128-row tile) with one unit
// per 64-key tile over all of the sequence's keys; segments are ordered by
// sequence, then KV head, then row tile, and the resulting sequence of units
// is cut into one contiguous range per CTA. The CTA writes one partial per
// segment it touches, in slot (its range index - the segment's first range
// index).
#pragma once

#include "common.cuh"

namespace sa {

constexpr int kTcKeyTile = 64;    // keys per K/V tile
constexpr int kTcRowTile = 128;   // query rows per tile (tensor-memory lanes)
constexpr int kTcMaxPieces = 8;   // partial slots a segment may use

struct TcSeq {
    int tiles, mtiles, units;  // 64-key tiles, 128-row tiles, units of the whole sequence
};

__device__ __forceinline__ TcSeq tc_seq(int T, int n, int G, int Hkv, int max_q_len, int max_pages,
                                        int min_rows) {
    TcSeq s{0, 0, 0};
    if (min_rows <= 0 || n <= 0 || n > T || n > max_q_len) return s;
    if ((T + kPageSize - 1) / kPageSize > max_pages || G * n < min_rows) return s;
    s.tiles = (T + kTcKeyTile - 1) / kTcKeyTile;
    s.mtiles = (G * n + kTcRowTile - 1) / kTcRowTile;
    s.units = Hkv * s.mtiles * s.tiles;
    return s;
}

// Every CTA gets C or C + 1 units when that keeps C >= C_min (so that no
// segment is cut into more than kTcMaxPieces pieces); otherwise ranges of
// C_min units and the last CTAs stay idle.
struct TcRanges {
    int C, rem;
    __device__ __forceinline__ int begin(int w) const { return w * C + min(w, rem); }
    __device__ __forceinline__ int range_of(int t) const {
        const int big = rem * (C + 1);
        return t < big ? t / (C + 1) : rem + (t - big) / C;
    }
};

__device__ __forceinline__ TcRanges make_tc_ranges(int total, int W, int max_tiles) {
    const int C_min = max(1, (max_tiles + kTcMaxPieces - 2) / (kTcMaxPieces - 1));
    const int even = total / W;
    if (even >= C_min) return TcRanges{even, total - even * W};
    return TcRanges{C_min, 0};
}

// Waves of whole segments, for batches whose sequences all have the same
// length and query count (chunked prefill) and at least two segments per
// CTA: CTA c takes segments c, c + W, c + 2 W, ... (W CTAs) for `waves`
// waves, so that the CTAs running at the same time hold the row tiles of the
// same few (sequence, KV head) pairs and walk the same K/V tiles together
// (each tile comes from DRAM once and from L2 for the others); the segments
// left over are cut evenly between all CTAs as above, so that every CTA ends
// at the same time. `base` is the units of the waves (the cut's units are
// counted from there). A CTA writes the output of a segment it attends whole
// itself, from one copy of each row: so every row tile must hold more than
// 32 of the `rows` query rows per KV head (fewer are held four times).
struct TcWaves {
    int waves, seg_per_seq, base;
};

__device__ __forceinline__ TcWaves make_tc_waves(bool uniform, int B, const TcSeq &w, int Hkv, int W, int rows) {
    TcWaves v{0, 0, 0};
    if (!uniform || w.units == 0) return v;
    if (rows - (w.mtiles - 1) * kTcRowTile <= 32) return v;
    const int seg_per_seq = Hkv * w.mtiles;
    const long long nseg = static_cast<long long>(B) * seg_per_seq;
    if (nseg < 2LL * W) return v;
    v.waves = static_cast<int>(nseg / W) - 1;
    v.seg_per_seq = seg_per_seq;
    v.base = v.waves * W * w.tiles;
    return v;
}

}  // namespace sa
