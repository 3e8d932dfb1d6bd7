// defrag.cu -- compaction of a fragmented page pool.
//
// ExLlamaV2 "Dynamic Generator" page, "Continuous batching": finished jobs
// free their pages, which leaves holes; the block table need not be
// contiguous, and the cache can be defragmented (the generator does so only
// when its job queue is empty). The page gives no procedure. Here: with L
// live pages (named by a table within its sequence's length), each live page
// at id >= L moves into a free id below L, in increasing order on both
// sides, and the tables are rewritten through that map. Every move reads a
// page no move writes, so all moves are made by one kernel, in any order.
//
// The planner is host code (it runs when the queue is empty, on host
// tables). The copy is pure bandwidth: each CTA moves 32 KiB chunks of a
// page with 16-byte coalesced loads (all eight in flight per thread) and
// streaming stores; the grid covers every chunk of every moved page of both
// pools, a few CTAs per SM.
#include "common.cuh"

#include <vector>

namespace sa {

namespace {

constexpr int kCopyThreads = 256;
constexpr int kVecPerThread = 8;                                  // 16-byte vectors per thread
constexpr int64_t kChunkVecs = kCopyThreads * kVecPerThread;      // 32 KiB per CTA step

__device__ __forceinline__ uint4 load_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Two pools of pages of page_vecs 16-byte vectors each (the K and V pools,
// or any pair of pools paged alike); a page's last chunk may be partial.
__global__ void __launch_bounds__(kCopyThreads) defrag_kernel(uint4 *k_pages, uint4 *v_pages,
                                                               const int32_t *__restrict__ moves,
                                                               int n_moves, int num_pages,
                                                               int64_t page_vecs, int32_t *err) {
    const int64_t chunks = (page_vecs + kChunkVecs - 1) / kChunkVecs;  // per page and pool
    const int64_t units = static_cast<int64_t>(n_moves) * 2 * chunks;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
        const int m = static_cast<int>(u / (2 * chunks));
        const int64_t r = u % (2 * chunks);
        const int from = moves[2 * m], to = moves[2 * m + 1];
        if (from < 0 || from >= num_pages || to < 0 || to >= num_pages) {
            if (threadIdx.x == 0 && r == 0) flag_error(err, kErrBitPageOOB);
            continue;
        }
        uint4 *pool = r < chunks ? k_pages : v_pages;
        const int64_t off = (r % chunks) * kChunkVecs + threadIdx.x;
        const uint4 *src = pool + static_cast<int64_t>(from) * page_vecs + off;
        uint4 *dst = pool + static_cast<int64_t>(to) * page_vecs + off;
        uint4 x[kVecPerThread];
#pragma unroll
        for (int i = 0; i < kVecPerThread; ++i)
            if (off + i * kCopyThreads < page_vecs) x[i] = load_stream(src + i * kCopyThreads);
#pragma unroll
        for (int i = 0; i < kVecPerThread; ++i)
            if (off + i * kCopyThreads < page_vecs) __stcs(dst + i * kCopyThreads, x[i]);
    }
}

}  // namespace

int defrag_plan_host(int num_seqs, int num_pages, int max_pages, const int32_t *block_table,
                     const int32_t *seq_lens, int32_t *new_table, int32_t *moves, int32_t *n_moves,
                     int32_t *n_live) {
    // live pages: named by a table within its sequence's length
    std::vector<uint8_t> live(static_cast<size_t>(num_pages), 0);
    for (int b = 0; b < num_seqs; ++b) {
        if (seq_lens[b] < 0) return SA_ERR_ARG;
        const int64_t used = (static_cast<int64_t>(seq_lens[b]) + kPageSize - 1) / kPageSize;
        if (used > max_pages) return SA_ERR_ARG;
        const int32_t *row = block_table + static_cast<int64_t>(b) * max_pages;
        for (int64_t j = 0; j < used; ++j) {
            if (row[j] < 0 || row[j] >= num_pages) return SA_ERR_PAGE_OOB;
            live[row[j]] = 1;
        }
    }
    int32_t L = 0;
    for (uint8_t x : live) L += x;
    // free ids below L, in increasing order; the live ids at or above L take
    // them in increasing order
    std::vector<int32_t> map(static_cast<size_t>(num_pages));
    for (int p = 0; p < num_pages; ++p) map[p] = p;
    std::vector<int32_t> holes;
    for (int p = 0; p < L; ++p)
        if (!live[p]) holes.push_back(p);
    int32_t m = 0;
    for (int p = L; p < num_pages; ++p) {
        if (!live[p]) continue;
        map[p] = holes[m];
        moves[2 * m] = p;
        moves[2 * m + 1] = holes[m];
        ++m;
    }
    for (int b = 0; b < num_seqs; ++b) {
        const int64_t used = (static_cast<int64_t>(seq_lens[b]) + kPageSize - 1) / kPageSize;
        const int64_t base = static_cast<int64_t>(b) * max_pages;
        for (int64_t j = 0; j < max_pages; ++j)
            new_table[base + j] = j < used ? map[block_table[base + j]] : -1;
    }
    *n_moves = m;
    *n_live = L;
    return SA_OK;
}

cudaError_t launch_defrag(void *k_pages, void *v_pages, const int32_t *moves, int n_moves,
                          int num_pages, int64_t page_bytes, int32_t *err, int sms, cudaStream_t stream) {
    const int64_t page_vecs = page_bytes / 16;
    const int64_t units = static_cast<int64_t>(n_moves) * 2 * ((page_vecs + kChunkVecs - 1) / kChunkVecs);
    const int grid = static_cast<int>(std::min<int64_t>(units, static_cast<int64_t>(sms) * 8));
    defrag_kernel<<<grid, kCopyThreads, 0, stream>>>(reinterpret_cast<uint4 *>(k_pages),
                                                     reinterpret_cast<uint4 *>(v_pages), moves, n_moves,
                                                     num_pages, page_vecs, err);
    return cudaGetLastError();
}

}  // namespace sa
