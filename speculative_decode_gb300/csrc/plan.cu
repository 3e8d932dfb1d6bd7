// plan.cu -- host planner: find page runs that several sequences share.
//
// ExLlamaV2 "Dynamic Generator" page, "Deduplication": sequences with a common
// prefix index the same physical pages. The planner inserts every sequence's
// block-table row into a trie keyed by physical page id; a trie node that
// several sequences pass through is a page they share at the same logical
// position. Maximal chains of nodes with the same member set form runs. A run
// with enough query rows per KV head is handed to the tensor-core kernel,
// which streams each of its pages once for all members; the split kernel then
// starts each member at the first page after its shared runs.
#include <cuda_runtime.h>

#include <algorithm>
#include <map>
#include <new>
#include <utility>
#include <vector>

#include "plan.h"

struct sa_plan {
    sa::PlanHost host;
    sa::PlanDevice dev{};
    void *dev_buf = nullptr;
};

namespace sa {

namespace {

struct TrieNode {
    std::vector<int32_t> members;
};

}  // namespace

PlanHost build_plan(const sa_dims &d, const int32_t *bt, const int32_t *seq_lens,
                    const int32_t *q_lens, int sms, int min_rows) {
    PlanHost P;
    P.dims = d;
    const int B = d.num_seqs;
    const int G = d.num_q_heads / d.num_kv_heads;
    P.skip_pages.assign(B, 0);
    P.run_slots.assign(B, 0);
    std::vector<int32_t> qstart(B + 1, 0);
    for (int b = 0; b < B; ++b) qstart[b + 1] = qstart[b] + std::max(0, q_lens[b]);

    // ---- trie of block-table rows
    std::vector<TrieNode> nodes;
    std::map<std::pair<int, int>, int> child;
    std::vector<std::vector<int>> path(B);
    for (int b = 0; b < B; ++b) {
        const int T = seq_lens[b], n = q_lens[b];
        if (n <= 0 || n > T || n > d.max_q_len) continue;
        const int np = (T + kPageSize - 1) / kPageSize;
        if (np > d.max_pages_per_seq) continue;
        // only pages every key of which is in the cache can be shared on the
        // tensor cores (a partly written page may hold stale, non-finite data
        // that a zero probability would still multiply); the last partial page
        // stays on the split kernel
        const int full = T / kPageSize;
        int cur = -1;
        for (int j = 0; j < full; ++j) {
            const int page = bt[static_cast<int64_t>(b) * d.max_pages_per_seq + j];
            if (page < 0 || page >= d.num_pages) break;  // left to the split kernel, which flags it
            auto key = std::make_pair(cur, page);
            auto it = child.find(key);
            int node;
            if (it == child.end()) {
                node = static_cast<int>(nodes.size());
                nodes.emplace_back();
                child.emplace(key, node);
            } else {
                node = it->second;
            }
            nodes[node].members.push_back(b);
            path[b].push_back(node);
            cur = node;
        }
    }

    // ---- runs: maximal chains of nodes with one member set of size >= 2
    struct Run {
        int page_lo, page_hi;
        std::vector<int32_t> members;
        int rows;
        bool taken;
    };
    std::vector<Run> runs;
    std::map<std::pair<int, int>, int> run_id;  // (first node, last node)
    std::vector<std::vector<int>> runs_of(B);
    for (int b = 0; b < B; ++b) {
        size_t j = 0;
        while (j < path[b].size()) {
            const auto &mem = nodes[path[b][j]].members;
            if (mem.size() < 2) break;
            size_t k = j;
            while (k + 1 < path[b].size() && nodes[path[b][k + 1]].members == mem) ++k;
            auto key = std::make_pair(path[b][j], path[b][k]);
            auto it = run_id.find(key);
            int r;
            if (it == run_id.end()) {
                r = static_cast<int>(runs.size());
                int rows = 0;
                for (int m : mem) rows += G * q_lens[m];
                runs.push_back({static_cast<int>(j), static_cast<int>(k + 1), mem, rows, rows >= min_rows});
                run_id.emplace(key, r);
            } else {
                r = it->second;
            }
            runs_of[b].push_back(r);
            j = k + 1;
        }
    }
    // member sets shrink with depth, so the taken runs of a path are a prefix of it
    int n_taken = 0;
    for (auto &r : runs) {
        if (!r.taken) continue;
        ++n_taken;
        P.num_members += static_cast<int32_t>(r.members.size());
        P.num_run_pages += r.page_hi - r.page_lo;
    }
    P.num_runs = n_taken;
    if (n_taken == 0) return P;

    // ---- page chunks: enough work items for about one CTA per SM
    int64_t base_items = 0;
    for (auto &r : runs)
        if (r.taken) base_items += static_cast<int64_t>(d.num_kv_heads) * ((r.rows + kPrefixTileRows - 1) / kPrefixTileRows);
    // a member's runs together use at most 8 partial slots (the merge takes 16
    // per row, 8 of which belong to the split kernel's pieces)
    int max_runs_per_seq = 1;
    for (int b = 0; b < B; ++b) {
        int k = 0;
        for (int r : runs_of[b]) {
            if (!runs[r].taken) break;
            ++k;
        }
        max_runs_per_seq = std::max(max_runs_per_seq, k);
    }
    const int64_t chunk_cap = std::max(1, 8 / max_runs_per_seq);
    const int64_t chunks_wanted = std::min<int64_t>(
        chunk_cap, std::max<int64_t>(1, (std::max(sms, 1) + base_items - 1) / base_items));

    std::vector<int> run_index(runs.size(), -1), run_chunk_pages(runs.size(), 0), run_chunks(runs.size(), 0);
    std::vector<int> slot_base_of;  // filled per (run, member) below
    for (size_t r = 0; r < runs.size(); ++r) {
        if (!runs[r].taken) continue;
        const int pages = runs[r].page_hi - runs[r].page_lo;
        const int nch = static_cast<int>(std::min<int64_t>(pages, chunks_wanted));
        run_chunk_pages[r] = (pages + nch - 1) / nch;
        run_chunks[r] = (pages + run_chunk_pages[r] - 1) / run_chunk_pages[r];
    }
    // slots: each member's taken runs in depth order, one slot per chunk
    std::map<std::pair<int, int>, int> member_slot;  // (run, b) -> first slot
    for (int b = 0; b < B; ++b) {
        int next = 0;
        for (int r : runs_of[b]) {
            if (!runs[r].taken) break;
            member_slot[{r, b}] = next;
            next += run_chunks[r];
            P.skip_pages[b] = runs[r].page_hi;
        }
        P.run_slots[b] = next;
        P.max_run_slots = std::max(P.max_run_slots, next);
    }
    // the first token of rows [first, first + min(n, 128)) if row k of them is
    // token first_token + k / G with head k % G, else -1
    auto box_token = [&](int first, int n) -> int32_t {
        if (kPrefixTileRows % G != 0) return -1;
        const int32_t tok0 = P.rows[first].token;
        for (int k = 0; k < std::min(n, kPrefixTileRows); ++k) {
            const RunRow &rw = P.rows[first + k];
            if (rw.token != tok0 + k / G || rw.head_local != k % G) return -1;
        }
        return tok0;
    };
    // rows and descriptors
    for (size_t r = 0; r < runs.size(); ++r) {
        if (!runs[r].taken) continue;
        run_index[r] = static_cast<int>(P.run_desc.size() / kRunDescInts);
        const int row_begin = static_cast<int>(P.rows.size());
        for (int b : runs[r].members) {
            const int T = seq_lens[b], n = q_lens[b];
            for (int i = 0; i < n; ++i)
                for (int h = 0; h < G; ++h)
                    P.rows.push_back({qstart[b] + i, h, T - n + i, member_slot[{static_cast<int>(r), b}]});
        }
        const int row_count = static_cast<int>(P.rows.size()) - row_begin;
        P.run_desc.insert(P.run_desc.end(), {runs[r].page_lo, runs[r].page_hi, row_begin, row_count,
                                             run_chunk_pages[r], runs[r].members[0]});
        // row tiles of one (KV head, page chunk) are adjacent so that they run
        // together and the second and later ones read the chunk from L2
        for (int g = 0; g < d.num_kv_heads; ++g)
            for (int c = 0; c < run_chunks[r]; ++c)
                for (int t = 0; t < row_count; t += kPrefixTileRows) {
                    const int lo = runs[r].page_lo + c * run_chunk_pages[r];
                    const int hi = std::min(runs[r].page_hi, lo + run_chunk_pages[r]);
                    P.tiles.insert(P.tiles.end(), {run_index[r], g, t, lo, hi, c, box_token(row_begin + t, row_count - t)});
                }
    }
    return P;
}

int plan_run_slots(const sa_plan *plan) { return plan ? plan->dev.max_run_slots : 0; }

bool plan_matches(const sa_plan *plan, const sa_dims &d) {
    const sa_dims &p = plan->host.dims;
    return p.num_seqs == d.num_seqs && p.num_q_heads == d.num_q_heads &&
           p.num_kv_heads == d.num_kv_heads && p.total_q == d.total_q &&
           p.max_q_len == d.max_q_len && p.max_pages_per_seq == d.max_pages_per_seq &&
           p.num_pages == d.num_pages;
}

const PlanDevice *plan_device(const sa_plan *plan) { return plan ? &plan->dev : nullptr; }

}  // namespace sa

using namespace sa;

namespace {

constexpr int kMinRunRows = 32;
// Whether plans hand their shared runs to the tensor-core kernel (otherwise
// they only describe them and every page goes through the split kernel).
constexpr bool kPrefixPathReady = true;

int check_plan_args(const sa_dims *d, const int32_t *bt, const int32_t *sl, const int32_t *ql) {
    if (d == nullptr || d->num_seqs < 0 || d->num_q_heads <= 0 || d->num_kv_heads <= 0 ||
        d->num_q_heads % d->num_kv_heads != 0 || d->max_pages_per_seq < 0 || d->total_q < 0)
        return SA_ERR_ARG;
    if (d->head_dim != kHeadDim || d->page_size != kPageSize || d->max_q_len > kPlanMaxQLen)
        return SA_ERR_UNSUPPORTED;
    if (d->num_seqs > 0 && (bt == nullptr || sl == nullptr || ql == nullptr)) return SA_ERR_ARG;
    int64_t tq = 0;
    for (int b = 0; b < d->num_seqs; ++b) tq += std::max(0, ql[b]);
    if (tq != d->total_q) return SA_ERR_ARG;
    return SA_OK;
}

}  // namespace

extern "C" {

int sa_plan_analyze(const sa_dims *dims, const int32_t *block_table_host,
                    const int32_t *seq_lens_host, const int32_t *q_lens_host, int32_t sm_count,
                    int32_t *skip_pages_out, int32_t *run_slots_out, int32_t *num_runs,
                    int32_t *num_tiles) {
    int rc = check_plan_args(dims, block_table_host, seq_lens_host, q_lens_host);
    if (rc) return rc;
    PlanHost P = build_plan(*dims, block_table_host, seq_lens_host, q_lens_host, sm_count, kMinRunRows);
    for (int b = 0; b < dims->num_seqs; ++b) {
        if (skip_pages_out) skip_pages_out[b] = P.skip_pages[b];
        if (run_slots_out) run_slots_out[b] = P.run_slots[b];
    }
    if (num_runs) *num_runs = P.num_runs;
    if (num_tiles) *num_tiles = static_cast<int32_t>(P.tiles.size() / kTileInts);
    return SA_OK;
}

int sa_plan_create(const sa_dims *dims, const int32_t *block_table_host,
                   const int32_t *seq_lens_host, const int32_t *q_lens_host, sa_plan **out) {
    if (out == nullptr) return SA_ERR_ARG;
    *out = nullptr;
    int rc = check_plan_args(dims, block_table_host, seq_lens_host, q_lens_host);
    if (rc) return rc;
    int sms = device_sm_count();
    if (sms <= 0) return SA_ERR_CUDA;
    sa_plan *plan = new (std::nothrow) sa_plan;
    if (plan == nullptr) return SA_ERR_ARG;
    plan->host = build_plan(*dims, block_table_host, seq_lens_host, q_lens_host, sms, kMinRunRows);
    const PlanHost &H = plan->host;
    PlanDevice &D = plan->dev;
    D.num_runs = H.num_runs;
    D.num_tiles = kPrefixPathReady ? static_cast<int32_t>(H.tiles.size() / kTileInts) : 0;
    D.max_run_slots = kPrefixPathReady ? H.max_run_slots : 0;
    if (D.num_tiles > 0) {
        const int B = dims->num_seqs;
        const size_t n_ints = 2 * static_cast<size_t>(B) + H.run_desc.size() + 4 * H.rows.size() + H.tiles.size();
        std::vector<int32_t> blob;
        blob.reserve(n_ints);
        blob.insert(blob.end(), H.skip_pages.begin(), H.skip_pages.end());
        blob.insert(blob.end(), H.run_slots.begin(), H.run_slots.end());
        blob.insert(blob.end(), H.run_desc.begin(), H.run_desc.end());
        for (const RunRow &r : H.rows) blob.insert(blob.end(), {r.token, r.head_local, r.limit, r.slot});
        blob.insert(blob.end(), H.tiles.begin(), H.tiles.end());
        if (cudaMalloc(&plan->dev_buf, blob.size() * sizeof(int32_t)) != cudaSuccess) {
            delete plan;
            return SA_ERR_CUDA;
        }
        if (cudaMemcpy(plan->dev_buf, blob.data(), blob.size() * sizeof(int32_t),
                       cudaMemcpyHostToDevice) != cudaSuccess) {
            cudaFree(plan->dev_buf);
            delete plan;
            return SA_ERR_CUDA;
        }
        const int32_t *p = static_cast<const int32_t *>(plan->dev_buf);
        D.skip_pages = p;
        D.run_slots = p + B;
        D.run_desc = p + 2 * B;
        D.run_rows = D.run_desc + H.run_desc.size();
        D.tiles = D.run_rows + 4 * H.rows.size();
    }
    *out = plan;
    return SA_OK;
}

void sa_plan_destroy(sa_plan *plan) {
    if (plan == nullptr) return;
    if (plan->dev_buf) cudaFree(plan->dev_buf);
    delete plan;
}

int sa_plan_stats(const sa_plan *plan, int32_t *num_runs, int32_t *num_members, int32_t *num_pages) {
    if (plan == nullptr) return SA_ERR_ARG;
    if (num_runs) *num_runs = plan->host.num_runs;
    if (num_members) *num_members = plan->host.num_members;
    if (num_pages) *num_pages = plan->host.num_run_pages;
    return SA_OK;
}

}  // extern "C"
