// verify.cu -- greedy verification: vocab-wide argmax of each verifier row,
// then the left-to-right accept rule.
//
// Hugging Face "Assisted Generation" page, "Assisted Generation loop": the
// verifier's predicted token at every position is compared with the draft
// candidates from the left (step 3); at the first mismatch the verifier's
// token is kept and the later candidates are dropped (step 4); the draft
// window grows by 2 when every candidate matched and shrinks by 1 otherwise
// (step 5), and the loop drafts again with that window (step 1). Readings:
// ties go to the lowest index, -0.0 == +0.0, NaN never wins (an all-NaN row
// gives 0), the window never drops below 1, with no mismatch the correction
// token is the verifier's bonus token after the last candidate, and the
// call's new tokens are the previous step's last token followed by the
// candidates (so the next call keeps seq_len - q_len + 1 + accepted tokens and
// opens with the correction token and min(window, k_max) candidates).
//
// Design: the logits rows (fp32, 128256 wide for a Llama-3 vocabulary) are the
// only real traffic. Each row is cut into chunks; one CTA streams one chunk
// with 16-byte loads and reduces it to a (value, index) pair ordered by
// (larger value, then lower index). The last CTA of a sequence to finish
// (one atomic counter per sequence, no spinning) reduces that sequence's
// chunk pairs row by row and applies the accept rule. The counter is reset by
// that CTA, so the workspace is ready for the next call.
#include <climits>

#include "common.cuh"

namespace sa {

namespace {

__device__ __forceinline__ void take_if_better(float v, int i, float &bv, int &bi) {
    // NaN fails both comparisons and is never taken.
    if (v > bv || (v == bv && i < bi)) {
        bv = v;
        bi = i;
    }
}

__global__ void __launch_bounds__(256) argmax_accept_kernel(const VerifyParams P) {
    __shared__ float s_val[8];
    __shared__ int s_idx[8];
    __shared__ int s_tok[16];
    __shared__ int s_last;
    const int K1 = P.k_max + 1;
    const int chunk = blockIdx.x;
    const int rowid = blockIdx.y;
    const int b = rowid / K1;
    const int j = rowid % K1;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int n = P.n_cand[b];
    const bool bad = n < 0 || n > P.k_max;

    if (!bad && j <= n) {
        const int64_t lo = static_cast<int64_t>(chunk) * P.chunk;
        const int64_t hi = min(static_cast<int64_t>(P.V), lo + P.chunk);
        const float *row = P.logits + static_cast<int64_t>(rowid) * P.V;
        float bv = -INFINITY;
        int bi = INT_MAX;
        if ((P.V & 3) == 0) {
            // rows are 16-byte aligned and chunk bounds are multiples of 4.
            // Four 16-byte loads per thread per step with the next step's
            // loads in flight while this step is reduced, into four
            // independent (value, index) pairs merged at the end (the order
            // (larger value, then lower index) makes the merge exact).
            constexpr int kStep = 4 * 4 * 256;  // elements per CTA step
            float4 cur[4], nxt[4];
            float pv[4];
            int pi[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                pv[u] = -INFINITY;
                pi[u] = INT_MAX;
            }
            auto load_step = [&](int64_t e, float4 (&x)[4]) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int64_t eu = e + u * 1024;
                    x[u] = eu < hi ? __ldcs(reinterpret_cast<const float4 *>(row + eu))
                                   : make_float4(NAN, NAN, NAN, NAN);
                }
            };
            int64_t e = lo + threadIdx.x * 4;
            load_step(e, cur);
            for (; e < hi; e += kStep) {
                load_step(e + kStep, nxt);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int base = static_cast<int>(e + u * 1024);
                    take_if_better(cur[u].x, base, pv[u], pi[u]);
                    take_if_better(cur[u].y, base + 1, pv[u], pi[u]);
                    take_if_better(cur[u].z, base + 2, pv[u], pi[u]);
                    take_if_better(cur[u].w, base + 3, pv[u], pi[u]);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) cur[u] = nxt[u];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) take_if_better(pv[u], pi[u], bv, bi);
        } else {
            for (int64_t e = lo + threadIdx.x; e < hi; e += blockDim.x)
                take_if_better(__ldcs(row + e), static_cast<int>(e), bv, bi);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            take_if_better(ov, oi, bv, bi);
        }
        if (lane == 0) {
            s_val[warp] = bv;
            s_idx[warp] = bi;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int w = 1; w < (blockDim.x >> 5); ++w) take_if_better(s_val[w], s_idx[w], bv, bi);
            const int64_t at = static_cast<int64_t>(rowid) * P.n_chunks + chunk;
            P.part_val[at] = bv;
            P.part_idx[at] = bi;
        }
    }

    // ---- count this CTA; the last one of sequence b finishes the sequence
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const int prev = atomicAdd(&P.counters[b], 1);
        s_last = prev == K1 * P.n_chunks - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (bad) {
        if (threadIdx.x == 0) {
            flag_error(P.err, kErrBitQlen);
            P.counters[b] = 0;
        }
        return;
    }
    for (int r = warp; r <= n; r += blockDim.x >> 5) {
        float bv = -INFINITY;
        int bi = INT_MAX;
        const int64_t base = (static_cast<int64_t>(b) * K1 + r) * P.n_chunks;
        for (int c = lane; c < P.n_chunks; c += 32)
            take_if_better(__ldcg(P.part_val + base + c), __ldcg(P.part_idx + base + c), bv, bi);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            take_if_better(ov, oi, bv, bi);
        }
        if (lane == 0) s_tok[r] = bi == INT_MAX ? 0 : bi;  // all-NaN row -> 0
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int a = 0;
        while (a < n && P.candidates[static_cast<int64_t>(b) * P.k_max + a] == s_tok[a]) ++a;
        P.accepted[b] = a;
        P.next_tok[b] = s_tok[a];
        if (P.seq_lens) {
            // the next call (the loop drafts again with the adjusted window):
            // it keeps the tokens before this call, this call's first token
            // and the accepted candidates, then opens with the correction
            // token followed by min(window, k_max) candidates
            const int ql = P.q_lens[b], T = P.seq_lens[b];
            if (ql < n + 1 || T < ql) {
                flag_error(P.err, kErrBitQlen);
            } else {
                const int w = P.window[b];
                const int w2 = a == n ? w + 2 : (w - 1 > 1 ? w - 1 : 1);
                const int nn = w2 < P.k_max ? w2 : P.k_max;
                P.window[b] = w2;
                P.n_cand_next[b] = nn;
                P.q_lens[b] = nn + 1;
                P.seq_lens[b] = T - ql + 1 + a + nn + 1;
            }
        } else if (P.window) {
            const int w = P.window[b];
            P.window[b] = a == n ? w + 2 : (w - 1 > 1 ? w - 1 : 1);
        }
        P.counters[b] = 0;
    }
}

}  // namespace

cudaError_t launch_verify(const VerifyParams &p, cudaStream_t stream) {
    if (p.B == 0) return cudaSuccess;
    dim3 grid(p.n_chunks, p.B * (p.k_max + 1));
    argmax_accept_kernel<<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace sa
