// kv_append.cu -- write the new tokens' K/V rows into their pages.
//
// ExLlamaV2 "Dynamic Generator" page, "Continuous batching": a sequence's
// keys and values live in fixed 256-token pages that its block table names;
// new token i of sequence b sits at position seq_len - q_len + i and goes to
// page block_table[b][pos / 256], slot pos % 256, for every KV head.
//
// One CTA per (query token slot, sequence); one warp per KV head copies the
// 256-byte K row and V row with 8-byte coalesced accesses. Pure bandwidth.
// For quantised pages (the page names the Q4 cache mode, and a Q8 mode to
// come, and gives no format) the warp quantises each row instead, in fp32:
// int8 pages take scale = amax / 127 and 128 codes, int4 pages scale =
// amax / 7 and 128 codes as offset nibbles (64 bytes), codes rounded half to
// even; the warp writes the codes and the scale.
#include "common.cuh"

namespace sa {

namespace {

// Quantised pages: a (token, KV head) row of 128 values becomes 128 codes and
// one scale, scale = amax / Cmax and code = round-half-even(x / scale), both
// in binary32 (IEEE division), clamped to [-Cmax, Cmax]; a zero row gets scale
// 0 and codes 0. int8: Cmax = 127, one byte per code. int4: Cmax = 7, the
// nibble code + 8, value 2c in the low nibble of byte c.
struct QPages {
    uint8_t *k_codes, *v_codes;
    float *k_scales, *v_scales;
};

// This lane's four values (dims 4 lane .. 4 lane + 3) of a row -> four codes:
// one 32-bit word (int8) or one 16-bit word of nibbles (int4); lane 0 stores
// the row's scale.
template <int KB>
__device__ __forceinline__ void quantize_row4(uint2 w, int lane, uint8_t *codes, float *scale) {
    constexpr int kMax = KB == 8 ? 127 : 7;
    const float x[4] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y)};
    float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float sc = __fdiv_rn(amax, static_cast<float>(kMax));
    uint32_t packed = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int c = sc > 0.f ? max(-kMax, min(kMax, __float2int_rn(__fdiv_rn(x[k], sc)))) : 0;
        if constexpr (KB == 8) packed |= (static_cast<uint32_t>(c) & 0xffu) << (8 * k);
        else packed |= static_cast<uint32_t>(c + 8) << (4 * k);
    }
    if constexpr (KB == 8) *reinterpret_cast<uint32_t *>(codes + lane * 4) = packed;
    else *reinterpret_cast<uint16_t *>(codes + lane * 2) = static_cast<uint16_t>(packed);
    if (lane == 0) *scale = sc;
}

// KB: 16 for bf16 pages, 8 for int8 pages, 4 for int4 pages.
template <int KB>
__global__ void __launch_bounds__(256) kv_append_kernel(
    const uint16_t *__restrict__ k_new, const uint16_t *__restrict__ v_new,
    uint16_t *__restrict__ k_pages, uint16_t *__restrict__ v_pages, QPages qp,
    const int32_t *__restrict__ block_table, const int32_t *__restrict__ seq_lens,
    const int32_t *__restrict__ q_lens, int32_t *err, int Hkv, int num_pages, int max_pages,
    int max_q_len, int total_q) {
    // the attention kernel that follows may start its set-up now: it reads
    // the pages only after this grid has completed
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int i = blockIdx.x;
    const int b = blockIdx.y;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    // one round of independent loads: this sequence's lengths and the query
    // counts of the sequences before it (for its first packed row)
    const int n = q_lens[b];
    const int T = seq_lens[b];
    int qstart = 0;
    for (int k = lane; k < b; k += 32) qstart += q_lens[k];
    qstart = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(qstart)));
    if (i >= n) return;
    if (n > T || n > max_q_len || qstart + n > total_q) {  // q_lens disagree with seq_lens or dims
        if (threadIdx.x == 0) flag_error(err, kErrBitQlen);
        return;
    }
    // second round: the page id and the new rows, independent of each other
    const int pos = T - n + i;
    const int j = pos / kPageSize;
    const int pid = j < max_pages ? block_table[static_cast<int64_t>(b) * max_pages + j] : -1;
    const int64_t row = qstart + i;
    const int slot = pos % kPageSize;
    for (int g = warp; g < Hkv; g += blockDim.x >> 5) {
        const int64_t src = (row * Hkv + g) * kHeadDim + lane * 4;
        const uint2 kw = *reinterpret_cast<const uint2 *>(k_new + src);
        const uint2 vw = *reinterpret_cast<const uint2 *>(v_new + src);
        if (pid < 0 || pid >= num_pages) {
            if (threadIdx.x == 0) flag_error(err, kErrBitPageOOB);
            return;
        }
        const int64_t prow = (static_cast<int64_t>(pid) * Hkv + g) * kPageSize + slot;
        if constexpr (KB < 16) {
            constexpr int kCodeRow = kHeadDim * KB / 8;  // bytes of one row's codes
            quantize_row4<KB>(kw, lane, qp.k_codes + prow * kCodeRow, qp.k_scales + prow);
            quantize_row4<KB>(vw, lane, qp.v_codes + prow * kCodeRow, qp.v_scales + prow);
        } else {
            *reinterpret_cast<uint2 *>(k_pages + prow * kHeadDim + lane * 4) = kw;
            *reinterpret_cast<uint2 *>(v_pages + prow * kHeadDim + lane * 4) = vw;
        }
    }
}

}  // namespace

cudaError_t launch_kv_append(const sa_dims &d, const uint16_t *k_new, const uint16_t *v_new,
                             uint16_t *k_pages, uint16_t *v_pages, const int32_t *block_table,
                             const int32_t *seq_lens, const int32_t *q_lens, int32_t *err,
                             cudaStream_t stream) {
    if (d.num_seqs == 0 || d.max_q_len == 0) return cudaSuccess;
    const int threads = 32 * (d.num_kv_heads < 8 ? d.num_kv_heads : 8);
    dim3 grid(d.max_q_len, d.num_seqs);
    kv_append_kernel<16><<<grid, threads, 0, stream>>>(k_new, v_new, k_pages, v_pages, QPages{},
                                                          block_table, seq_lens, q_lens, err,
                                                          d.num_kv_heads, d.num_pages,
                                                          d.max_pages_per_seq, d.max_q_len, d.total_q);
    return cudaGetLastError();
}

cudaError_t launch_kv_append_quant(const sa_dims &d, int code_bits, const uint16_t *k_new,
                                   const uint16_t *v_new, uint8_t *k_codes, uint8_t *v_codes,
                                   float *k_scales, float *v_scales, const int32_t *block_table,
                                   const int32_t *seq_lens, const int32_t *q_lens, int32_t *err,
                                   cudaStream_t stream) {
    if (d.num_seqs == 0 || d.max_q_len == 0) return cudaSuccess;
    const int threads = 32 * (d.num_kv_heads < 8 ? d.num_kv_heads : 8);
    dim3 grid(d.max_q_len, d.num_seqs);
    if (code_bits != 8 && code_bits != 4) return cudaErrorInvalidValue;
    auto kernel = code_bits == 8 ? kv_append_kernel<8> : kv_append_kernel<4>;
    kernel<<<grid, threads, 0, stream>>>(k_new, v_new, nullptr, nullptr,
                                                         QPages{k_codes, v_codes, k_scales, v_scales},
                                                         block_table, seq_lens, q_lens, err,
                                                         d.num_kv_heads, d.num_pages,
                                                         d.max_pages_per_seq, d.max_q_len, d.total_q);
    return cudaGetLastError();
}

}  // namespace sa
