// Uniform multi-token decode (mla_decode_multi_token).
//
// vLLM mla_attention API docs, QueryLenSupport.UNIFORM: every request has the
// same query length T > 1 (speculative decoding), and the query block is
// causal unless the attention group allows a non-causal one
// (MLACommonMetadataBuilder.build). The T new tokens are in the cache already,
// so query token i of a request with L tokens sits at position L - T + i and,
// causally, sees the first L - T + 1 + i tokens.
//
// Two ways, chosen by the plan's shape:
//   * T * N <= 128 (the plan has T * N heads): q [B, T, N, 576] is q [B, T * N,
//     576], so the T query tokens' heads are the rows of one decode, which
//     reads each page once; the kernels end each row's tokens at its own
//     causal limit.
//   * otherwise (the plan has B * T rows of N heads): each (request, query
//     token) becomes a row of the decode: a small kernel writes, into caller
//     scratch, each row's block-table row (a copy of its request's) and its
//     visible length, and the decode runs over the B * T rows. Every row reads
//     its request's pages. Under the page-balanced schedule the rows go in
//     token-major order (row r = i * B + b: every request's token 0, then
//     every request's token 1, ...), so the equal cut gives the CTA pairs of
//     token i the same requests' pages at the same time as those of token 0
//     and the rereads of a page mostly hit L2; q, out and lse stay
//     [B, T, N, ...] (the decode maps row r to tensor row b * T + i). Under
//     the split schedule the rows are request-major (r = b * T + i), the
//     tensors' own order.
#include <cuda_runtime.h>

#include <cstdint>

#include "mla_internal.h"

namespace mla {
namespace {

__global__ void mla_expand_rows_kernel(const int32_t* __restrict__ block_table,
                                       const int32_t* __restrict__ seq_lens, int q_len,
                                       int causal, int max_blocks, int batch, int token_major,
                                       int32_t* __restrict__ table_out,
                                       int32_t* __restrict__ lens_out) {
    const int r = blockIdx.x;
    const int b = token_major ? r % batch : r / q_len;
    const int i = token_major ? r / batch : r - b * q_len;
    const int32_t* src = block_table + int64_t(b) * max_blocks;
    int32_t* dst = table_out + int64_t(r) * max_blocks;
    for (int j = threadIdx.x; j < max_blocks; j += blockDim.x) dst[j] = src[j];
    if (threadIdx.x == 0) {
        const int L = seq_lens[b];
        int eff = L;
        // A length outside [0, max_blocks * 64] passes through unchanged so
        // that the decode reports it (MLA_ERR_BAD_SEQ_LEN).
        if (causal && L >= 0 && int64_t(L) <= int64_t(max_blocks) * kPageSize) {
            eff = L - (q_len - 1 - i);
            if (eff < 0) eff = 0;
        }
        lens_out[r] = eff;
    }
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" size_t mla_multi_token_scratch_bytes(int batch, int q_len, int max_blocks_per_seq) {
    if (batch < 0 || q_len < 1 || max_blocks_per_seq < 1) return 0;
    const size_t rows = size_t(batch) * size_t(q_len);
    return round256(rows * size_t(max_blocks_per_seq) * 4) + round256(rows * 4);
}

extern "C" int mla_decode_multi_token(const mla_decode_plan_t* plan, int q_len, int num_heads,
                                      int causal, const void* q, const void* latent_cache,
                                      int64_t num_blocks, const int32_t* block_table,
                                      const int32_t* seq_lens, float softmax_scale, void* out,
                                      float* lse, void* workspace, size_t workspace_bytes,
                                      void* scratch, size_t scratch_bytes, void* stream) {
    if (!plan || q_len < 1 || num_heads < 1 || plan->batch < 0) return MLA_ERR_INVALID_ARG;
    if (int64_t(plan->num_heads) == int64_t(q_len) * num_heads)   // the tokens' heads as rows
        return decode_impl(plan, q, latent_cache, num_blocks, block_table, seq_lens,
                           softmax_scale, out, lse, workspace, workspace_bytes, stream, q_len,
                           num_heads, causal ? 1 : 0);
    if (plan->num_heads != num_heads || plan->batch % q_len != 0) return MLA_ERR_INVALID_ARG;
    const int batch = plan->batch / q_len;
    if (batch == 0) return MLA_OK;
    if (!block_table || !seq_lens) return MLA_ERR_INVALID_ARG;
    const int max_blocks = plan->max_blocks_per_seq;
    const size_t need = mla_multi_token_scratch_bytes(batch, q_len, max_blocks);
    if (need == 0) return MLA_ERR_INVALID_ARG;
    if (!scratch || scratch_bytes < need || (reinterpret_cast<uintptr_t>(scratch) & 255u) != 0)
        return MLA_ERR_WORKSPACE;
    const size_t rows = size_t(batch) * size_t(q_len);
    int32_t* table_rows = static_cast<int32_t*>(scratch);
    int32_t* lens_rows = reinterpret_cast<int32_t*>(static_cast<char*>(scratch) +
                                                    round256(rows * size_t(max_blocks) * 4));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int token_major = plan->sched_pairs > 0 ? 1 : 0;
    mla_expand_rows_kernel<<<unsigned(rows), 128, 0, st>>>(block_table, seq_lens, q_len,
                                                           causal ? 1 : 0, max_blocks, batch,
                                                           token_major, table_rows, lens_rows);
    if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
    return decode_impl(plan, q, latent_cache, num_blocks, table_rows, lens_rows, softmax_scale,
                       out, lse, workspace, workspace_bytes, stream, 1, num_heads, 0,
                       token_major ? q_len : 1);
}
