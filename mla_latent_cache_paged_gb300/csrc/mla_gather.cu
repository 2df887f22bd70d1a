// Test hook: gather each request's cache rows, in logical token order, into a
// dense buffer (mla_debug_gather_pages). Token t of request b is row t % 64 of
// block block_table[b, t / 64] -- the page-table reading every decode kernel
// here uses (the pages show the table's shape, not the formula: ModelOpt
// mla_attention_decode, block_table; vLLM's gather_cache / cp_gather_cache
// calls in mla_attention, _compute_prefill_context).
#include <cuda_runtime.h>

#include "mla_device.cuh"

namespace mla {
namespace {

constexpr int kGatherThreads = 256;
constexpr int kRowChunks = kD * 2 / 16;   // 72 x 16 bytes per row

__global__ void __launch_bounds__(kGatherThreads) mla_gather_kernel(
        const uint16_t* __restrict__ cache, int64_t num_blocks,
        const int32_t* __restrict__ block_table, const int32_t* __restrict__ seq_lens,
        int max_blocks, int dst_max_tokens, uint16_t* __restrict__ dst, int32_t* status) {
    const int b = blockIdx.y;
    int L = seq_lens[b];
    if (L < 0 || int64_t(L) > int64_t(max_blocks) * kPageSize || L > dst_max_tokens) {
        if (threadIdx.x == 0 && blockIdx.x == 0) record_error(status, MLA_ERR_BAD_SEQ_LEN, L);
        return;
    }
    const int32_t* table = block_table + size_t(b) * max_blocks;
    const int total = L * kRowChunks;
    for (int idx = blockIdx.x * kGatherThreads + threadIdx.x; idx < total;
         idx += gridDim.x * kGatherThreads) {
        const int t = idx / kRowChunks;
        const int c = idx % kRowChunks;
        const int blk = table[t / kPageSize];
        if (blk < 0 || int64_t(blk) >= num_blocks) {
            if (c == 0) record_error(status, MLA_ERR_BAD_BLOCK_ID, blk);
            continue;
        }
        const uint4* src = reinterpret_cast<const uint4*>(
            cache + (size_t(blk) * kPageSize + (t % kPageSize)) * kD);
        uint4* d = reinterpret_cast<uint4*>(dst + (size_t(b) * dst_max_tokens + t) * kD);
        d[c] = __ldg(src + c);
    }
}

}  // namespace

int launch_gather(const uint16_t* cache, int64_t num_blocks, const int32_t* block_table,
                  const int32_t* seq_lens, int batch, int max_blocks, int dst_max_tokens,
                  uint16_t* dst, int32_t* status, void* stream) {
    if (batch == 0) return 0;
    dim3 grid(64, batch);
    mla_gather_kernel<<<grid, kGatherThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        cache, num_blocks, block_table, seq_lens, max_blocks, dst_max_tokens, dst, status);
    return int(cudaGetLastError());
}

}  // namespace mla
