// LSE-weighted merge of split partials (mla_merge_splits).
//
// One warp per (request, head) row. The S log-sum-exps are reduced first
// (max, then the sum of exponentials), giving the merged LSE and one weight
// per split; the warp then streams the S partial rows of v_dim fp32 values,
// 16 bytes per lane per load, and writes the weighted sum rounded to bf16.
// Formula: the merge the vLLM pages call merge_attn_states (mla_attention API
// docs, "Chunked Prefill"); a zero partial with -inf LSE is the neutral
// element (neutralize_empty_context_partials).
#include <cuda_runtime.h>

#include <cmath>

#include "mla_device.cuh"

namespace mla {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kRowsPerCta = kMergeThreads / 32;

__global__ void __launch_bounds__(kMergeThreads) mla_merge_kernel(
        const float* __restrict__ o_part, const float* __restrict__ lse_part, int rows,
        int S, int v_dim, uint16_t* __restrict__ out, float* __restrict__ lse) {
    __shared__ float weights[kRowsPerCta][kMaxMergeSplits];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kRowsPerCta + warp;
    if (row >= rows) return;

    const float* ls = lse_part + size_t(row) * S;
    float m = -INFINITY;
    for (int s = lane; s < S; s += 32) m = fmaxf(m, ls[s]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));

    float* w = weights[warp];
    float total = -INFINITY;
    if (m != -INFINITY) {
        float z = 0.f;
        for (int s = lane; s < S; s += 32) z += expf(ls[s] - m);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
        total = m + logf(z);
        for (int s = lane; s < S; s += 32) w[s] = expf(ls[s] - total);
    } else {
        for (int s = lane; s < S; s += 32) w[s] = 0.f;
    }
    __syncwarp();
    if (lane == 0 && lse != nullptr) lse[row] = total;

    const float* base = o_part + size_t(row) * S * v_dim;
    uint16_t* dst = out + size_t(row) * v_dim;
    for (int d = lane * 4; d < v_dim; d += 128) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s = 0; s < S; ++s) {
            const float ws = w[s];
            if (ws == 0.f) continue;   // neutral partials (also skips their contents)
            const float4 v = __ldg(reinterpret_cast<const float4*>(base + size_t(s) * v_dim + d));
            acc.x = fmaf(ws, v.x, acc.x);
            acc.y = fmaf(ws, v.y, acc.y);
            acc.z = fmaf(ws, v.z, acc.z);
            acc.w = fmaf(ws, v.w, acc.w);
        }
        uint2 packed;
        packed.x = uint32_t(f32_to_bf16_bits_rn(acc.x)) | (uint32_t(f32_to_bf16_bits_rn(acc.y)) << 16);
        packed.y = uint32_t(f32_to_bf16_bits_rn(acc.z)) | (uint32_t(f32_to_bf16_bits_rn(acc.w)) << 16);
        *reinterpret_cast<uint2*>(dst + d) = packed;
    }
}

}  // namespace

int launch_merge(const float* o_part, const float* lse_part, int rows, int num_splits,
                 int v_dim, uint16_t* out, float* lse, void* stream) {
    if (rows == 0) return 0;
    dim3 grid((rows + kRowsPerCta - 1) / kRowsPerCta);
    mla_merge_kernel<<<grid, kMergeThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        o_part, lse_part, rows, num_splits, v_dim, out, lse);
    return int(cudaGetLastError());
}

}  // namespace mla
