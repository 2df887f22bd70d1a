// CUDA-core split-KV decode kernel (MLA_KERNEL_SIMT).
//
// One CTA per (head group of 16, split, request). The CTA streams its split's
// cached tokens in chunks of 32 through shared memory, computes the scaled
// scores with fp32 FMAs, keeps an online softmax (running max m and sum l per
// head, base-2 exponent with the scale folded into log2(e)), and accumulates
// O = sum_t p_t V_t in registers. It is the path for small head counts (the
// 16-head case is HBM- and launch-bound) and the baseline the tensor-core
// kernel is measured against.
//
// Math: vLLM mla_attention API docs, module docstring, "Data-Movement Friendly
// Approach (i.e. forward_mqa)" -- K is the whole 576-wide entry, V its first
// 512 columns; the LSE is the natural log of sum exp(scaled scores) as in
// ModelOpt mla_attention_decode (return_lse).
#include <cuda_runtime.h>

#include <cmath>

#include "mla_device.cuh"

namespace mla {
namespace {

constexpr int kHG = 16;                 // heads per CTA
constexpr int kTT = 32;                 // tokens per chunk
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kDimsPerWarp = kD / kWarps;      // 72
constexpr int kDimsPerThread = kDimsPerWarp / 2;  // 36
constexpr int kChunks16 = kD * 2 / 16;         // 72 16-byte chunks per row
constexpr float kLn2 = 0.693147180559945309f;

struct __align__(16) SimtSmem {
    uint16_t ks[kTT][kD];            // chunk of cache rows (bf16)
    float red[kWarps][kHG][kTT + 1]; // per-warp partial dot products
    float ps[kHG][kTT];              // scores, then probabilities
    float alpha[kHG];
    float m[kHG];
    float l[kHG];
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__global__ void __launch_bounds__(kThreads, 2) mla_decode_simt_kernel(DecodeParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SimtSmem& sm = *reinterpret_cast<SimtSmem*>(smem_raw);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int h0 = blockIdx.x * kHG;
    const int split = blockIdx.y;
    const int b = blockIdx.z;
    const int N = p.num_heads;
    const int S = p.num_splits;

    const int L = checked_seq_len(p, b);
    int t_lo, t_hi;
    split_range(L, S, split, &t_lo, &t_hi);

    // This thread's slice of q for the score step: head (lane % 16), 36 dims.
    const int my_h = lane & 15;
    const int my_d0 = warp * kDimsPerWarp + (lane >> 4) * kDimsPerThread;
    float qreg[kDimsPerThread];
    {
#pragma unroll
        for (int i = 0; i < kDimsPerThread; ++i) qreg[i] = 0.f;
        if ((h0 + my_h) < N) {
            const uint16_t* qrow = p.q + (size_t(b) * N + (h0 + my_h)) * kD + my_d0;
#pragma unroll
            for (int i = 0; i < kDimsPerThread; ++i) qreg[i] = bf16_bits_to_f32(qrow[i]);
        }
    }
    if (tid < kHG) {
        sm.m[tid] = -INFINITY;
        sm.l[tid] = 0.f;
        sm.alpha[tid] = 1.f;
    }
    __syncthreads();

    // Output accumulators: dims 2*tid, 2*tid+1 for every head of the group.
    float acc[kHG][2];
#pragma unroll
    for (int h = 0; h < kHG; ++h) acc[h][0] = acc[h][1] = 0.f;

    const int32_t* table = p.block_table + size_t(b) * p.max_blocks;

    for (int c0 = t_lo; c0 < t_hi; c0 += kTT) {
        // 1. Gather the chunk's rows through the block table (zero past t_hi).
        for (int idx = tid; idx < kTT * kChunks16; idx += kThreads) {
            const int t = idx / kChunks16;
            const int c = idx % kChunks16;
            const int tok = c0 + t;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (tok < t_hi) {
                const int blk = table[tok / kPageSize];
                if (blk >= 0 && int64_t(blk) < p.num_blocks) {
                    const uint4* src = reinterpret_cast<const uint4*>(
                        p.cache + (size_t(blk) * kPageSize + (tok % kPageSize)) * kD);
                    v = __ldg(src + c);
                } else if (c == 0) {
                    record_error(p.status, MLA_ERR_BAD_BLOCK_ID, blk);
                }
            }
            reinterpret_cast<uint4*>(&sm.ks[t][0])[c] = v;
        }
        __syncthreads();

        // 2. Partial scores over this thread's 36 dims, summed over the warp pair.
        for (int t = 0; t < kTT; ++t) {
            const uint2* kp = reinterpret_cast<const uint2*>(&sm.ks[t][my_d0]);
            float a = 0.f;
#pragma unroll
            for (int i = 0; i < kDimsPerThread / 4; ++i) {
                uint2 w = kp[i];
                a = fmaf(qreg[4 * i + 0], bf16_bits_to_f32(w.x & 0xffffu), a);
                a = fmaf(qreg[4 * i + 1], bf16_bits_to_f32(w.x >> 16), a);
                a = fmaf(qreg[4 * i + 2], bf16_bits_to_f32(w.y & 0xffffu), a);
                a = fmaf(qreg[4 * i + 3], bf16_bits_to_f32(w.y >> 16), a);
            }
            a += __shfl_xor_sync(0xffffffffu, a, 16);
            if (lane < 16) sm.red[warp][my_h][t] = a;
        }
        __syncthreads();

        // 3. Reduce over warps -> scaled scores in the log2 domain, masked.
        for (int pair = tid; pair < kHG * kTT; pair += kThreads) {
            const int h = pair / kTT;
            const int t = pair % kTT;
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) s += sm.red[w][h][t];
            const bool seen = c0 + t < t_hi && c0 + t < L - row_shift(p, h0 + h);
            sm.ps[h][t] = seen ? s * p.scale_log2 : -INFINITY;
        }
        __syncthreads();

        // 4. Online softmax: warp w owns heads 2w and 2w+1, lane = token.
#pragma unroll
        for (int j = 0; j < kHG / kWarps; ++j) {
            const int h = warp * (kHG / kWarps) + j;
            const float x = sm.ps[h][lane];
            const float m_old = sm.m[h];
            const float m_new = fmaxf(m_old, warp_max(x));
            float alpha, pr;
            if (m_new == -INFINITY) {
                alpha = 1.f;
                pr = 0.f;
            } else {
                alpha = exp2f(m_old - m_new);
                pr = exp2f(x - m_new);
            }
            const float lsum = warp_sum(pr);
            sm.ps[h][lane] = pr;
            __syncwarp();
            if (lane == 0) {
                sm.alpha[h] = alpha;
                sm.m[h] = m_new;
                sm.l[h] = sm.l[h] * alpha + lsum;
            }
        }
        __syncthreads();

        // 5. O = alpha * O + sum_t p_t * V_t (V = first 512 columns).
        {
#pragma unroll
            for (int h = 0; h < kHG; ++h) {
                const float al = sm.alpha[h];
                acc[h][0] *= al;
                acc[h][1] *= al;
            }
            const int d = 2 * tid;
            for (int t = 0; t < kTT; ++t) {
                const uint32_t w = *reinterpret_cast<const uint32_t*>(&sm.ks[t][d]);
                const float v0 = bf16_bits_to_f32(w & 0xffffu);
                const float v1 = bf16_bits_to_f32(w >> 16);
#pragma unroll
                for (int h = 0; h < kHG; ++h) {
                    const float pr = sm.ps[h][t];
                    acc[h][0] = fmaf(pr, v0, acc[h][0]);
                    acc[h][1] = fmaf(pr, v1, acc[h][1]);
                }
            }
        }
        __syncthreads();
    }

    // 6. Epilogue: normalise; final bf16 output or the split's partial row
    // (bf16, or fp32).
    const int d = 2 * tid;
#pragma unroll
    for (int h = 0; h < kHG; ++h) {
        const int head = h0 + h;
        if (head >= N) break;
        const float l = sm.l[h];
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const float lse = l > 0.f ? (sm.m[h] + log2f(l)) * kLn2 : -INFINITY;
        const size_t row = size_t(b) * N + head;
        if (S == 1) {
            const uint32_t packed = uint32_t(f32_to_bf16_bits_rn(acc[h][0] * inv)) |
                                    (uint32_t(f32_to_bf16_bits_rn(acc[h][1] * inv)) << 16);
            *reinterpret_cast<uint32_t*>(p.out + row * kLkv + d) = packed;
            if (tid == 0 && p.lse != nullptr) p.lse[row] = lse;
        } else {
            const size_t prow = (row * S + split) * kLkv + d;
            if (p.part_bf16) {
                *reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(p.o_part) + prow) =
                    uint32_t(f32_to_bf16_bits_rn(acc[h][0] * inv)) |
                    (uint32_t(f32_to_bf16_bits_rn(acc[h][1] * inv)) << 16);
            } else {
                *reinterpret_cast<float2*>(p.o_part + prow) =
                    make_float2(acc[h][0] * inv, acc[h][1] * inv);
            }
            if (tid == 0) p.lse_part[row * S + split] = lse;
        }
    }
}

}  // namespace

int launch_decode_simt(const DecodeParams& p, void* stream) {
    const size_t smem = sizeof(SimtSmem);
    cudaError_t e = cudaFuncSetAttribute(mla_decode_simt_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return int(e);
    dim3 grid((p.num_heads + kHG - 1) / kHG, p.num_splits, p.batch);
    mla_decode_simt_kernel<<<grid, kThreads, smem, static_cast<cudaStream_t>(stream)>>>(p);
    return int(cudaGetLastError());
}

}  // namespace mla
