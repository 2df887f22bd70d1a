// LSE-weighted merge of split partials (mla_merge_splits).
//
// One warp per (request, head) row, or per row and 128-column group when the
// rows are few. The S log-sum-exps are reduced first (max, then the sum of
// exponentials), giving the merged LSE and one weight per split; the warp then
// streams the S partial rows of fp32 values, 16 bytes per lane per load, and
// writes the weighted sum rounded to bf16.
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

// Few rows (a small batch with many splits) leave most SMs idle with one warp
// per row, so the value columns are then cut into 128-wide groups, one per
// CTA row of the grid: CTA (x, y) covers rows 8x..8x+7 and columns
// 128y..128y+127, and each warp keeps four partials' loads in flight.
// Otherwise CTA x covers rows 8x..8x+7 and each warp walks its whole row
// (with at most 4 partials, issuing all of its loads first).
// Every warp first forms its row's LSE and the S weights; a partial with
// weight 0 (an empty split, a rank without tokens) is never read.
//
// Partial s of row r starts at o_part + r * o_row + s * o_split (elements,
// multiples of 4) and its LSE is lse_part[r * l_row + s * l_split]: the split
// schedule's [rows, S, v_dim] and the context-parallel [S, rows, v_dim] are
// both such layouts. The partials are fp32 or bf16 (TP = uint16_t).
constexpr int kChunkedMergeRows = 2048;   // below this many rows: column groups

struct MergeArgs {
    const float* lse_part;
    int rows, S, v_dim;
    int64_t o_row, o_split, l_row, l_split;
    uint16_t* out;
    float* lse;
};

__device__ __forceinline__ float4 load_partial4(const float* p) {
    return __ldg(reinterpret_cast<const float4*>(p));
}

__device__ __forceinline__ float4 load_partial4(const uint16_t* p) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}

__device__ __forceinline__ void store_bf16x4(uint16_t* p, float4 r) {
    uint2 packed;
    packed.x = uint32_t(f32_to_bf16_bits_rn(r.x)) | (uint32_t(f32_to_bf16_bits_rn(r.y)) << 16);
    packed.y = uint32_t(f32_to_bf16_bits_rn(r.z)) | (uint32_t(f32_to_bf16_bits_rn(r.w)) << 16);
    *reinterpret_cast<uint2*>(p) = packed;
}

// Row layouts with at most 4 partials of 512 values: a lane issues the loads
// of two column groups for every partial (8) before using any.
constexpr int kFewSplits = 4;

template <typename TP, int kMode>   // 0: whole rows, 1: column groups, 2: few partials
__global__ void __launch_bounds__(kMergeThreads, 4) mla_merge_kernel(const TP* __restrict__ o_part,
                                                                   const MergeArgs a) {
    __shared__ float weights[kRowsPerCta][kMaxMergeSplits];
    // Launched as a programmatic dependent of the decode kernel: the CTAs may
    // be placed while its grid finishes; this waits for it (and its writes).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kRowsPerCta + warp;
    if (row >= a.rows) return;
    const int S = a.S;

    const float* ls = a.lse_part + row * a.l_row;
    float m = -INFINITY;
    for (int s = lane; s < S; s += 32) m = fmaxf(m, ls[s * a.l_split]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));

    float* w = weights[warp];
    float total = -INFINITY;
    if (m != -INFINITY) {
        float z = 0.f;
        for (int s = lane; s < S; s += 32) z += expf(ls[s * a.l_split] - m);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
        total = m + logf(z);
        for (int s = lane; s < S; s += 32) w[s] = expf(ls[s * a.l_split] - total);
    } else {
        for (int s = lane; s < S; s += 32) w[s] = 0.f;
    }
    __syncwarp();
    if (lane == 0 && a.lse != nullptr && blockIdx.y == 0) a.lse[row] = total;

    const TP* base = o_part + row * a.o_row;
    uint16_t* dst = a.out + size_t(row) * a.v_dim;
    if constexpr (kMode == 2) {
        float wk[kFewSplits];
#pragma unroll
        for (int k = 0; k < kFewSplits; ++k) wk[k] = k < S ? w[k] : 0.f;
#pragma unroll
        for (int g0 = 0; g0 < 4; g0 += 2) {   // two column groups' loads at a time
            float4 v[2][kFewSplits];
#pragma unroll
            for (int g = 0; g < 2; ++g)
#pragma unroll
                for (int k = 0; k < kFewSplits; ++k)
                    v[g][k] = wk[k] != 0.f
                                  ? load_partial4(base + k * a.o_split + (g0 + g) * 128 + lane * 4)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int k = 0; k < kFewSplits; ++k) {
                    acc.x = fmaf(wk[k], v[g][k].x, acc.x);
                    acc.y = fmaf(wk[k], v[g][k].y, acc.y);
                    acc.z = fmaf(wk[k], v[g][k].z, acc.z);
                    acc.w = fmaf(wk[k], v[g][k].w, acc.w);
                }
                store_bf16x4(dst + (g0 + g) * 128 + lane * 4, acc);
            }
        }
    } else if constexpr (kMode == 1) {
        const int d = int(blockIdx.y) * 128 + lane * 4;
        if (d >= a.v_dim) return;
        float4 acc[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s0 = 0; s0 < S; s0 += 4) {
            float4 v[4];
            float ws[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int s = s0 + k;
                ws[k] = s < S ? w[s] : 0.f;
                v[k] = ws[k] != 0.f ? load_partial4(base + s * a.o_split + d)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                acc[k].x = fmaf(ws[k], v[k].x, acc[k].x);
                acc[k].y = fmaf(ws[k], v[k].y, acc[k].y);
                acc[k].z = fmaf(ws[k], v[k].z, acc[k].z);
                acc[k].w = fmaf(ws[k], v[k].w, acc[k].w);
            }
        }
        store_bf16x4(dst + d, make_float4((acc[0].x + acc[1].x) + (acc[2].x + acc[3].x),
                              (acc[0].y + acc[1].y) + (acc[2].y + acc[3].y),
                              (acc[0].z + acc[1].z) + (acc[2].z + acc[3].z),
                              (acc[0].w + acc[1].w) + (acc[2].w + acc[3].w)));
    } else {
        for (int d = lane * 4; d < a.v_dim; d += 128) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            const TP* p = base + d;
            for (int s = 0; s < S; ++s, p += a.o_split) {
                const float ws = w[s];
                if (ws == 0.f) continue;
                const float4 v = load_partial4(p);
                acc.x = fmaf(ws, v.x, acc.x);
                acc.y = fmaf(ws, v.y, acc.y);
                acc.z = fmaf(ws, v.z, acc.z);
                acc.w = fmaf(ws, v.w, acc.w);
            }
            store_bf16x4(dst + d, acc);
        }
    }
}

template <typename TP>
int launch_merge_strided(const TP* o_part, const MergeArgs& a, cudaStream_t st) {
    if (a.rows == 0) return 0;
    if (a.v_dim % 4 != 0 || a.o_row % 4 != 0 || a.o_split % 4 != 0)
        return int(cudaErrorInvalidValue);
    const dim3 rows_grid((a.rows + kRowsPerCta - 1) / kRowsPerCta);
    // A programmatic dependent of the kernel before it on the stream (the
    // decode kernel lets its dependents launch as soon as it starts); the
    // kernel waits for that grid before reading anything.
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kMergeThreads, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (a.rows < kChunkedMergeRows) {
        cfg.gridDim = dim3(rows_grid.x, (a.v_dim + 127) / 128);
        e = cudaLaunchKernelEx(&cfg, mla_merge_kernel<TP, 1>, o_part, a);
    } else if (a.S <= kFewSplits && a.v_dim == 512) {
        cfg.gridDim = rows_grid;
        e = cudaLaunchKernelEx(&cfg, mla_merge_kernel<TP, 2>, o_part, a);
    } else {
        cfg.gridDim = rows_grid;
        e = cudaLaunchKernelEx(&cfg, mla_merge_kernel<TP, 0>, o_part, a);
    }
    return int(e);
}

// Merge of the page-balanced schedule: CTA (b, y) handles request b, heads
// 8y..8y+7, one warp per head. The request's page offset and the batch's page
// total come from a block reduction over seq_lens, which gives the CTA pairs
// whose ranges touch the request (the same cut as the decode kernel's). A
// request inside one range was written by the decode kernel; a request
// without pages gets O = 0 and LSE = -inf; the others combine one partial per
// range, slot 2c or 2c + 1, with the LSE-weighted sum of merge_attn_states.
constexpr int kBalMergeWarps = 8;
constexpr int32_t kMergeWaitSite = 20;   // detail of MLA_ERR_TIMEOUT: the merge's wait for pieces

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__global__ void __launch_bounds__(kBalMergeWarps * 32) mla_merge_balanced_kernel(const DecodeParams p) {
    __shared__ int64_t red_before[kBalMergeWarps], red_total[kBalMergeWarps];
    __shared__ float weights[kBalMergeWarps][kMaxBalancedPairs];
    __shared__ int slots[kMaxBalancedPairs];
    __shared__ int pieces_ready;
    const int b = blockIdx.x;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int N = p.num_heads;
    const int h = blockIdx.y * kBalMergeWarps + warp;
    auto pages_checked = [&](int i) {
        const int L = p.seq_lens[i];
        return (L < 0 || int64_t(L) > int64_t(p.max_blocks) * kPageSize) ? 0 : pages_of(L);
    };
    int64_t before = 0, total = 0;   // work units
    for (int i = threadIdx.x; i < p.batch; i += blockDim.x) {
        const int pg = work_units(pages_checked(i));
        total += pg;
        if (i < b) before += pg;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        before += __shfl_xor_sync(0xffffffffu, before, o);
        total += __shfl_xor_sync(0xffffffffu, total, o);
    }
    if (lane == 0) {
        red_before[warp] = before;
        red_total[warp] = total;
    }
    __syncthreads();
    before = 0;
    total = 0;
    for (int w = 0; w < kBalMergeWarps; ++w) {
        before += red_before[w];
        total += red_total[w];
    }
    const int pages_b = pages_checked(b);
    // The request's pages occupy units [pb, pe), after its fixed cost.
    const int64_t pb = before + kSegmentCostPages, pe = before + work_units(pages_b);
    const int C = p.sched_pairs;

    if (pages_b == 0) {
        // No pages: O = 0, LSE = -inf.
        if (h < N) {
            const size_t orow = size_t(io_row(p, b)) * N + h;
            uint4* dst = reinterpret_cast<uint4*>(p.out + orow * kLkv);
            for (int i = lane; i < kLkv / 8; i += 32) dst[i] = make_uint4(0, 0, 0, 0);
            if (lane == 0 && p.lse != nullptr) p.lse[orow] = -INFINITY;
        }
        return;
    }
    const int c_lo = pair_of_page(pb, C, total);
    const int c_hi = pair_of_page(pe - 1, C, total);
    if (c_lo == c_hi) return;   // inside one range: written by the decode kernel
    const int pieces = c_hi - c_lo + 1;
    for (int i = threadIdx.x; i < pieces; i += blockDim.x) {
        const int c = c_lo + i;
        // b is the first request with pages in range c unless an earlier
        // request's pages reach into it (its range starts before b's units).
        slots[i] = pair_begin(c, C, total) >= before ? 2 * c : 2 * c + 1;
    }
    // This kernel may run while the decode grid is still working on other
    // requests: wait until every piece of request b is written (each piece
    // counts kPieceArrivals softmax warps). Bounded: four times the call's
    // wait limit (4 s), then MLA_ERR_TIMEOUT and no output for the request.
    int32_t* ready = p.counters + kReadyWord + b;
    if (threadIdx.x == 0) {
        const int target = kPieceArrivals * pieces;
        const uint64_t t0 = globaltimer_ns();
        int ok = 1;
        while (*reinterpret_cast<volatile int32_t*>(ready) < target) {
            if (globaltimer_ns() - t0 > 4 * p.timeout_ns) {
                record_error(p.status, MLA_ERR_TIMEOUT, kMergeWaitSite);
                ok = 0;
                break;
            }
            __nanosleep(200);
        }
        pieces_ready = ok;
    }
    __syncthreads();
    __threadfence();
    const bool go = pieces_ready != 0;
    if (go && h < N) {
        float* w = weights[warp];
        float m = -INFINITY;
        for (int i = lane; i < pieces; i += 32)
            m = fmaxf(m, __ldcg(p.lse_part + size_t(slots[i]) * N + h));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float lse_h = -INFINITY;
        if (m != -INFINITY) {
            float z = 0.f;
            for (int i = lane; i < pieces; i += 32)
                z += expf(__ldcg(p.lse_part + size_t(slots[i]) * N + h) - m);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
            lse_h = m + logf(z);
            for (int i = lane; i < pieces; i += 32)
                w[i] = expf(__ldcg(p.lse_part + size_t(slots[i]) * N + h) - lse_h);
        } else {
            for (int i = lane; i < pieces; i += 32) w[i] = 0.f;
        }
        __syncwarp();
        const size_t orow = size_t(io_row(p, b)) * N + h;
        if (lane == 0 && p.lse != nullptr) p.lse[orow] = lse_h;
        // Lane l owns columns 4l + 128k (k = 0..3): four independent 16-byte
        // loads per piece in flight (L2 only: the rows were written by
        // another grid that may still be running).
        float4 acc[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i = 0; i < pieces; ++i) {
            const float wi = w[i];
            if (wi == 0.f) continue;
            const float* src = p.o_part + (size_t(slots[i]) * N + h) * kLkv + lane * 4;
            float4 v[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) v[k] = __ldcg(reinterpret_cast<const float4*>(src + 128 * k));
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                acc[k].x = fmaf(wi, v[k].x, acc[k].x);
                acc[k].y = fmaf(wi, v[k].y, acc[k].y);
                acc[k].z = fmaf(wi, v[k].z, acc[k].z);
                acc[k].w = fmaf(wi, v[k].w, acc[k].w);
            }
        }
        uint16_t* dst = p.out + orow * kLkv + lane * 4;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint2 packed;
            packed.x = uint32_t(f32_to_bf16_bits_rn(acc[k].x)) |
                       (uint32_t(f32_to_bf16_bits_rn(acc[k].y)) << 16);
            packed.y = uint32_t(f32_to_bf16_bits_rn(acc[k].z)) |
                       (uint32_t(f32_to_bf16_bits_rn(acc[k].w)) << 16);
            *reinterpret_cast<uint2*>(dst + 128 * k) = packed;
        }
    }
    // Every warp of the request's CTAs counts itself once its CTA has seen
    // the pieces; the last one resets both counters for the next call.
    __syncwarp();
    if (lane == 0 && go) {
        int32_t* done = p.counters + kDoneWord + b;
        if (atomicAdd(done, 1) == int(gridDim.y) * kBalMergeWarps - 1) {
            *reinterpret_cast<volatile int32_t*>(ready) = 0;
            *reinterpret_cast<volatile int32_t*>(done) = 0;
        }
    }
}

}  // namespace

int launch_merge_balanced(const DecodeParams& p, void* stream) {
    if (p.batch == 0) return 0;
    if (p.sched_pairs < 1 || p.sched_pairs > kMaxBalancedPairs) return int(cudaErrorInvalidValue);
    const dim3 grid(unsigned(p.batch), unsigned((p.num_heads + kBalMergeWarps - 1) / kBalMergeWarps));
    // A programmatic dependent of the decode kernel: its CTAs (about 9 KB of
    // shared memory each, so none fits beside a decode CTA) start on SMs the
    // decode grid has left and wait for their requests' pieces themselves.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kBalMergeWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return int(cudaLaunchKernelEx(&cfg, mla_merge_balanced_kernel, p));
}

int launch_merge(const float* o_part, const float* lse_part, int rows, int num_splits,
                 int v_dim, uint16_t* out, float* lse, void* stream) {
    const MergeArgs a{lse_part, rows, num_splits, v_dim, int64_t(num_splits) * v_dim, v_dim,
                      num_splits, 1, out, lse};
    return launch_merge_strided(o_part, a, static_cast<cudaStream_t>(stream));
}

int launch_merge_bf16(const uint16_t* o_part, const float* lse_part, int rows, int num_splits,
                      int v_dim, uint16_t* out, float* lse, void* stream) {
    const MergeArgs a{lse_part, rows, num_splits, v_dim, int64_t(num_splits) * v_dim, v_dim,
                      num_splits, 1, out, lse};
    return launch_merge_strided(o_part, a, static_cast<cudaStream_t>(stream));
}

int launch_rank_combine(const uint16_t* out_parts, const float* lse_parts, int world, int rows,
                        int v_dim, uint16_t* out, float* lse, void* stream) {
    const MergeArgs a{lse_parts, rows, world, v_dim, v_dim, int64_t(rows) * v_dim,
                      1, rows, out, lse};
    return launch_merge_strided(out_parts, a, static_cast<cudaStream_t>(stream));
}

}  // namespace mla
