// Small device helpers shared by the kernels of libmla_decode.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "mla_internal.h"

namespace mla {

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
    return __uint_as_float(bits16 << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits_rn(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t*>(&h);
}

// Record the first device-side error of a call; later ones are dropped.
__device__ __forceinline__ void record_error(int32_t* status, int32_t code, int32_t detail) {
    if (status != nullptr && atomicCAS(status, 0, code) == 0) {
        atomicExch(status + 1, detail);
    }
}

// Token range [*lo, *hi) of split `s` of a request with L tokens: page-aligned
// chunks of C = page_size * ceil(ceil(L / page_size) / S) tokens.
__device__ __forceinline__ void split_range(int L, int S, int s, int* lo, int* hi) {
    int pages = (L + kPageSize - 1) / kPageSize;
    int chunk = kPageSize * ((pages + S - 1) / S);
    int a = s * chunk;
    int e = a + chunk;
    *lo = a < L ? a : L;
    *hi = e < L ? e : L;
}

// Validated sequence length: a value outside [0, max_blocks * page_size] is
// recorded and the request treated as empty.
__device__ __forceinline__ int checked_seq_len(const DecodeParams& p, int b) {
    int L = p.seq_lens[b];
    if (L < 0 || int64_t(L) > int64_t(p.max_blocks) * kPageSize) {
        record_error(p.status, MLA_ERR_BAD_SEQ_LEN, L);
        return 0;
    }
    return L;
}

}  // namespace mla
