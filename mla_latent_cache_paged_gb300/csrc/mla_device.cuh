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

// Tokens row h must not see at the end of its request (multi-token rows).
__device__ __forceinline__ int row_shift(const DecodeParams& p, int h) {
    if (p.q_len <= 1 || !p.causal) return 0;
    const int tok = h / p.heads_per_token;
    return tok < p.q_len ? p.q_len - 1 - tok : 0;
}

// The q / out / lse tensor row of work row r (token-major multi-token rows).
__device__ __forceinline__ int io_row(const DecodeParams& p, int r) {
    return p.row_tokens > 1 ? (r % p.row_batch) * p.row_tokens + r / p.row_batch : r;
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

// ------------------------------------------------------ page-balanced schedule
// Work units: a request with p > 0 pages is kSegmentCostPages units of fixed
// cost followed by its p pages; an empty request is nothing. The batch's
// units, request after request (prefix pfx[b] = units of requests 0..b-1,
// total T), are cut into `pairs` contiguous ranges of near-equal length; CTA
// pair c works through the pages that fall in units
// [pair_begin(c), pair_begin(c + 1)). A request whose pages lie inside one
// range is written directly; one whose pages cross a range boundary leaves a
// partial result in each range it touches, and the merge combines them. A
// range holds at most two partial pieces: that of its first request with
// pages in the range (slot 2c) and that of its last (slot 2c + 1).
__device__ __forceinline__ int work_units(int pages) {
    return pages > 0 ? pages + kSegmentCostPages : 0;
}

__device__ __forceinline__ int64_t pair_begin(int c, int pairs, int64_t total_pages) {
    return int64_t(c) * total_pages / pairs;
}

// The range c holding page g (0 <= g < total_pages).
__device__ __forceinline__ int pair_of_page(int64_t g, int pairs, int64_t total_pages) {
    return int(((g + 1) * pairs + total_pages - 1) / total_pages) - 1;
}

__device__ __forceinline__ int pages_of(int L) { return (L + kPageSize - 1) / kPageSize; }

}  // namespace mla
