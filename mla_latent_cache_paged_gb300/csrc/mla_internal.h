// Internal declarations shared by the translation units of libmla_decode.
#pragma once

#include <cstddef>
#include <cstdint>

#include "mla_decode.h"

namespace mla {

constexpr int kLkv = 512;          // latent width = V head dim of the absorbed path
constexpr int kRope = 64;          // RoPE width
constexpr int kD = kLkv + kRope;   // one cache entry = absorbed q/k head dim
constexpr int kPageSize = 64;      // tokens per block
constexpr int kMaxHeads = 128;
constexpr size_t kStatusBytes = 8192;  // status header at the start of the workspace
constexpr int kMaxMergeSplits = 1024;
constexpr int kMaxBalancedBatch = 512;   // the page-balanced schedule keeps B+1 offsets in smem
constexpr int kMaxBalancedPairs = 256;   // pieces one merged row can have
// Page-balanced schedule: a request with pages counts as its pages plus this
// many pages of work for the cut (q staging and the epilogue a CTA pair pays
// for each request it touches).
constexpr int kSegmentCostPages = 5;
constexpr int kReadyWord = 64;
constexpr int kDoneWord = kReadyWord + kMaxBalancedBatch;
constexpr int kPieceArrivals = 8;   // increments of kReadyWord + b per partial row set
static_assert((kDoneWord + kMaxBalancedBatch) * 4 <= int(kStatusBytes), "status header too small");

// Layout of the status header (int32 words).
//   [0] first MLA_ERR_* recorded by a kernel (0 = none)
//   [1] detail: the offending block id / seq_len / wait site
//   [kReadyWord + b]  page-balanced schedule: softmax warps (4 per CTA, both
//                     CTAs of a pair) that wrote their part of a partial row
//                     set of request b in this call
//   [kDoneWord + b]   merge warps done with request b; the last one resets
//                     both words to 0 for the next call
constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;   // 1 s
// Test-only behaviour of the tensor-core decode kernel (DecodeParams.debug):
// CTA 0 never issues its first K-ring load, so the score warp's wait for it
// runs out (no fault: the wait is bounded and the kernel drains and returns).
constexpr uint32_t kDebugWithholdLoad = 0x1u;
// Wait limit that MLA_PLAN_DEBUG_WITHHOLD_LOAD sets (2 ms).
constexpr uint64_t kDebugTimeoutNs = 2000000ull;

struct StatusWords {
    int32_t code;
    int32_t detail;
};

// Everything a decode kernel needs for one call.
struct DecodeParams {
    const uint16_t* q;            // bf16 [B, N, 576]
    const uint16_t* cache;        // bf16 [num_blocks, 64, 576]
    int64_t num_blocks;
    const int32_t* block_table;   // [B, max_blocks]
    const int32_t* seq_lens;      // [B]
    int32_t max_blocks;
    int32_t batch;
    int32_t num_heads;
    int32_t num_splits;           // S of the split schedule (1 when sched_pairs > 0)
    int32_t sched_pairs;          // > 0: page-balanced schedule over this many CTA pairs
    float scale_log2;             // softmax_scale * log2(e) (* k_scale for an fp8 cache)
    float v_scale;                // multiplies the output: 1, or k_scale for an fp8 cache
    uint16_t* out;                // bf16 [B, N, 512]
    float* lse;                   // fp32 [B, N] or null
    float* o_part;                // fp32 partial rows: [B, N, S, 512] (split, S > 1)
                                  //                    or [2 * pairs, N, 512] (balanced)
    float* lse_part;              // fp32 [B, N, S] or [2 * pairs, N]
    int32_t part_bf16;            // split schedule: partial rows stored as bf16
    int32_t* status;              // error word and its detail (int32[2])
    int32_t* counters;            // status header holding the page-balanced merge's
                                  // per-request counters ([kReadyWord + b], [kDoneWord + b])
    uint64_t timeout_ns;          // limit of a bounded wait (kDefaultTimeoutNs unless a
                                  // test shortens it)
    uint32_t debug;               // kDebug* bits (tests only; 0 in normal calls)
    uint16_t* dump;               // loader dump: bf16 [2, B, dump_max_tokens, 576] or null
    int32_t dump_max_tokens;
    // Uniform multi-token decode with the query tokens' heads as rows: row h
    // is head h % heads_per_token of query token h / heads_per_token; with
    // `causal` that token sees q_len - 1 - token fewer of the request's
    // tokens. A plain decode has q_len = 1.
    int32_t q_len;
    int32_t heads_per_token;
    int32_t causal;
    // Multi-token rows in token-major order (row r = i * row_batch + b is
    // query token i of request b): q, out and lse of row r are at tensor row
    // b * row_tokens + i. row_tokens <= 1: row r is tensor row r.
    int32_t row_tokens;
    int32_t row_batch;
};


// Launchers (return a cudaError_t as int; 0 = success).
int launch_decode_simt(const DecodeParams& p, void* stream);
int launch_decode_tc(const DecodeParams& p, int grid_ctas, void* stream);
// The tensor-core kernel's page loaders alone (no MMAs): every page each CTA
// receives is copied from its shared-memory rings to p.dump.
int launch_decode_tc_loader_dump(const DecodeParams& p, int grid_ctas, void* stream);
// The tensor-core kernel over an fp8 (E4M3) cache: p.cache holds the codes.
int launch_decode_tc_fp8(const DecodeParams& p, int grid_ctas, void* stream);
int launch_merge(const float* o_part, const float* lse_part, int rows, int num_splits,
                 int v_dim, uint16_t* out, float* lse, void* stream);
// The same over bf16 partial rows.
int launch_merge_bf16(const uint16_t* o_part, const float* lse_part, int rows, int num_splits,
                      int v_dim, uint16_t* out, float* lse, void* stream);
// Combine of per-rank results in rank-major layout: bf16 [world, rows, v_dim]
// and fp32 [world, rows] -> bf16 [rows, v_dim], fp32 [rows].
int launch_rank_combine(const uint16_t* out_parts, const float* lse_parts, int world, int rows,
                        int v_dim, uint16_t* out, float* lse, void* stream);
int launch_merge_balanced(const DecodeParams& p, void* stream);
// Merge of split partials [B, N, S, 512] straight into the up-projection by
// W_UV [N, 512, 128] (mla_bmm.cu): out bf16 [B, N, 128], lse [B, N] and the
// merged bf16 rows [B, N, 512] (each optional: null skips it).
// (o_part holds bf16 rows when part_bf16.)
int launch_merge_up_proj(const void* o_part, bool part_bf16, const float* lse_part, int batch,
                         int num_heads, int num_splits, const void* w_uv, uint16_t* out,
                         float* lse, uint16_t* latent, int32_t* status, void* stream);
constexpr int kMaxFusedMergeSplits = 512;
int launch_gather(const uint16_t* cache, int64_t num_blocks, const int32_t* block_table,
                  const int32_t* seq_lens, int batch, int max_blocks, int dst_max_tokens,
                  uint16_t* dst, int32_t* status, void* stream);

// The parameters of one decode call under `plan` (status and counters both
// in the status header `ws` unless `status` is given).
DecodeParams make_decode_params(const mla_decode_plan_t* plan, const void* q,
                                const void* latent_cache, int64_t num_blocks,
                                const int32_t* block_table, const int32_t* seq_lens,
                                float softmax_scale, void* out, float* lse, char* ws,
                                int32_t* status, int q_len, int heads_per_token, int causal);
// The decode kernel of `plan` (the fp8-cache kernel with `fp8`), then its
// merge (S > 1 or page-balanced).
int launch_decode_and_merge(const DecodeParams& p, const mla_decode_plan_t* plan, void* stream,
                            bool fp8 = false);

// mla_decode with multi-token rows (q_len query tokens' heads as the rows;
// q_len = 1 is the plain decode).
int decode_impl(const mla_decode_plan_t* plan, const void* q, const void* latent_cache,
                int64_t num_blocks, const int32_t* block_table, const int32_t* seq_lens,
                float softmax_scale, void* out, float* lse, void* workspace,
                size_t workspace_bytes, void* stream, int q_len, int heads_per_token,
                int causal, int row_tokens = 1);

// Host-side helpers from mla_plan.cpp.
int validate_plan(const mla_decode_plan_t* plan);
bool tc_kernel_built();
int tc_max_blocks();

}  // namespace mla
