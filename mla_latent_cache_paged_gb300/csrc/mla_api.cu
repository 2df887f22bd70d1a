// C ABI entry points of libmla_decode (declared in include/mla_decode.h).
// Host-side argument checks happen before anything is enqueued; device work
// goes onto the caller's stream without any host synchronisation.
#include <cuda_runtime.h>

#include <cfloat>
#include <climits>
#include <cmath>
#include <cstdint>

#include "mla_internal.h"

using namespace mla;

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int cuda_status(int e) { return e == 0 ? MLA_OK : MLA_ERR_CUDA; }

}  // namespace

extern "C" int mla_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
    if (!workspace || workspace_bytes < kStatusBytes || !aligned(workspace, 256))
        return MLA_ERR_WORKSPACE;
    return cuda_status(int(cudaMemsetAsync(workspace, 0, kStatusBytes,
                                           static_cast<cudaStream_t>(stream))));
}

namespace mla {

DecodeParams make_decode_params(const mla_decode_plan_t* plan, const void* q,
                                const void* latent_cache, int64_t num_blocks,
                                const int32_t* block_table, const int32_t* seq_lens,
                                float softmax_scale, void* out, float* lse, char* ws,
                                int32_t* status, int q_len, int heads_per_token, int causal) {
    const int S = plan->num_kv_splits;
    DecodeParams p{};
    p.q = static_cast<const uint16_t*>(q);
    p.cache = static_cast<const uint16_t*>(latent_cache);
    p.num_blocks = num_blocks;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.max_blocks = plan->max_blocks_per_seq;
    p.batch = plan->batch;
    p.num_heads = plan->num_heads;
    p.num_splits = S;
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    // A zero scale weighs every token 1; the smallest normal scale does the
    // same in fp32 (every scaled score rounds 2^x to 1) and keeps the
    // tensor-core kernel's scaled masking sentinel at -inf.
    if (p.scale_log2 == 0.f) p.scale_log2 = FLT_MIN;
    p.v_scale = 1.f;
    p.out = static_cast<uint16_t*>(out);
    p.lse = lse;
    p.status = status ? status : reinterpret_cast<int32_t*>(ws);
    p.counters = reinterpret_cast<int32_t*>(ws);
    p.sched_pairs = plan->sched_pairs;
    p.q_len = q_len;
    p.heads_per_token = heads_per_token;
    p.causal = causal;
    p.timeout_ns = kDefaultTimeoutNs;
    if (plan->flags & MLA_PLAN_DEBUG_WITHHOLD_LOAD) {
        p.debug = kDebugWithholdLoad;
        p.timeout_ns = kDebugTimeoutNs;
    }
    if (S > 1 || plan->sched_pairs > 0) {
        p.o_part = reinterpret_cast<float*>(ws + plan->partial_offset);
        p.lse_part = reinterpret_cast<float*>(ws + plan->lse_partial_offset);
        p.part_bf16 = plan->sched_pairs == 0 && !(plan->flags & MLA_PLAN_FP32_PARTIALS);
    }
    return p;
}

int launch_decode_and_merge(const DecodeParams& p, const mla_decode_plan_t* plan, void* stream,
                            bool fp8) {
    int e = fp8 ? launch_decode_tc_fp8(p, plan->grid_ctas, stream)
            : plan->kernel == MLA_KERNEL_TC ? launch_decode_tc(p, plan->grid_ctas, stream)
                                            : launch_decode_simt(p, stream);
    if (e != 0) return MLA_ERR_CUDA;
    if (plan->sched_pairs > 0) {
        if (launch_merge_balanced(p, stream) != 0) return MLA_ERR_CUDA;
    } else if (plan->num_kv_splits > 1) {
        e = p.part_bf16
                ? launch_merge_bf16(reinterpret_cast<const uint16_t*>(p.o_part), p.lse_part,
                                    plan->batch * plan->num_heads, plan->num_kv_splits, kLkv,
                                    p.out, p.lse, stream)
                : launch_merge(p.o_part, p.lse_part, plan->batch * plan->num_heads,
                               plan->num_kv_splits, kLkv, p.out, p.lse, stream);
        if (e != 0) return MLA_ERR_CUDA;
    }
    return MLA_OK;
}

int decode_impl(const mla_decode_plan_t* plan, const void* q, const void* latent_cache,
                int64_t num_blocks, const int32_t* block_table, const int32_t* seq_lens,
                float softmax_scale, void* out, float* lse, void* workspace,
                size_t workspace_bytes, void* stream, int q_len, int heads_per_token,
                int causal, int row_tokens) {
    int rc = validate_plan(plan);
    if (rc != MLA_OK) return rc;
    if (!q || !latent_cache || !block_table || !seq_lens || !out) return MLA_ERR_INVALID_ARG;
    if (num_blocks < 1 || !std::isfinite(softmax_scale)) return MLA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(latent_cache, 16) || !aligned(out, 16) ||
        !aligned(block_table, 4) || !aligned(seq_lens, 4) || (lse && !aligned(lse, 4)))
        return MLA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < plan->workspace_bytes || !aligned(workspace, 256))
        return MLA_ERR_WORKSPACE;
    if (plan->kernel == MLA_KERNEL_TC && num_blocks > tc_max_blocks()) return MLA_ERR_UNSUPPORTED;
    if (plan->batch == 0) return MLA_OK;
    DecodeParams p = make_decode_params(plan, q, latent_cache, num_blocks, block_table,
                                        seq_lens, softmax_scale, out, lse,
                                        static_cast<char*>(workspace), nullptr, q_len,
                                        heads_per_token, causal);
    if (row_tokens > 1) {
        p.row_tokens = row_tokens;
        p.row_batch = plan->batch / row_tokens;
    }
    return launch_decode_and_merge(p, plan, stream);
}

}  // namespace mla

extern "C" int mla_decode(const mla_decode_plan_t* plan, const void* q, const void* latent_cache,
                          int64_t num_blocks, const int32_t* block_table, const int32_t* seq_lens,
                          float softmax_scale, void* out, float* lse, void* workspace,
                          size_t workspace_bytes, void* stream) {
    return decode_impl(plan, q, latent_cache, num_blocks, block_table, seq_lens, softmax_scale,
                       out, lse, workspace, workspace_bytes, stream, 1,
                       plan ? plan->num_heads : 1, 0);
}

extern "C" int mla_decode_fp8(const mla_decode_plan_t* plan, const void* q,
                              const void* latent_cache_fp8, int64_t num_blocks,
                              const int32_t* block_table, const int32_t* seq_lens,
                              float softmax_scale, float k_scale, void* out, float* lse,
                              void* workspace, size_t workspace_bytes, void* stream) {
    int rc = validate_plan(plan);
    if (rc != MLA_OK) return rc;
    if (plan->kernel != MLA_KERNEL_TC) return MLA_ERR_UNSUPPORTED;
    if (!q || !latent_cache_fp8 || !block_table || !seq_lens || !out) return MLA_ERR_INVALID_ARG;
    if (num_blocks < 1 || !std::isfinite(softmax_scale) || !std::isfinite(k_scale) ||
        !(k_scale > 0.f))
        return MLA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(latent_cache_fp8, 16) || !aligned(out, 16) ||
        !aligned(block_table, 4) || !aligned(seq_lens, 4) || (lse && !aligned(lse, 4)))
        return MLA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < plan->workspace_bytes || !aligned(workspace, 256))
        return MLA_ERR_WORKSPACE;
    if (num_blocks > tc_max_blocks()) return MLA_ERR_UNSUPPORTED;
    if (plan->batch == 0) return MLA_OK;
    // The cache codes times k_scale are the entries: the scale multiplies
    // every score (folded into the softmax scale) and every output row.
    DecodeParams p = make_decode_params(plan, q, latent_cache_fp8, num_blocks, block_table,
                                        seq_lens, softmax_scale * k_scale, out, lse,
                                        static_cast<char*>(workspace), nullptr, 1,
                                        plan->num_heads, 0);
    p.v_scale = k_scale;
    return launch_decode_and_merge(p, plan, stream, true);
}

extern "C" int mla_decode_v_up_proj(const mla_decode_plan_t* plan, const void* q,
                                    const void* latent_cache, int64_t num_blocks,
                                    const int32_t* block_table, const int32_t* seq_lens,
                                    float softmax_scale, const void* w_uv, void* out, float* lse,
                                    void* latent_out, void* workspace, size_t workspace_bytes,
                                    void* stream) {
    int rc = validate_plan(plan);
    if (rc != MLA_OK) return rc;
    if (!q || !latent_cache || !block_table || !seq_lens || !w_uv || !out)
        return MLA_ERR_INVALID_ARG;
    if (num_blocks < 1 || !std::isfinite(softmax_scale)) return MLA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(latent_cache, 16) || !aligned(out, 16) ||
        !aligned(w_uv, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
        (lse && !aligned(lse, 4)) || (latent_out && !aligned(latent_out, 16)))
        return MLA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < plan->workspace_bytes || !aligned(workspace, 256))
        return MLA_ERR_WORKSPACE;
    if (plan->kernel == MLA_KERNEL_TC && num_blocks > tc_max_blocks()) return MLA_ERR_UNSUPPORTED;
    const bool fused = plan->sched_pairs == 0 && plan->num_kv_splits > 1 &&
                       plan->num_kv_splits <= kMaxFusedMergeSplits;
    // Without a split merge to fuse into, the decode writes the latent rows
    // and the up-projection reads them back: the caller provides them.
    if (!fused && !latent_out) return MLA_ERR_INVALID_ARG;
    if (plan->batch == 0) return MLA_OK;
    char* ws = static_cast<char*>(workspace);
    if (!fused) {
        const DecodeParams p = make_decode_params(plan, q, latent_cache, num_blocks, block_table,
                                                  seq_lens, softmax_scale, latent_out, lse, ws,
                                                  nullptr, 1, plan->num_heads, 0);
        rc = launch_decode_and_merge(p, plan, stream);
        if (rc != MLA_OK) return rc;
        return mla_v_up_proj(latent_out, w_uv, plan->batch, plan->num_heads, out, workspace,
                             workspace_bytes, stream);
    }
    // Split schedule: the decode leaves fp32 partials, merged straight into
    // the up-projection's operand tile.
    const DecodeParams p = make_decode_params(plan, q, latent_cache, num_blocks, block_table,
                                              seq_lens, softmax_scale, out, lse, ws, nullptr, 1,
                                              plan->num_heads, 0);
    int e = plan->kernel == MLA_KERNEL_TC ? launch_decode_tc(p, plan->grid_ctas, stream)
                                          : launch_decode_simt(p, stream);
    if (e != 0) return MLA_ERR_CUDA;
    e = launch_merge_up_proj(p.o_part, p.part_bf16 != 0, p.lse_part, plan->batch, plan->num_heads,
                             plan->num_kv_splits, w_uv, static_cast<uint16_t*>(out), lse,
                             static_cast<uint16_t*>(latent_out), p.status, stream);
    return e == 0 ? MLA_OK : MLA_ERR_CUDA;
}

extern "C" int mla_merge_splits(const float* o_part, const float* lse_part, int batch,
                                int num_heads, int num_splits, int v_dim, void* out, float* lse,
                                void* stream) {
    if (batch < 0 || num_heads < 0 || num_splits < 1 || num_splits > kMaxMergeSplits)
        return MLA_ERR_INVALID_ARG;
    if (int64_t(batch) * num_heads > INT_MAX) return MLA_ERR_UNSUPPORTED;
    if (v_dim < 8 || v_dim > 2048 || v_dim % 8 != 0) return MLA_ERR_UNSUPPORTED;
    if (batch == 0 || num_heads == 0) return MLA_OK;
    if (!o_part || !lse_part || !out) return MLA_ERR_INVALID_ARG;
    if (!aligned(o_part, 16) || !aligned(lse_part, 4) || !aligned(out, 8) ||
        (lse && !aligned(lse, 4)))
        return MLA_ERR_INVALID_ARG;
    return cuda_status(launch_merge(o_part, lse_part, batch * num_heads, num_splits, v_dim,
                                    static_cast<uint16_t*>(out), lse, stream));
}

extern "C" int mla_dcp_combine(const void* out_parts, const float* lse_parts, int world,
                               int batch, int num_heads, int v_dim, void* out, float* lse,
                               void* stream) {
    if (batch < 0 || num_heads < 0 || world < 1 || world > kMaxMergeSplits)
        return MLA_ERR_INVALID_ARG;
    if (int64_t(batch) * num_heads > INT_MAX) return MLA_ERR_UNSUPPORTED;
    if (v_dim < 8 || v_dim > 2048 || v_dim % 8 != 0) return MLA_ERR_UNSUPPORTED;
    if (batch == 0 || num_heads == 0) return MLA_OK;
    if (!out_parts || !lse_parts || !out) return MLA_ERR_INVALID_ARG;
    if (!aligned(out_parts, 8) || !aligned(lse_parts, 4) || !aligned(out, 8) ||
        (lse && !aligned(lse, 4)))
        return MLA_ERR_INVALID_ARG;
    return cuda_status(launch_rank_combine(static_cast<const uint16_t*>(out_parts), lse_parts,
                                           world, batch * num_heads, v_dim,
                                           static_cast<uint16_t*>(out), lse, stream));
}

extern "C" int mla_read_error(void* workspace, int* device_status, void* stream) {
    if (!workspace || !device_status) return MLA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_CUDA;
    int32_t words[2] = {0, 0};
    if (cudaMemcpy(words, workspace, sizeof(words), cudaMemcpyDeviceToHost) != cudaSuccess)
        return MLA_ERR_CUDA;
    if (cudaMemset(workspace, 0, sizeof(words)) != cudaSuccess) return MLA_ERR_CUDA;
    *device_status = words[0];
    return MLA_OK;
}

extern "C" int mla_debug_loader_pages(const mla_decode_plan_t* plan, const void* latent_cache,
                                      int64_t num_blocks, const int32_t* block_table,
                                      const int32_t* seq_lens, int dst_max_tokens, void* dst,
                                      void* workspace, size_t workspace_bytes, void* stream) {
    int rc = validate_plan(plan);
    if (rc != MLA_OK) return rc;
    if (plan->kernel != MLA_KERNEL_TC) return MLA_ERR_UNSUPPORTED;
    if (!latent_cache || !block_table || !seq_lens || !dst || dst_max_tokens < 0 ||
        num_blocks < 1)
        return MLA_ERR_INVALID_ARG;
    if (!aligned(latent_cache, 16) || !aligned(dst, 16) || !aligned(block_table, 4) ||
        !aligned(seq_lens, 4))
        return MLA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < kStatusBytes || !aligned(workspace, 256))
        return MLA_ERR_WORKSPACE;
    if (num_blocks > tc_max_blocks()) return MLA_ERR_UNSUPPORTED;
    if (plan->batch == 0) return MLA_OK;
    DecodeParams p{};
    p.cache = static_cast<const uint16_t*>(latent_cache);
    p.num_blocks = num_blocks;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.max_blocks = plan->max_blocks_per_seq;
    p.batch = plan->batch;
    p.num_heads = plan->num_heads;
    p.num_splits = plan->num_kv_splits;
    p.sched_pairs = plan->sched_pairs;
    p.status = static_cast<int32_t*>(workspace);
    p.counters = static_cast<int32_t*>(workspace);
    p.q_len = 1;
    p.heads_per_token = plan->num_heads;
    p.timeout_ns = kDefaultTimeoutNs;
    p.dump = static_cast<uint16_t*>(dst);
    p.dump_max_tokens = dst_max_tokens;
    return cuda_status(launch_decode_tc_loader_dump(p, plan->grid_ctas, stream));
}

extern "C" int mla_debug_gather_pages(const void* latent_cache, int64_t num_blocks,
                                      const int32_t* block_table, const int32_t* seq_lens,
                                      int batch, int max_blocks_per_seq, int dst_max_tokens,
                                      void* dst, void* workspace, size_t workspace_bytes,
                                      void* stream) {
    if (batch < 0 || max_blocks_per_seq < 1 || dst_max_tokens < 0 || num_blocks < 1)
        return MLA_ERR_INVALID_ARG;
    if (batch == 0) return MLA_OK;
    if (!latent_cache || !block_table || !seq_lens || !dst) return MLA_ERR_INVALID_ARG;
    if (!aligned(latent_cache, 16) || !aligned(dst, 16)) return MLA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < kStatusBytes || !aligned(workspace, 256))
        return MLA_ERR_WORKSPACE;
    return cuda_status(launch_gather(static_cast<const uint16_t*>(latent_cache), num_blocks,
                                     block_table, seq_lens, batch, max_blocks_per_seq,
                                     dst_max_tokens, static_cast<uint16_t*>(dst),
                                     static_cast<int32_t*>(workspace), stream));
}
