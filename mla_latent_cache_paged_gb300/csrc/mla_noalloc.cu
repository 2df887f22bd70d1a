// mla_decode_noalloc: the decode for callers that cannot allocate device memory.
//
// Some callers have no way to hand us a workspace: code running inside a
// region that must not allocate (allocation can synchronise the device or is
// forbidden in a latency-critical serving loop), runtimes that own all device
// memory up front through their own pools and expose no allocator, or
// bindings that pass only the tensors of the operation itself. This variant
// runs the same decode kernels as mla_decode, but its scratch (the status
// word and the split partials) lives in one file-scope device array of fixed
// size that every GPU which loads the library keeps until the process exits.
#include <cuda_runtime.h>

#include <cfloat>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "mla_internal.h"

namespace mla {
namespace {

// 32 MiB: room for the status header plus B*N*S split partials up to
// B*N*S = 16,000 or so (2,052 bytes each), e.g. B=32, N=128, S=4.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device. The symbol name
// is only a host-side stand-in, so the address is looked up once per device
// (with that device current) and cached.
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return MLA_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MLA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" int mla_decode_noalloc(const mla_decode_plan_t* plan, const void* q,
                                  const void* latent_cache, int64_t num_blocks,
                                  const int32_t* block_table, const int32_t* seq_lens,
                                  float softmax_scale, void* out, float* lse,
                                  int32_t* device_status, void* stream) {
    int rc = validate_plan(plan);
    if (rc != MLA_OK) return rc;
    if (!q || !latent_cache || !block_table || !seq_lens || !out) return MLA_ERR_INVALID_ARG;
    if (num_blocks < 1 || !std::isfinite(softmax_scale)) return MLA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(latent_cache, 16) || !aligned(out, 16) ||
        !aligned(block_table, 4) || !aligned(seq_lens, 4) || (lse && !aligned(lse, 4)) ||
        (device_status && !aligned(device_status, 4)))
        return MLA_ERR_INVALID_ARG;
    if (plan->workspace_bytes > kNoAllocScratchBytes) return MLA_ERR_SCRATCH_LIMIT;
    if (plan->kernel == MLA_KERNEL_TC && num_blocks > tc_max_blocks()) return MLA_ERR_UNSUPPORTED;
    if (plan->batch == 0) return MLA_OK;

    void* scratch = nullptr;
    rc = scratch_address(&scratch);
    if (rc != MLA_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(scratch);
    int32_t* status = device_status ? device_status : reinterpret_cast<int32_t*>(ws);
    // The array keeps whatever the previous call left: the status words must
    // start at zero; the split partials are written before they are read.
    if (cudaMemsetAsync(status, 0, 2 * sizeof(int32_t), s) != cudaSuccess) return MLA_ERR_CUDA;

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
    p.out = static_cast<uint16_t*>(out);
    p.lse = lse;
    p.status = status;
    p.sched_pairs = plan->sched_pairs;
    if (S > 1 || plan->sched_pairs > 0) {
        p.o_part = reinterpret_cast<float*>(ws + plan->partial_offset);
        p.lse_part = reinterpret_cast<float*>(ws + plan->lse_partial_offset);
    }
    int e = plan->kernel == MLA_KERNEL_TC ? launch_decode_tc(p, plan->grid_ctas, stream)
                                          : launch_decode_simt(p, stream);
    if (e != 0) return MLA_ERR_CUDA;
    if (plan->sched_pairs > 0) {
        if (launch_merge_balanced(p, stream) != 0) return MLA_ERR_CUDA;
    } else if (S > 1) {
        e = launch_merge(p.o_part, p.lse_part, plan->batch * plan->num_heads, S, kLkv, p.out,
                         lse, stream);
        if (e != 0) return MLA_ERR_CUDA;
    }
    return MLA_OK;
}
