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

#include <cmath>
#include <cstdint>
#include <mutex>

#include "mla_internal.h"

namespace mla {
namespace {

// 32 MiB: room for the 8 KiB status header plus the partial rows of a plan,
// each of its two arrays rounded up to 256 bytes. A split row (request, head,
// split) takes 1,028 bytes (bf16 row + fp32 LSE): up to 32,632 rows, e.g.
// B=32, N=128, S=7 (28,672 rows; S=8 is 32,768); with MLA_PLAN_FP32_PARTIALS
// 2,052 bytes: up to 16,348 rows. A page-balanced plan over C CTA pairs has
// 2*C*N fp32 rows (C=32, N=128: 8,192).
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
    // The array keeps whatever the previous call left. The status words
    // start at zero; so do the page-balanced merge's counters, which stay in
    // the array's own status header even when the status goes to
    // device_status (a call that timed out may have left them non-zero, and
    // the caller cannot re-initialise this array). The split partials are
    // written before they are read.
    if (cudaMemsetAsync(ws, 0, kStatusBytes, s) != cudaSuccess) return MLA_ERR_CUDA;
    if (device_status && cudaMemsetAsync(device_status, 0, 2 * sizeof(int32_t), s) != cudaSuccess)
        return MLA_ERR_CUDA;
    const DecodeParams p = make_decode_params(plan, q, latent_cache, num_blocks, block_table,
                                              seq_lens, softmax_scale, out, lse, ws,
                                              device_status, 1, plan->num_heads, 0);
    return launch_decode_and_merge(p, plan, stream);
}
