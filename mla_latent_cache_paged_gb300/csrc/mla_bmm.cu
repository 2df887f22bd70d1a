// Per-head batched matmuls on either side of the decode, on the tensor cores.
//
//   front end  (mla_q_absorb_concat_cache):
//       ql_nope[b, n, :] = q[b, n, 0:128] . W_UK_T[n]      W_UK_T bf16 [N, 128, 512]
//       mqa_q[b, n, :]   = [ql_nope[b, n, :] | q[b, n, 128:192]]
//       cache row `slot_mapping[b]` = [kv_c[b] | k_pe[b]]
//   up-projection (mla_v_up_proj):
//       out[b, n, :]     = x[b, n, :] . W_UV[n]            W_UV bf16 [N, 512, 128]
//   merge + up-projection (mla_merge_splits_v_up_proj):
//       x[b, n, :]       = LSE-weighted merge of the S split partials of (b, n),
//                          rounded to bf16 in shared memory (never written out
//                          unless asked), then the up-projection above
//
// vLLM mla_attention API docs, MLAAttention.forward_impl (torch.bmm of
// (N, B, P) by W_UK_T, then the q concat) and _v_up_proj (torch.bmm by W_UV);
// raon-1-mini MLA page, _decode_concat_cache (query concat fused with the
// latent cache insert) and the weight layouts it prepares (W_UK_T =
// W_UK.permute(1, 2, 0), W_UV transposed to (N, Lkv, V)).
//
// CTA (x, n) computes rows 128x..128x+127 (requests) of head n: M = 128
// batch rows, the whole J-wide result (512 or 128 fp32 columns) accumulated
// in TMEM, K streamed in 64-wide chunks. A (the activations) is K-major: a
// TMA box of 128 rows x 64 k at column n * head_stride + 64c of the [B, N *
// head_stride] view. The weight chunk is MN-major: J / 64 boxes of 64 k-rows
// x 64 columns of the [N * K, J] view. Both use the 128-byte swizzle.
// Warp 0 lane 0 loads (a ring of STAGES chunks), warp 1 lane 0 issues
// tcgen05.mma (M = 128, N = min(J, 256), K = 16), and all four warps read the
// accumulator back (thread = row), round to bf16, stage it in shared memory
// (the idle ring, 128-byte swizzled) and write it with TMA stores. In the
// front end the q_pe tile arrives by TMA after the A chunks and leaves by
// TMA store, and warps 2-3 insert the new tokens' latent rows (the CTAs of
// a batch tile share them out by head) while the MMAs run. Every wait is bounded (MLA_ERR_TIMEOUT);
// a slot outside the cache is recorded (MLA_ERR_BAD_BLOCK_ID), not written.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>

#include "mla_device.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace {

constexpr int kBmmThreads = 128;
constexpr int kMergeUpThreads = 256;         // + six warps that merge the A tile
constexpr int kMergeWarps = 6;
constexpr int kMaxFusedSplits = 512;         // merge weights: 6 warps x 512 fp32 in the q_pe area
// Kernel modes: the up-projection, the front end, the merge + up-projection.
constexpr int kModeUp = 0, kModeFront = 1, kModeMergeUp = 2;
constexpr int kM = 128;                      // batch rows per CTA
constexpr int kChunk = 64;                   // K per ring stage
constexpr int kABytes = kM * kChunk * 2;     // 16 KB
constexpr int kWBlockBytes = kChunk * 64 * 2;   // one 64 x 64 weight box: 8 KB
constexpr uint64_t kBmmTimeoutNs = 1000000000ull;
constexpr uint32_t kBmmSuspendNs = 20000;
constexpr int kNope = 128;                   // qk_nope_head_dim
constexpr int kQHead = kNope + kRope;        // q head width (P + R)

enum BmmSite : int32_t { kSiteRingEmpty = 30, kSiteRingFull, kSiteAccFull, kSiteRingDrain };

// Shared memory: the whole A tile (all K chunks, all requested up front so
// that each request's row is read in one burst, each chunk with its own
// barrier so that its MMAs start as soon as it lands), a ring of STAGES
// weight chunks, the front end's q_pe tile, then the barriers. The result is
// staged over the A tile and the ring once the MMAs are done.
template <int J, int KD, int STAGES>
struct BmmShape {
    static constexpr int kWBytes = (J / 64) * kWBlockBytes;   // one weight chunk
    static constexpr int kChunks = KD / kChunk;
    static constexpr int kAllABytes = kChunks * kABytes;
    static constexpr int kRingOff = kAllABytes;
    static constexpr int kPiece = J > 256 ? 256 : J;       // N of one MMA
    static constexpr int kPieces = J / kPiece;
    static constexpr int kTmemCols = J < 32 ? 32 : J;
    static constexpr int kPeOff = kRingOff + STAGES * kWBytes;   // front end: q_pe, 128 x 64
    static constexpr int kBarOff = kPeOff + kABytes;   // a_full, w_full[S], w_empty[S], acc, slot, abort
    static constexpr int kAChunkBarOff = kBarOff + 128;  // one "A chunk landed" barrier per chunk
    static constexpr int kSmemBytes = kBarOff + 256 + 1024;   // + alignment slack
    static_assert(KD % kChunk == 0 && J % 64 == 0 && J <= 512, "shape");
    static_assert((J & (J - 1)) == 0, "TMEM allocation is a power of two");
    static_assert(kSmemBytes <= 232448, "shared memory");
    static_assert(16 * STAGES + 24 <= 128 && 128 + 8 * kChunks <= 256, "barrier area");
    static_assert(kPeOff >= (J / 64) * kM * 128, "epilogue staging fits A and the ring");
};

struct BmmParams {
    int batch, heads;
    int a_head;                  // columns from one head's A to the next (192 or 512)
    const uint16_t* q;           // front end: q [B, N, 192] (for q_pe)
    const uint16_t* w;           // the weights [N, KD, J] (for the L2 prefetch)
    uint16_t* out;               // element (b, n, j) at out + b * out_row + n * out_head + j
    int64_t out_row;
    int out_head;
    const uint16_t* kv_c;        // front end: [B, 512]
    const uint16_t* k_pe;        // front end: [B, 64]
    const int64_t* slots;        // front end: [B] or null
    uint16_t* cache;             // front end: [num_blocks, 64, 576]
    int64_t num_blocks;
    int32_t* status;
    const void* o_part;          // merge + up-projection: [B, N, S, 512] fp32 or bf16
    bool part_bf16;
    const float* lse_part;       //                        fp32 [B, N, S]
    int splits;
    float* lse;                  //                        merged LSE [B, N] or null
    uint16_t* latent;            //                        merged rows bf16 [B, N, 512] or null
};

__device__ __forceinline__ bool bmm_wait(uint32_t bar, uint32_t parity, volatile int32_t* abort,
                                         int32_t* status, int32_t site, bool ignore_abort) {
    if (ptx::mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
        for (int i = 0; i < 4; ++i)
            if (ptx::mbar_try_wait_sleep(bar, parity, kBmmSuspendNs)) return true;
        if (!ignore_abort && *abort != 0) return false;
        if (ptx::globaltimer() - t0 > kBmmTimeoutNs) {
            *abort = 1;
            record_error(status, MLA_ERR_TIMEOUT, site);
            return false;
        }
    }
}

// Tiled TMA store of the box at (x, y) from shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_2d(const void* tmap, int32_t x, int32_t y, uint32_t src) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
            reinterpret_cast<uint64_t>(tmap)),
        "r"(x), "r"(y), "r"(src)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Merge + up-projection: the merger warps build the A tile (row r = request
// m0 + r of head n) from the split partials: per row the S log-sum-exps give
// the merged LSE and one weight per split (merge_attn_states, vLLM
// mla_attention API docs, "Chunked Prefill"; a -inf partial weighs 0), lane
// l sums columns 16l..16l+15 over the splits in split order, and the bf16
// result goes to A chunk l / 4 in the 128-byte swizzled K-major layout the
// MMAs read. Rows past the batch are left as they are (their products are
// never stored).
// Four partials' values for the 16 columns of one lane (fp32 or bf16 rows).
// A partial past S reads as zero.
__device__ __forceinline__ void load_group(const BmmParams& p, int64_t base, int s0, int S,
                                           float4 (&v)[4][4]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int s = s0 + q;
        const int64_t e0 = base + int64_t(s) * kLkv;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (s >= S) {
                v[q][k] = make_float4(0.f, 0.f, 0.f, 0.f);
            } else if (p.part_bf16) {
                const uint2 u = __ldg(reinterpret_cast<const uint2*>(
                    static_cast<const uint16_t*>(p.o_part) + e0 + 4 * k));
                v[q][k] = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                                      __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
            } else {
                v[q][k] = __ldg(reinterpret_cast<const float4*>(
                    static_cast<const float*>(p.o_part) + e0) + k);
            }
        }
    }
}

// acc += w * v over a group, a partial of weight 0 (a neutral split, whose
// row may hold anything) contributing nothing.
__device__ __forceinline__ void fma_group(const float* wts, int s0, int S, const float4 (&v)[4][4],
                                          float4 (&acc)[4]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float w = s0 + q < S ? wts[s0 + q] : 0.f;
        if (w == 0.f) continue;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            acc[k].x = fmaf(w, v[q][k].x, acc[k].x);
            acc[k].y = fmaf(w, v[q][k].y, acc[k].y);
            acc[k].z = fmaf(w, v[q][k].z, acc[k].z);
            acc[k].w = fmaf(w, v[q][k].w, acc[k].w);
        }
    }
}

__device__ void merge_rows_into_a(const BmmParams& p, unsigned char* smem, float* wts, int m0,
                                  int n, int mw, int lane) {
    const int S = p.splits;
    const int rows = min(kM, p.batch - m0);
    for (int r = mw; r < rows; r += kMergeWarps) {
        const int64_t row = int64_t(m0 + r) * p.heads + n;
        const int64_t base = row * S * kLkv + lane * 16;   // element index of split 0
        // The first partials' loads go out with the LSEs' (their addresses do
        // not depend on the weights), so a row costs one round trip to memory.
        float4 va[4][4], vb[4][4];
        load_group(p, base, 0, S, va);
        const float* ls = p.lse_part + row * S;
        float m = -INFINITY;
        for (int s = lane; s < S; s += 32) m = fmaxf(m, ls[s]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float total = -INFINITY;
        if (m != -INFINITY) {
            float z = 0.f;
            for (int s = lane; s < S; s += 32) z += expf(ls[s] - m);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
            total = m + logf(z);
            for (int s = lane; s < S; s += 32) wts[s] = expf(ls[s] - total);
        } else {
            for (int s = lane; s < S; s += 32) wts[s] = 0.f;
        }
        __syncwarp();
        if (lane == 0 && p.lse != nullptr) p.lse[row] = total;
        float4 acc[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        // The next group's loads go out before this group's sums.
        for (int s0 = 0; s0 < S; s0 += 8) {
            if (s0 + 4 < S) load_group(p, base, s0 + 4, S, vb);
            fma_group(wts, s0, S, va, acc);
            if (s0 + 4 >= S) break;
            if (s0 + 8 < S) load_group(p, base, s0 + 8, S, va);
            fma_group(wts, s0 + 4, S, vb, acc);
        }
        __syncwarp();
        uint32_t h[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            h[2 * k] = uint32_t(f32_to_bf16_bits_rn(acc[k].x)) |
                       (uint32_t(f32_to_bf16_bits_rn(acc[k].y)) << 16);
            h[2 * k + 1] = uint32_t(f32_to_bf16_bits_rn(acc[k].z)) |
                           (uint32_t(f32_to_bf16_bits_rn(acc[k].w)) << 16);
        }
        // columns 16 lane .. 16 lane + 15: chunk lane / 4, 16-byte pieces
        // 2 (lane % 4) and 2 (lane % 4) + 1 of the row
        unsigned char* arow = smem + (lane >> 2) * kABytes + r * 128;
        const int pc = 2 * (lane & 3);
        *reinterpret_cast<uint4*>(arow + ((pc ^ (r & 7)) * 16)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(arow + (((pc + 1) ^ (r & 7)) * 16)) =
            make_uint4(h[4], h[5], h[6], h[7]);
        if (p.latent != nullptr) {
            uint4* dst = reinterpret_cast<uint4*>(p.latent + row * kLkv + lane * 16);
            dst[0] = make_uint4(h[0], h[1], h[2], h[3]);
            dst[1] = make_uint4(h[4], h[5], h[6], h[7]);
        }
    }
}

template <int J, int KD, int STAGES, int kMode>
__global__ void __launch_bounds__(kMode == kModeMergeUp ? kMergeUpThreads : kBmmThreads, 1)
mla_bmm_kernel(const BmmParams p, const __grid_constant__ CUtensorMap tmap_a,
               const __grid_constant__ CUtensorMap tmap_w,
               const __grid_constant__ CUtensorMap tmap_o) {
    using Sh = BmmShape<J, KD, STAGES>;
    constexpr bool kFrontEnd = kMode == kModeFront;
    constexpr bool kMergeA = kMode == kModeMergeUp;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    const uint32_t sbase = raw + pad;
    unsigned char* smem = smem_raw + pad;
    const uint32_t b_afull = sbase + Sh::kBarOff;
    const uint32_t b_full = b_afull + 8;
    const uint32_t b_empty = b_full + 8 * STAGES;
    const uint32_t b_acc = b_empty + 8 * STAGES;
    const uint32_t b_achunk = sbase + Sh::kAChunkBarOff;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Sh::kBarOff + 16 * STAGES + 16);
    volatile int32_t* abort = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n = blockIdx.y;
    const int m0 = blockIdx.x * kM;

    // A programmatic dependent launch of the next kernel may start its setup
    // now; it waits for this grid before touching global memory, as this one
    // waits for its predecessor below.
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        ptx::mbar_init(b_afull, kMergeA ? kMergeWarps * 32 : 1);
        for (int c = 0; c < Sh::kChunks; ++c) ptx::mbar_init(b_achunk + 8 * c, 1);
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(b_full + 8 * s, 1);
            ptx::mbar_init(b_empty + 8 * s, 1);
        }
        ptx::mbar_init(b_acc, 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), Sh::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp == 0) {
        // Producer: A chunk c and weight chunk c side by side while the ring
        // has room, the rest of A (and q_pe), then weight chunk c into stage
        // c % STAGES once its previous use is done.
        int issued = 0;
        if (ptx::elect_one()) {
            auto load_a = [&](int c) {
                ptx::mbar_arrive_expect_tx(b_achunk + 8 * c, kABytes);
                ptx::tma_load_2d(sbase + uint32_t(c * kABytes), &tmap_a,
                                 n * p.a_head + c * kChunk, m0, b_achunk + 8 * c);
            };
            auto load_w = [&](int c) {
                const int s = c % STAGES;
                const uint32_t st = sbase + uint32_t(Sh::kRingOff + s * Sh::kWBytes);
                ptx::mbar_arrive_expect_tx(b_full + 8 * s, Sh::kWBytes);
#pragma unroll
                for (int jb = 0; jb < J / 64; ++jb)
                    ptx::tma_load_2d(st + uint32_t(jb * kWBlockBytes), &tmap_w, jb * 64,
                                     n * KD + c * kChunk, b_full + 8 * s);
            };
            constexpr int kFirst = Sh::kChunks < STAGES ? Sh::kChunks : STAGES;
            for (int c = 0; c < kFirst; ++c) {
                if constexpr (!kMergeA) load_a(c);
                load_w(c);
            }
            issued = kFirst;
            // The weight chunks that wait for a free ring stage are pulled
            // into L2 now, so that their loads are L2 round trips (not in the
            // merge mode, whose A tile is built from partials meanwhile:
            // measured slower there).
            if constexpr (!kMergeA)
                for (int c = kFirst; c < Sh::kChunks; ++c)
                    ptx::prefetch_l2(p.w + (size_t(n) * KD + size_t(c) * kChunk) * J,
                                     uint32_t(kChunk * J * 2));
            if constexpr (!kMergeA)
                for (int c = kFirst; c < Sh::kChunks; ++c) load_a(c);
            if constexpr (kFrontEnd) {   // q_pe: columns 128..191 of the head, next to q_nope
                ptx::mbar_arrive_expect_tx(b_afull, kABytes);
                ptx::tma_load_2d(sbase + Sh::kPeOff, &tmap_a, n * p.a_head + kNope, m0, b_afull);
            }
            for (int c = kFirst; c < Sh::kChunks; ++c) {
                const int s = c % STAGES;
                if (!bmm_wait(b_empty + 8 * s, ((c / STAGES) - 1) & 1, abort, p.status,
                              kSiteRingEmpty, false))
                    break;
                load_w(c);
                ++issued;
            }
            // Copies still in flight (after an abort) land before the CTA exits.
            if constexpr (!kMergeA)
                for (int c = 0; c < Sh::kChunks; ++c)
                    bmm_wait(b_achunk + 8 * c, 0, abort, p.status, kSiteRingDrain, true);
            if constexpr (kFrontEnd) bmm_wait(b_afull, 0, abort, p.status, kSiteRingDrain, true);
            for (int c = issued - STAGES < 0 ? 0 : issued - STAGES; c < issued; ++c)
                bmm_wait(b_full + 8 * (c % STAGES), (c / STAGES) & 1, abort, p.status,
                         kSiteRingDrain, true);
        }
        __syncwarp();
    } else if (warp == 1) {
        // MMA issuer.
        constexpr uint32_t idesc = ptx::idesc_bf16_f32(Sh::kPiece, true);
        if (ptx::elect_one()) {
            bool ok = !kMergeA || bmm_wait(b_afull, 0, abort, p.status, kSiteRingFull, false);
            for (int c = 0; c < Sh::kChunks && ok; ++c) {
                const int s = c % STAGES;
                if constexpr (!kMergeA)
                    if (!bmm_wait(b_achunk + 8 * c, 0, abort, p.status, kSiteRingFull, false)) break;
                ok = bmm_wait(b_full + 8 * s, (c / STAGES) & 1, abort, p.status, kSiteRingFull,
                              false);
                if (!ok) break;
                ptx::tc_fence_after();
                const uint32_t a_st = sbase + uint32_t(c * kABytes);
                const uint32_t w_st = sbase + uint32_t(Sh::kRingOff + s * Sh::kWBytes);
                // A: K-major, 16 k = 32 bytes per step; W: MN-major, 16 k-rows
                // = 2 KB per step, 64-column blocks 8 KB apart.
                const uint64_t a0 = ptx::desc_sw128(a_st, 16, 1024);
                const uint64_t a1 = ptx::desc_sw128(a_st + 32, 16, 1024);
                const uint64_t a2 = ptx::desc_sw128(a_st + 64, 16, 1024);
                const uint64_t a3 = ptx::desc_sw128(a_st + 96, 16, 1024);
#pragma unroll
                for (int pc = 0; pc < Sh::kPieces; ++pc) {
                    const uint32_t wp = w_st + uint32_t(pc * (Sh::kPiece / 64) * kWBlockBytes);
                    ptx::mma4_ss(tmem + uint32_t(pc * Sh::kPiece), a0, a1, a2, a3,
                                 ptx::desc_sw128(wp, kWBlockBytes, 1024),
                                 ptx::desc_sw128(wp + 2048, kWBlockBytes, 1024),
                                 ptx::desc_sw128(wp + 4096, kWBlockBytes, 1024),
                                 ptx::desc_sw128(wp + 6144, kWBlockBytes, 1024), idesc,
                                 c > 0 ? 1u : 0u);
                }
                ptx::mma_commit(b_empty + 8 * s);
            }
            // Arrives when every MMA issued above has completed (also after an
            // abort, so the accumulator is idle before TMEM is freed).
            ptx::mma_commit(b_acc);
        }
        __syncwarp();
    } else if (kMergeA) {
        // warps 2-7: the A tile from the split partials, then A is full
        float* wts = reinterpret_cast<float*>(smem + Sh::kPeOff) + (warp - 2) * kMaxFusedSplits;
        merge_rows_into_a(p, smem, wts, m0, n, warp - 2, lane);
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(b_afull);
    } else if (kFrontEnd) {
        const int t = threadIdx.x - 64;   // warps 2-3
        // q_pe: its tile (on the a_full barrier) goes out as four 32-row boxes
        // to columns 512..575 of the head.
        if (t == 0 && bmm_wait(b_afull, 0, abort, p.status, kSiteRingFull, false)) {
            for (int slab = 0; slab < kM / 32 && m0 + 32 * slab < p.batch; ++slab)
                tma_store_2d(&tmap_o, n * p.out_head + J, m0 + 32 * slab,
                             sbase + uint32_t(Sh::kPeOff + slab * 4096));
            bulk_commit();
        }
        // Cache insert: rows n, n + N, ... of this tile, 72 16-byte pieces each,
        // four loads in flight per thread before their stores.
        if (p.slots != nullptr) {
            constexpr int kPieces = kD / 8;
            const int rows = (kM - 1 - n) / p.heads + 1;
            const int total = rows * kPieces;
            const int64_t limit = p.num_blocks * kPageSize;
            for (int i0 = t; i0 < total; i0 += 4 * 64) {
                uint4 v[4];
                uint16_t* dst[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    dst[k] = nullptr;
                    const int i = i0 + 64 * k;
                    if (i >= total) continue;
                    const int b = m0 + n + (i / kPieces) * p.heads;
                    const int piece = i % kPieces;
                    if (b >= p.batch) continue;
                    const int64_t slot = p.slots[b];
                    if (slot < 0) continue;
                    if (slot >= limit) {
                        if (piece == 0)
                            record_error(p.status, MLA_ERR_BAD_BLOCK_ID, int32_t(slot / kPageSize));
                        continue;
                    }
                    const uint16_t* src = piece < kLkv / 8
                                              ? p.kv_c + int64_t(b) * kLkv + 8 * piece
                                              : p.k_pe + int64_t(b) * kRope + 8 * (piece - kLkv / 8);
                    v[k] = __ldg(reinterpret_cast<const uint4*>(src));
                    dst[k] = p.cache + slot * kD + 8 * piece;
                }
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (dst[k] != nullptr) *reinterpret_cast<uint4*>(dst[k]) = v[k];
            }
        }
    }

    // Epilogue: thread = row of the tile = TMEM lane. Each warp stages its 32
    // rows, 64 columns at a time, in the (now idle) ring in the 128-byte
    // swizzled layout of the output tensor map and stores them by TMA; rows
    // past the batch fall outside the map and are not written.
    bool acc_ok = warp < 4;   // the four warps of the accumulator's lanes
    if (acc_ok && lane == 0)
        acc_ok = bmm_wait(b_acc, 0, abort, p.status, kSiteAccFull, true);
    acc_ok = __shfl_sync(0xffffffffu, acc_ok ? 1 : 0, 0) != 0 && *abort == 0;
    ptx::tc_fence_after();
    if (acc_ok) {
        const uint32_t stage_w = sbase + uint32_t(warp * (J / 64) * 4096);
#pragma unroll 1
        for (int cb = 0; cb < J / 64; ++cb) {
            uint32_t r0[32], r1[32];
            const uint32_t taddr = tmem + (uint32_t(warp * 32) << 16) + uint32_t(cb * 64);
            ptx::tmem_ld32(taddr, r0);
            ptx::tmem_ld32(taddr + 32, r1);
            const uint32_t row = stage_w + uint32_t(cb * 4096 + lane * 128);
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                const uint32_t* r = ch < 4 ? r0 : r1;
                const int o = (ch & 3) * 8;
                uint32_t w[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    w[i] = uint32_t(f32_to_bf16_bits_rn(__uint_as_float(r[o + 2 * i]))) |
                           (uint32_t(f32_to_bf16_bits_rn(__uint_as_float(r[o + 2 * i + 1]))) << 16);
                const uint32_t addr = row + uint32_t(((ch ^ (lane & 7)) * 16));
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]),
                             "r"(w[1]), "r"(w[2]), "r"(w[3])
                             : "memory");
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && m0 + warp * 32 < p.batch)
                tma_store_2d(&tmap_o, n * p.out_head + cb * 64, m0 + warp * 32,
                             stage_w + uint32_t(cb * 4096));
        }
        if (lane == 0) bulk_commit();
    }
    if (lane == 0) bulk_wait_all();   // stores issued by this thread have completed
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem, Sh::kTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 bmm_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// Row-major bf16 [rows, cols] view, boxes of box_rows x 64 columns, 128-byte swizzle.
bool encode_2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = bmm_encoder();
    if (encode == nullptr) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int J, int KD, int STAGES, int kMode>
int launch_bmm(const BmmParams& p, const void* a, const void* w, cudaStream_t st) {
    using Sh = BmmShape<J, KD, STAGES>;
    CUtensorMap ta, tw, to;
    // (merge + up-projection: A is built in shared memory; the map over the
    // output stands in for the unused A map)
    if (!encode_2d(&ta, kMode == kModeMergeUp ? static_cast<const void*>(p.out) : a,
                   uint64_t(p.heads) * (kMode == kModeMergeUp ? p.out_head : p.a_head),
                   uint64_t(p.batch), kMode == kModeMergeUp ? 32 : kM) ||
        !encode_2d(&tw, w, J, uint64_t(p.heads) * KD, kChunk) ||
        !encode_2d(&to, p.out, uint64_t(p.heads) * p.out_head, uint64_t(p.batch), 32))
        return int(cudaErrorInvalidValue);
    BmmParams pw = p;
    pw.w = static_cast<const uint16_t*>(w);
    auto kernel = mla_bmm_kernel<J, KD, STAGES, kMode>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Sh::kSmemBytes);
    if (e != cudaSuccess) return int(e);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned((p.batch + kM - 1) / kM), unsigned(p.heads));
    cfg.blockDim = dim3(kMode == kModeMergeUp ? kMergeUpThreads : kBmmThreads, 1, 1);
    cfg.dynamicSmemBytes = Sh::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return int(cudaLaunchKernelEx(&cfg, kernel, pw, ta, tw, to));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int status_of(int e) { return e == 0 ? MLA_OK : MLA_ERR_CUDA; }

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" int mla_q_absorb_concat_cache(const void* q, const void* w_uk_t, const void* kv_c,
                                         const void* k_pe, const int64_t* slot_mapping,
                                         void* latent_cache, int64_t num_blocks, int batch,
                                         int num_heads, void* mqa_q, void* workspace,
                                         size_t workspace_bytes, void* stream) {
    if (batch < 0 || num_heads < 0 || num_heads > kMaxHeads || num_blocks < 0)
        return MLA_ERR_INVALID_ARG;
    if (batch == 0 || num_heads == 0) return MLA_OK;
    if (!q || !w_uk_t || !mqa_q) return MLA_ERR_INVALID_ARG;
    if (slot_mapping && (!kv_c || !k_pe || !latent_cache)) return MLA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < kStatusBytes ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return MLA_ERR_WORKSPACE;
    if (!aligned16(q) || !aligned16(w_uk_t) || !aligned16(mqa_q) ||
        (slot_mapping && (!aligned16(kv_c) || !aligned16(k_pe) || !aligned16(latent_cache) ||
                          (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0)))
        return MLA_ERR_INVALID_ARG;
    BmmParams p{};
    p.batch = batch;
    p.heads = num_heads;
    p.a_head = kQHead;
    p.q = static_cast<const uint16_t*>(q);
    p.out = static_cast<uint16_t*>(mqa_q);
    p.out_row = int64_t(num_heads) * kD;
    p.out_head = kD;
    p.kv_c = static_cast<const uint16_t*>(kv_c);
    p.k_pe = static_cast<const uint16_t*>(k_pe);
    p.slots = slot_mapping;
    p.cache = static_cast<uint16_t*>(latent_cache);
    p.num_blocks = num_blocks;
    p.status = static_cast<int32_t*>(workspace);
    return status_of(launch_bmm<kLkv, kNope, 2, kModeFront>(p, q, w_uk_t,
                                                      static_cast<cudaStream_t>(stream)));
}

extern "C" int mla_v_up_proj(const void* x, const void* w_uv, int batch, int num_heads, void* out,
                             void* workspace, size_t workspace_bytes, void* stream) {
    if (batch < 0 || num_heads < 0 || num_heads > kMaxHeads) return MLA_ERR_INVALID_ARG;
    if (batch == 0 || num_heads == 0) return MLA_OK;
    if (!x || !w_uv || !out) return MLA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < kStatusBytes ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return MLA_ERR_WORKSPACE;
    if (!aligned16(x) || !aligned16(w_uv) || !aligned16(out)) return MLA_ERR_INVALID_ARG;
    BmmParams p{};
    p.batch = batch;
    p.heads = num_heads;
    p.a_head = kLkv;
    p.out = static_cast<uint16_t*>(out);
    p.out_row = int64_t(num_heads) * kNope;
    p.out_head = kNope;
    p.status = static_cast<int32_t*>(workspace);
    return status_of(launch_bmm<kNope, kLkv, 4, kModeUp>(p, x, w_uv,
                                                         static_cast<cudaStream_t>(stream)));
}

namespace mla {

int launch_merge_up_proj(const void* o_part, bool part_bf16, const float* lse_part, int batch,
                         int num_heads, int num_splits, const void* w_uv, uint16_t* out,
                         float* lse, uint16_t* latent, int32_t* status, void* stream) {
    BmmParams p{};
    p.batch = batch;
    p.heads = num_heads;
    p.a_head = kLkv;
    p.out = out;
    p.out_row = int64_t(num_heads) * kNope;
    p.out_head = kNope;
    p.status = status;
    p.o_part = o_part;
    p.part_bf16 = part_bf16;
    p.lse_part = lse_part;
    p.splits = num_splits;
    p.lse = lse;
    p.latent = latent;
    return launch_bmm<kNope, kLkv, 4, kModeMergeUp>(p, nullptr, w_uv,
                                                    static_cast<cudaStream_t>(stream));
}

}  // namespace mla

extern "C" int mla_merge_splits_v_up_proj(const float* o_part, const float* lse_part, int batch,
                                          int num_heads, int num_splits, const void* w_uv,
                                          void* out, float* lse, void* latent_out,
                                          void* workspace, size_t workspace_bytes,
                                          void* stream) {
    if (batch < 0 || num_heads < 0 || num_heads > kMaxHeads || num_splits < 1)
        return MLA_ERR_INVALID_ARG;
    if (num_splits > kMaxFusedSplits) return MLA_ERR_UNSUPPORTED;
    if (batch == 0 || num_heads == 0) return MLA_OK;
    if (!o_part || !lse_part || !w_uv || !out) return MLA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < kStatusBytes ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return MLA_ERR_WORKSPACE;
    if (!aligned16(o_part) || (reinterpret_cast<uintptr_t>(lse_part) & 3u) != 0 ||
        !aligned16(w_uv) || !aligned16(out) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) ||
        (latent_out && !aligned16(latent_out)))
        return MLA_ERR_INVALID_ARG;
    return status_of(launch_merge_up_proj(o_part, false, lse_part, batch, num_heads, num_splits,
                                          w_uv,
                                          static_cast<uint16_t*>(out), lse,
                                          static_cast<uint16_t*>(latent_out),
                                          static_cast<int32_t*>(workspace), stream));
}
