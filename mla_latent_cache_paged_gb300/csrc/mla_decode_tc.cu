// Tensor-core decode kernel for sm_103a (MLA_KERNEL_TC): tcgen05 MMAs with
// TMEM accumulators, TMA page loads, and a two-CTA cluster per work item.
//
// What it computes is the absorbed ("forward_mqa") MLA decode of the vLLM
// mla_attention API docs, module docstring, "Data-Movement Friendly
// Approach": for one request and one split of its cached tokens, all heads
// attend to every token with K = the 576-wide latent entry and V = its first
// 512 columns. The design is this file's own:
//
// * Work item = (request, split), one 2-CTA cluster. The 576 feature dims are
//   divided between the pair: CTA 0 owns dims [0,256) + the RoPE dims
//   [512,576), CTA 1 owns [256,512). Each CTA TMA-loads only its own columns
//   of every 64-token page (SWIZZLE_128B boxes of 64 rows x 64 columns), so a
//   page crosses HBM once and the pair splits it 40 KB / 32 KB.
// * Scores: each CTA computes the partial S_c = Q[:, dims_c] K[:, dims_c]^T
//   for all (up to) 128 heads x 64 tokens with tcgen05.mma (M=128, N=64,
//   K=16 steps) into TMEM. q's 256 latent dims live in TMEM as the A operand;
//   CTA 0's 64 RoPE dims come from shared memory. The partial scores are
//   swapped through distributed shared memory and both CTAs form S = S_0+S_1
//   (bitwise the same in both, as fp32 addition commutes).
// * Softmax: 128 threads, one per head (= TMEM lane), keep the running max
//   and sum in fp32, base 2 with the scale folded in. The reference max only
//   moves when a tile raises it by more than 2^8, so the O rescale (a TMEM
//   read-modify-write) is rare; P is written to shared memory as bf16. O is
//   normalised by the sum of the rounded weights and the LSE uses the sum of
//   the unrounded ones.
// * O: each CTA accumulates its own half of the value columns,
//   O_c[128 x 256] += P[128 x 64] V_c[64 x 256], into TMEM (V = the same
//   page tile, read MN-major).
// * Pipelines: warp 0 issues TMA into a 4-stage ring, warp 1 issues MMAs
//   (QK of tile j+1 is in flight while the softmax of tile j runs), warps 2-5
//   run the softmax, the O correction and the epilogue.
// * Every wait is bounded: on expiry the kernel records MLA_ERR_TIMEOUT,
//   lets every role leave its loop, waits (bounded) for its TMA loads and
//   MMAs, frees TMEM and returns. A block id outside the pool is recorded
//   and loaded from a negative row, which TMA fills with zeros.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>

#include "mla_device.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace {

constexpr int kThreads = 192;               // 6 warps
constexpr int kStages = 4;
constexpr int kTile = 64;                   // tokens per tile = one page
constexpr int kBoxBytes = 64 * 128;         // 64 rows x 64 bf16 columns
constexpr int kStageBytes = 5 * kBoxBytes;  // CTA 0 loads 5 boxes, CTA 1 loads 4
constexpr int kOffQRope = 0;                // q RoPE dims, [128 x 64] bf16, SW128 K-major
constexpr int kOffP = 16384;                // P, [128 x 64] bf16, SW128 K-major
constexpr int kOffX = 32768;                // peer partial scores, [128 x 64] fp32
constexpr int kOffStages = 65536;
constexpr int kOffBar = kOffStages + kStages * kStageBytes;
constexpr int kSmemBytes = kOffBar + 256 + 1024;  // + slack to align the base to 1024

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;    // two 64-column score buffers
constexpr uint32_t kTmemQ = 128;  // 128 columns = 256 bf16 q dims (A operand)
constexpr uint32_t kTmemO = 256;  // 256 fp32 columns of O

constexpr uint64_t kTimeoutNs = 1000000000ull;  // 1 s per wait
constexpr float kLn2 = 0.693147180559945309f;
constexpr float kRescaleThreshold = 8.0f;       // log2 units

struct TcBars {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t s_full[2];
    uint64_t s_empty[2];
    uint64_t x_full;
    uint64_t x_empty;
    uint64_t p_full;
    uint64_t pv_done;
    uint64_t q_ready;
    uint64_t final_bar;
    uint32_t tmem_base;
    int32_t abort;
};
static_assert(sizeof(TcBars) <= 256, "barrier block too large");

enum WaitSite : int32_t {
    kSiteEmpty = 1, kSiteFull, kSiteSEmpty, kSiteSFull, kSiteXEmpty, kSiteXFull, kSitePFull,
    kSitePvDone, kSiteQReady, kSiteDrain
};

// Bounded wait on a local mbarrier phase. Returns false when the kernel is
// aborting (another role timed out) or when this wait expires.
__device__ __noinline__ bool wait_phase(uint32_t bar, uint32_t parity, TcBars* bars,
                                        int32_t* status, int32_t site, bool cluster_scope,
                                        bool ignore_abort = false) {
    for (int i = 0; i < 16; ++i) {
        if (cluster_scope ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity))
            return true;
    }
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
        for (int i = 0; i < 64; ++i) {
            if (cluster_scope ? ptx::mbar_try_wait_cluster(bar, parity)
                              : ptx::mbar_try_wait(bar, parity))
                return true;
        }
        if (!ignore_abort && *reinterpret_cast<volatile int32_t*>(&bars->abort) != 0) return false;
        if (ptx::globaltimer() - t0 > kTimeoutNs) {
            *reinterpret_cast<volatile int32_t*>(&bars->abort) = 1;
            record_error(status, MLA_ERR_TIMEOUT, site);
            return false;
        }
    }
}

__device__ __forceinline__ int box_column(uint32_t rank, int k) {
    return rank == 0 ? (k < 4 ? 64 * k : kLkv) : 256 + 64 * k;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __launch_bounds__(kThreads, 1)
mla_decode_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmap) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    TcBars* bars = reinterpret_cast<TcBars*>(smem + kOffBar);
    const uint32_t sbase = ptx::smem_addr(smem);
    const uint32_t stage_base = sbase + kOffStages;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const int S = p.num_splits;
    const int N = p.num_heads;
    const int item = blockIdx.x >> 1;
    const int b = item / S;
    const int split = item % S;

    const int L = checked_seq_len(p, b);
    int t_lo, t_hi;
    split_range(L, S, split, &t_lo, &t_hi);
    const int ntiles = (t_hi - t_lo + kTile - 1) / kTile;
    const int page0 = t_lo / kTile;

    const uint32_t b_full = ptx::smem_addr(&bars->full[0]);
    const uint32_t b_empty = ptx::smem_addr(&bars->empty[0]);
    const uint32_t b_sfull = ptx::smem_addr(&bars->s_full[0]);
    const uint32_t b_sempty = ptx::smem_addr(&bars->s_empty[0]);
    const uint32_t b_xfull = ptx::smem_addr(&bars->x_full);
    const uint32_t b_xempty = ptx::smem_addr(&bars->x_empty);
    const uint32_t b_pfull = ptx::smem_addr(&bars->p_full);
    const uint32_t b_pvdone = ptx::smem_addr(&bars->pv_done);
    const uint32_t b_qready = ptx::smem_addr(&bars->q_ready);
    const uint32_t b_final = ptx::smem_addr(&bars->final_bar);

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(b_full + 8 * s, 1);
            ptx::mbar_init(b_empty + 8 * s, 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(b_sfull + 8 * i, 1);
            ptx::mbar_init(b_sempty + 8 * i, 4);
        }
        ptx::mbar_init(b_xfull, 128);
        ptx::mbar_init(b_xempty, 128);
        ptx::mbar_init(b_pfull, 128);
        ptx::mbar_init(b_pvdone, 1);
        ptx::mbar_init(b_qready, 128);
        ptx::mbar_init(b_final, 1);
        bars->abort = 0;
        ptx::fence_mbarrier_init_cluster();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(&bars->tmem_base), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    ptx::cluster_sync();   // the peer's barriers exist before any remote arrive

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            const int nbox = rank == 0 ? 5 : 4;
            const uint32_t tx = uint32_t(nbox * kBoxBytes);
            const int32_t* table = p.block_table + size_t(b) * p.max_blocks;
            int next = ntiles > 0 ? table[page0] : 0;
            int issued = 0;
            for (int j = 0; j < ntiles; ++j) {
                const int blk = next;
                if (j + 1 < ntiles) next = table[page0 + j + 1];
                const int s = j % kStages;
                if (!wait_phase(b_empty + 8 * s, ((j / kStages) & 1) ^ 1, bars, p.status,
                                kSiteEmpty, false))
                    break;
                int32_t y;
                if (blk >= 0 && int64_t(blk) < p.num_blocks) {
                    y = blk * kTile;
                } else {
                    record_error(p.status, MLA_ERR_BAD_BLOCK_ID, blk);
                    y = -kTile;   // entirely outside the tensor: TMA writes zeros
                }
                ptx::mbar_arrive_expect_tx(b_full + 8 * s, tx);
                const uint32_t dst = stage_base + uint32_t(s * kStageBytes);
                for (int k = 0; k < nbox; ++k)
                    ptx::tma_load_2d(dst + uint32_t(k * kBoxBytes), &tmap, box_column(rank, k), y,
                                     b_full + 8 * s);
                issued = j + 1;
            }
            // Every issued load lands before the CTA may exit.
            for (int j = issued > kStages ? issued - kStages : 0; j < issued; ++j)
                wait_phase(b_full + 8 * (j % kStages), (j / kStages) & 1, bars, p.status,
                           kSiteDrain, false, true);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = ptx::idesc_bf16_f32(64, false);
            constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(256, true);
            const uint32_t qrope = sbase + kOffQRope;
            const uint32_t pbuf = sbase + kOffP;
            bool ok = wait_phase(b_qready, 0, bars, p.status, kSiteQReady, false);
            ptx::tc_fence_after();
            for (int j = 0; ok && j <= ntiles; ++j) {
                if (j < ntiles) {
                    const int s = j % kStages;
                    const int sb = j & 1;
                    if (!wait_phase(b_full + 8 * s, (j / kStages) & 1, bars, p.status, kSiteFull,
                                    false))
                        break;
                    if (!wait_phase(b_sempty + 8 * sb, ((j >> 1) & 1) ^ 1, bars, p.status,
                                    kSiteSEmpty, false))
                        break;
                    ptx::tc_fence_after();
                    const uint32_t st = stage_base + uint32_t(s * kStageBytes);
                    const uint32_t d = tmem + kTmemS + uint32_t(sb * 64);
#pragma unroll
                    for (int kb = 0; kb < 4; ++kb) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            ptx::mma_ts(d, tmem + kTmemQ + uint32_t(kb * 32 + kk * 8),
                                        ptx::desc_sw128(st + uint32_t(kb * kBoxBytes + kk * 32),
                                                        16, 1024),
                                        idesc_qk, (kb | kk) != 0 ? 1u : 0u);
                        }
                    }
                    if (rank == 0) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            ptx::mma_ss(d, ptx::desc_sw128(qrope + uint32_t(kk * 32), 16, 1024),
                                        ptx::desc_sw128(st + uint32_t(4 * kBoxBytes + kk * 32),
                                                        16, 1024),
                                        idesc_qk, 1u);
                        }
                    }
                    ptx::mma_commit(b_sfull + 8 * sb);
                }
                if (j >= 1) {
                    const int jj = j - 1;
                    if (!wait_phase(b_pfull, jj & 1, bars, p.status, kSitePFull, false)) break;
                    ptx::tc_fence_after();
                    const int s2 = jj % kStages;
                    const uint32_t st2 = stage_base + uint32_t(s2 * kStageBytes);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        ptx::mma_ss(tmem + kTmemO, ptx::desc_sw128(pbuf + uint32_t(kk * 32), 16, 1024),
                                    ptx::desc_sw128(st2 + uint32_t(kk * 16 * 128), 8192, 1024),
                                    idesc_pv, (jj > 0 || kk > 0) ? 1u : 0u);
                    }
                    ptx::mma_commit(b_pvdone);
                    ptx::mma_commit(b_empty + 8 * s2);
                }
            }
            // All MMAs of this CTA complete before TMEM is released.
            ptx::mma_commit(b_final);
            wait_phase(b_final, 0, bars, p.status, kSiteDrain, false, true);
        }
    } else {
        // ------------------------------------------- softmax / correction / epilogue
        const int quarter = warp & 3;
        const int h = quarter * 32 + lane;
        const uint32_t trow = tmem + (uint32_t(quarter * 32) << 16);
        const bool live_head = h < N;
        const size_t qrow = (size_t(b) * N + h) * kD;

        // q's latent dims of this CTA -> TMEM (A operand), RoPE dims -> smem.
        {
            const uint4* src = reinterpret_cast<const uint4*>(p.q + qrow + 256 * rank);
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = 0u;
                if (live_head) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint4 v = __ldg(src + c * 8 + i);
                        r[4 * i + 0] = v.x;
                        r[4 * i + 1] = v.y;
                        r[4 * i + 2] = v.z;
                        r[4 * i + 3] = v.w;
                    }
                }
                ptx::tmem_st32(trow + kTmemQ + uint32_t(c * 32), r);
            }
            if (rank == 0) {
                const uint4* rs = reinterpret_cast<const uint4*>(p.q + qrow + kLkv);
                unsigned char* row = smem + kOffQRope + h * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 v = make_uint4(0, 0, 0, 0);
                    if (live_head) v = __ldg(rs + c);
                    *reinterpret_cast<uint4*>(row + ((c ^ (h & 7)) * 16)) = v;
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(b_qready);
        }

        const uint32_t my_x = sbase + kOffX + uint32_t(h * 256);
        const uint32_t peer_x = ptx::mapa(my_x, peer);
        const uint32_t peer_xfull = ptx::mapa(b_xfull, peer);
        const uint32_t peer_xempty = ptx::mapa(b_xempty, peer);
        const float* my_x_ptr = reinterpret_cast<const float*>(smem + kOffX + h * 256);
        unsigned char* prow = smem + kOffP + h * 128;

        float m_ref = -INFINITY;
        float l_sum = 0.f;   // sum of fp32 weights (for the LSE)
        float l_bf = 0.f;    // sum of the bf16-rounded weights the MMA used (for O)
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            const int sb = j & 1;
            ok = wait_phase(b_sfull + 8 * sb, (j >> 1) & 1, bars, p.status, kSiteSFull, false);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            ptx::tc_fence_after();
            float s[64];
            {
                uint32_t r[32];
                ptx::tmem_ld32(trow + kTmemS + uint32_t(sb * 64), r);
#pragma unroll
                for (int i = 0; i < 32; ++i) s[i] = __uint_as_float(r[i]);
                ptx::tmem_ld32(trow + kTmemS + uint32_t(sb * 64 + 32), r);
#pragma unroll
                for (int i = 0; i < 32; ++i) s[32 + i] = __uint_as_float(r[i]);
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(b_sempty + 8 * sb);

            // Swap partial scores with the peer CTA.
            ok = wait_phase(b_xempty, (j & 1) ^ 1, bars, p.status, kSiteXEmpty, true);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
#pragma unroll
            for (int c = 0; c < 16; ++c)
                ptx::st_cluster_v4(peer_x + uint32_t((c ^ (h & 15)) * 16), s[4 * c], s[4 * c + 1],
                                   s[4 * c + 2], s[4 * c + 3]);
            ptx::mbar_arrive_remote(peer_xfull);
            ok = wait_phase(b_xfull, j & 1, bars, p.status, kSiteXFull, true);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const float4 v = *reinterpret_cast<const float4*>(my_x_ptr + 4 * (c ^ (h & 15)));
                s[4 * c] += v.x;
                s[4 * c + 1] += v.y;
                s[4 * c + 2] += v.z;
                s[4 * c + 3] += v.w;
            }
            ptx::mbar_arrive_remote(peer_xempty);

            // Online softmax in base 2 with a lazily moved reference max.
            const int valid = min(kTile, t_hi - (t_lo + j * kTile));
            float mx = -INFINITY;
#pragma unroll
            for (int t = 0; t < 64; ++t) {
                s[t] = t < valid ? s[t] * p.scale_log2 : -INFINITY;
                mx = fmaxf(mx, s[t]);
            }
            const float m_new = fmaxf(m_ref, mx);
            const bool rescale = m_new > m_ref + kRescaleThreshold;
            float alpha = 1.f;
            if (rescale) {
                alpha = ptx::ex2(m_ref - m_new);
                m_ref = m_new;
            }
            float rs = 0.f;
#pragma unroll
            for (int t = 0; t < 64; ++t) {
                s[t] = ptx::ex2(s[t] - m_ref);
                rs += s[t];
            }
            l_sum = l_sum * alpha + rs;
            // P goes to the MMA as bf16. O is normalised by the sum of those
            // rounded weights, so that it stays an exact weighted average of V
            // rows (a row that dominates the softmax comes out unchanged); the
            // LSE keeps the fp32 sum.
            uint32_t pk[32];
            float rs_bf = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                pk[i] = pack_bf16x2(s[2 * i], s[2 * i + 1]);
                rs_bf += __uint_as_float(pk[i] << 16) + __uint_as_float(pk[i] & 0xffff0000u);
            }
            l_bf = l_bf * alpha + rs_bf;

            if (j >= 1) {
                ok = wait_phase(b_pvdone, (j - 1) & 1, bars, p.status, kSitePvDone, false);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                ptx::tc_fence_after();
                if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
                    for (int c = 0; c < 256; c += 32) {
                        uint32_t o[32];
                        ptx::tmem_ld32(trow + kTmemO + uint32_t(c), o);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        ptx::tmem_st32(trow + kTmemO + uint32_t(c), o);
                    }
                }
            }
            // P row of this head: 64 tokens as bf16, 128-byte swizzled row.
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                *reinterpret_cast<uint4*>(prow + ((c ^ (h & 7)) * 16)) =
                    make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            }
            // Rows past the sequence end in the last page may hold anything
            // (even NaN): zero their value columns so that 0 * V stays 0.
            if (valid < kTile) {
                unsigned char* st = smem + kOffStages + (j % kStages) * kStageBytes;
                const int rows = kTile - valid;
                for (int idx = h; idx < rows * 32; idx += 128) {
                    const int r = valid + idx / 32;
                    const int box = (idx / 8) & 3;
                    const int ch = idx & 7;
                    *reinterpret_cast<uint4*>(st + box * kBoxBytes + r * 128 + ch * 16) =
                        make_uint4(0, 0, 0, 0);
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(b_pfull);
        }

        // Epilogue: O / l -> bf16 output, or the fp32 split partial.
        if (ok && ntiles > 0) {
            ok = wait_phase(b_pvdone, (ntiles - 1) & 1, bars, p.status, kSitePvDone, false);
            ok = __all_sync(0xffffffffu, ok);
            ptx::tc_fence_after();
        }
        if (ok) {
            const float inv = l_bf > 0.f ? 1.f / l_bf : 0.f;
            const float lse = l_sum > 0.f ? (m_ref + log2f(l_sum)) * kLn2 : -INFINITY;
            const size_t row = size_t(b) * N + h;
#pragma unroll 1
            for (int c = 0; c < 256; c += 32) {
                uint32_t o[32];
                if (ntiles > 0) {
                    ptx::tmem_ld32(trow + kTmemO + uint32_t(c), o);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                }
                const int col = 256 * int(rank) + c;
                if (!live_head) {
                    // padded head row: nothing to write
                } else if (S == 1) {
                    uint4* dst = reinterpret_cast<uint4*>(p.out + row * kLkv + col);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint4 v;
                        v.x = pack_bf16x2(__uint_as_float(o[8 * i + 0]) * inv,
                                          __uint_as_float(o[8 * i + 1]) * inv);
                        v.y = pack_bf16x2(__uint_as_float(o[8 * i + 2]) * inv,
                                          __uint_as_float(o[8 * i + 3]) * inv);
                        v.z = pack_bf16x2(__uint_as_float(o[8 * i + 4]) * inv,
                                          __uint_as_float(o[8 * i + 5]) * inv);
                        v.w = pack_bf16x2(__uint_as_float(o[8 * i + 6]) * inv,
                                          __uint_as_float(o[8 * i + 7]) * inv);
                        dst[i] = v;
                    }
                } else {
                    float4* dst = reinterpret_cast<float4*>(p.o_part + (row * S + split) * kLkv + col);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv,
                                             __uint_as_float(o[4 * i + 1]) * inv,
                                             __uint_as_float(o[4 * i + 2]) * inv,
                                             __uint_as_float(o[4 * i + 3]) * inv);
                }
            }
            if (rank == 0 && live_head) {
                if (S == 1) {
                    if (p.lse != nullptr) p.lse[row] = lse;
                } else {
                    p.lse_part[row * S + split] = lse;
                }
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem, kTmemCols);
    ptx::cluster_sync();   // no CTA leaves while its peer may still touch its smem
}

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
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

}  // namespace

bool tc_kernel_built() { return true; }

int tc_max_blocks() { return INT_MAX / kTile - 1; }

int launch_decode_tc(const DecodeParams& p, int grid_ctas, void* stream) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = get_encoder();
    if (encode == nullptr) return int(cudaErrorNotSupported);
    CUtensorMap tmap;
    const cuuint64_t dims[2] = {cuuint64_t(kD), cuuint64_t(p.num_blocks) * kTile};
    const cuuint64_t strides[1] = {cuuint64_t(kD) * 2};
    const cuuint32_t box[2] = {64, 64};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                        const_cast<uint16_t*>(p.cache), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return int(cudaErrorInvalidValue);
    cudaError_t e = cudaFuncSetAttribute(mla_decode_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return int(e);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid_ctas), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, mla_decode_tc_kernel, p, tmap);
    return int(e);
}

}  // namespace mla
