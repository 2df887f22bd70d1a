// Tensor-core decode kernel for sm_103a (MLA_KERNEL_TC): tcgen05 MMAs with
// TMEM accumulators, TMA page loads, and a two-CTA cluster per work item.
//
// What it computes is the absorbed ("forward_mqa") MLA decode of the vLLM
// mla_attention API docs, module docstring, "Data-Movement Friendly
// Approach": for one request and one split of its cached tokens, every head
// attends to every token with K = the 576-wide latent entry and V = its first
// 512 columns. The design is this file's own.
//
// Work item = (request, split) = one 2-CTA cluster; a tile is one 64-token
// page. CTA c (c = 0, 1) owns
//   * the scores of rows [32c, 32c+32) of every page: S_c = Q K_c^T for all
//     (up to) 128 heads, with the full 576-wide q resident (448 dims in TMEM
//     as the A operand, 128 dims in shared memory), tcgen05.mma M=128, N=32;
//   * the value columns [256c, 256c+256) of O: O_c[128 x 256] in TMEM,
//     accumulated from the bf16 weights of all 64 tokens of the page.
// So each page crosses HBM once: a CTA TMA-loads its 32 rows; the part of
// them that the other CTA needs as V (the other half of the value columns)
// is loaded once with cluster multicast into both CTAs.
//
// Softmax. 128 threads, one per head (= TMEM lane), keep the running
// reference max m (base 2, integer valued, with the scale folded in) and the
// sums in fp32. For each tile a CTA picks its own integer base: the current m,
// or ceil(tile max) when the tile max exceeds m by more than 8, so weights
// never exceed 2^8. It writes its 32 bf16 weights per head and its base and
// row sums, and pushes them to the other CTA with one bulk shared-memory copy
// (8 KB + 1.5 KB). Both CTAs then agree on the new m = the larger base,
// scale whichever half used the smaller base by an exact power of two, and
// rescale O by 2^(m_old - m_new) when m moved (rare; a TMEM read-modify-
// write). O is normalised by the sum of the rounded weights the MMA used and
// the LSE keeps the fp32 sum; both CTAs add the two halves in rank order, so
// their statistics agree bit for bit.
//
// Pipelines: warp 0 issues TMA into a 3-stage ring (each stage released by
// multicast tcgen05.commit from both CTAs), warp 1 issues MMAs whenever their
// inputs are ready (the score MMA of tile j+1 runs while the softmax of tile
// j waits for the other half), warps 2-5 run the softmax, the O correction
// and the epilogue. Weights are double-buffered so a tile's exchange overlaps
// the previous tile's P.V MMA.
//
// Every wait is bounded: on expiry the kernel records MLA_ERR_TIMEOUT, lets
// each role leave its loop, waits (bounded) for its own copies and MMAs,
// frees TMEM and returns. A block id outside the pool is recorded and loaded
// from negative rows, which TMA fills with zeros.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>

#include "mla_device.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace {

constexpr int kThreads = 192;                  // 6 warps
constexpr int kStages = 3;
constexpr int kTile = 64;                      // tokens per tile = one page
constexpr int kHalf = 32;                      // tokens per CTA per page
constexpr int kBoxBytes = kHalf * 128;         // 32 rows x 64 bf16 columns
constexpr int kStageBoxes = 13;
constexpr int kStageBytes = kStageBoxes * kBoxBytes;   // 53,248
// Stage layout (box index): [0,4) rows of CTA 0 x columns 256..511 (multicast),
// [4,8) rows of CTA 1 x columns 0..255 (multicast), [8,12) this CTA's rows x
// its own value columns, 12 this CTA's rows x RoPE columns 512..575.
constexpr int kBoxMc0 = 0;
constexpr int kBoxMc1 = 4;
constexpr int kBoxOwn = 8;
constexpr int kBoxRope = 12;

constexpr int kOffQS = 0;              // q dims 448..575: 2 x [128 x 64] bf16, SW128 K-major
constexpr int kOffP = 32768;           // P[buf 2][half 2] = [128 x 32] bf16, SW64 K-major
constexpr int kPHalfBytes = 8192;
constexpr int kOffSmall = 65536;       // small[buf 2][rank 2] = {base, rs, rs_bf}[128] fp32
constexpr int kSmallBytes = 3 * 128 * 4;
constexpr int kOffStages = kOffSmall + 4 * kSmallBytes;          // 71,680
constexpr int kOffBar = kOffStages + kStages * kStageBytes;      // 231,424
constexpr int kSmemBytes = kOffBar + 256;                        // dynamic smem base is 1 KB aligned
static_assert(kOffStages % 1024 == 0, "stage ring must be 1 KB aligned");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemQ = 0;     // 224 columns: q dims 0..447 as bf16 pairs (A operand)
constexpr uint32_t kTmemS = 224;   // 32 columns: scores of this CTA's 32 tokens
constexpr uint32_t kTmemO = 256;   // 256 fp32 columns of O
constexpr int kQTmemBlocks = 7;    // 64-dim blocks of q held in TMEM

constexpr uint64_t kTimeoutNs = 1000000000ull;   // 1 s per wait
constexpr float kLn2 = 0.693147180559945309f;
constexpr float kRescaleThreshold = 8.0f;         // log2 units
constexpr uint16_t kBothCtas = 0x3;

struct TcBars {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t s_full;
    uint64_t s_empty;
    uint64_t p_full[2];
    uint64_t p_free[2];
    uint64_t p_recv[2];
    uint64_t pv_done;
    uint64_t q_ready;
    uint64_t sm_sync;     // rendezvous of the 128 softmax threads
    uint64_t final_bar;
    uint32_t tmem_base;
    int32_t abort;
};
static_assert(sizeof(TcBars) <= 256, "barrier block too large");

enum WaitSite : int32_t {
    kSiteEmpty = 1, kSiteFull, kSiteSEmpty, kSiteSFull, kSitePFree, kSitePRecv, kSitePFull,
    kSitePvDone, kSiteQReady, kSiteDrain, kSiteMma, kSiteSmSync
};

__device__ __forceinline__ bool aborting(TcBars* bars) {
    return *reinterpret_cast<volatile int32_t*>(&bars->abort) != 0;
}

__device__ __forceinline__ void set_abort(TcBars* bars, int32_t* status, int32_t site) {
    *reinterpret_cast<volatile int32_t*>(&bars->abort) = 1;
    record_error(status, MLA_ERR_TIMEOUT, site);
}

// Bounded wait on a local mbarrier phase. Returns false when the kernel is
// aborting (another role timed out) or when this wait expires.
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, TcBars* bars,
                                       int32_t* status, int32_t site, bool ignore_abort) {
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (ptx::mbar_try_wait(bar, parity)) return true;
        if (!ignore_abort && aborting(bars)) return false;
        if (ptx::globaltimer() - t0 > kTimeoutNs) {
            set_abort(bars, status, site);
            return false;
        }
    }
}

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, TcBars* bars,
                                           int32_t* status, int32_t site,
                                           bool ignore_abort = false) {
    if (ptx::mbar_test_wait(bar, parity)) return true;
    return wait_slow(bar, parity, bars, status, site, ignore_abort);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Multiply the 32 bf16 values of one 64-byte P row by an exact power of two.
__device__ __forceinline__ void scale_p_row(unsigned char* row, float f) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint4* q = reinterpret_cast<uint4*>(row + 16 * c);
        uint4 v = *q;
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            w[i] = pack_bf16x2(__uint_as_float(w[i] << 16) * f,
                               __uint_as_float(w[i] & 0xffff0000u) * f);
        *q = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Box of this CTA's stage that holds K-block kb (dims 64kb..64kb+63) of its rows.
__device__ __forceinline__ int qk_box(uint32_t rank, int kb) {
    if (kb == 8) return kBoxRope;
    if (rank == 0) return kb < 4 ? kBoxOwn + kb : kBoxMc0 + (kb - 4);
    return kb < 4 ? kBoxMc1 + kb : kBoxOwn + (kb - 4);
}

// First box of the [32 tokens x 256 value columns] region, in this CTA's
// stage, of the rows of CTA r.
__device__ __forceinline__ int pv_box(uint32_t rank, int r) {
    if (rank == 0) return r == 0 ? kBoxOwn : kBoxMc1;
    return r == 0 ? kBoxMc0 : kBoxOwn;
}

__global__ void __launch_bounds__(kThreads, 1)
mla_decode_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmap) {
    extern __shared__ __align__(1024) unsigned char smem[];
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

    // Swizzled TMA boxes and UMMA descriptors assume a 1 KB aligned base.
    const bool aligned_ok = (sbase & 1023u) == 0u;
    const int L = checked_seq_len(p, b);
    int t_lo, t_hi;
    split_range(L, S, split, &t_lo, &t_hi);
    const int ntiles = aligned_ok ? (t_hi - t_lo + kTile - 1) / kTile : 0;
    const int page0 = t_lo / kTile;

    const uint32_t b_full = ptx::smem_addr(&bars->full[0]);
    const uint32_t b_empty = ptx::smem_addr(&bars->empty[0]);
    const uint32_t b_sfull = ptx::smem_addr(&bars->s_full);
    const uint32_t b_sempty = ptx::smem_addr(&bars->s_empty);
    const uint32_t b_pfull = ptx::smem_addr(&bars->p_full[0]);
    const uint32_t b_pfree = ptx::smem_addr(&bars->p_free[0]);
    const uint32_t b_precv = ptx::smem_addr(&bars->p_recv[0]);
    const uint32_t b_pvdone = ptx::smem_addr(&bars->pv_done);
    const uint32_t b_qready = ptx::smem_addr(&bars->q_ready);
    const uint32_t b_final = ptx::smem_addr(&bars->final_bar);
    const uint32_t b_smsync = ptx::smem_addr(&bars->sm_sync);

    if (tid == 0) {
        if (!aligned_ok) record_error(p.status, MLA_ERR_UNSUPPORTED, int32_t(sbase & 1023u));
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(b_full + 8 * s, 1);
            ptx::mbar_init(b_empty + 8 * s, 2);     // P.V of this stage done in both CTAs
        }
        ptx::mbar_init(b_sfull, 1);
        ptx::mbar_init(b_sempty, 4);
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(b_pfull + 8 * i, 128);
            ptx::mbar_init(b_pfree + 8 * i, 2);     // P.V of this buffer done in both CTAs
            ptx::mbar_init(b_precv + 8 * i, 1);
        }
        ptx::mbar_init(b_pvdone, 1);
        ptx::mbar_init(b_qready, 128);
        ptx::mbar_init(b_smsync, 128);
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
    ptx::cluster_sync();   // the peer's barriers exist before any remote arrive or copy

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            const int32_t* table = p.block_table + size_t(b) * p.max_blocks;
            int next = ntiles > 0 ? table[page0] : 0;
            int issued = 0;
            for (int j = 0; j < ntiles; ++j) {
                const int blk = next;
                if (j + 1 < ntiles) next = table[page0 + j + 1];
                const int s = j % kStages;
                if (!wait_phase(b_empty + 8 * s, ((j / kStages) & 1) ^ 1, bars, p.status,
                                kSiteEmpty))
                    break;
                int32_t y;
                if (blk >= 0 && int64_t(blk) < p.num_blocks) {
                    y = blk * kTile + kHalf * int(rank);
                } else {
                    record_error(p.status, MLA_ERR_BAD_BLOCK_ID, blk);
                    y = -kTile + kHalf * int(rank);   // wholly outside: TMA writes zeros
                }
                const uint32_t bar = b_full + 8 * s;
                const uint32_t st = stage_base + uint32_t(s * kStageBytes);
                ptx::mbar_arrive_expect_tx(bar, uint32_t(kStageBytes));
                // These rows x the value columns the other CTA accumulates: both CTAs.
                const int mc_box = rank == 0 ? kBoxMc0 : kBoxMc1;
                const int mc_col = rank == 0 ? 256 : 0;
                for (int k = 0; k < 4; ++k)
                    ptx::tma_load_2d_mc(st + uint32_t((mc_box + k) * kBoxBytes), &tmap,
                                        mc_col + 64 * k, y, bar, kBothCtas);
                // These rows x this CTA's own value columns, then the RoPE columns.
                const int own_col = rank == 0 ? 0 : 256;
                for (int k = 0; k < 4; ++k)
                    ptx::tma_load_2d(st + uint32_t((kBoxOwn + k) * kBoxBytes), &tmap,
                                     own_col + 64 * k, y, bar);
                ptx::tma_load_2d(st + uint32_t(kBoxRope * kBoxBytes), &tmap, kLkv, y, bar);
                issued = j + 1;
            }
            for (int j = issued > kStages ? issued - kStages : 0; j < issued; ++j)
                wait_phase(b_full + 8 * (j % kStages), (j / kStages) & 1, bars, p.status,
                           kSiteDrain, true);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = ptx::idesc_bf16_f32(kHalf, false);
            constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(256, true);
            const uint32_t qs = sbase + kOffQS;
            const uint32_t pbase = sbase + kOffP;
            bool ok = wait_phase(b_qready, 0, bars, p.status, kSiteQReady);
            ptx::tc_fence_after();
            int nq = 0;   // next score MMA
            int np = 0;   // next P.V MMA
            uint64_t idle_since = 0;
            uint32_t idle = 0;
            while (ok && np < ntiles) {
                bool did = false;
                if (nq < ntiles && ptx::mbar_test_wait(b_full + 8 * (nq % kStages),
                                                       (nq / kStages) & 1) &&
                    (nq == 0 || ptx::mbar_test_wait(b_sempty, (nq - 1) & 1))) {
                    ptx::tc_fence_after();
                    const uint32_t st = stage_base + uint32_t((nq % kStages) * kStageBytes);
                    const uint32_t d = tmem + kTmemS;
#pragma unroll
                    for (int kb = 0; kb < 9; ++kb) {
                        const uint32_t bb = st + uint32_t(qk_box(rank, kb) * kBoxBytes);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t bdesc = ptx::desc_sw128(bb + uint32_t(kk * 32), 16, 1024);
                            const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
                            if (kb < kQTmemBlocks)
                                ptx::mma_ts(d, tmem + kTmemQ + uint32_t(kb * 32 + kk * 8), bdesc,
                                            idesc_qk, acc);
                            else
                                ptx::mma_ss(d,
                                            ptx::desc_sw128(qs + uint32_t((kb - kQTmemBlocks) *
                                                                          16384 + kk * 32),
                                                            16, 1024),
                                            bdesc, idesc_qk, acc);
                        }
                    }
                    ptx::mma_commit(b_sfull);
                    ++nq;
                    did = true;
                } else if (np < nq &&
                           ptx::mbar_test_wait(b_pfull + 8 * (np & 1), (np >> 1) & 1)) {
                    ptx::tc_fence_after();
                    const int s = np % kStages;
                    const uint32_t st = stage_base + uint32_t(s * kStageBytes);
                    const uint32_t pb = pbase + uint32_t((np & 1) * 2 * kPHalfBytes);
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const uint32_t vb = st + uint32_t(pv_box(rank, r) * kBoxBytes);
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            ptx::mma_ss(tmem + kTmemO,
                                        ptx::desc_sw64(pb + uint32_t(r * kPHalfBytes + kk * 32), 512),
                                        ptx::desc_sw128(vb + uint32_t(kk * 16 * 128), kBoxBytes, 1024),
                                        idesc_pv, (np > 0 || r > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    ptx::mma_commit(b_pvdone);
                    ptx::mma_commit_mc(b_empty + 8 * s, kBothCtas);
                    ptx::mma_commit_mc(b_pfree + 8 * (np & 1), kBothCtas);
                    ++np;
                    did = true;
                }
                if (did) {
                    idle = 0;
                } else if (++idle == 1) {
                    idle_since = ptx::globaltimer();
                } else if ((idle & 255u) == 0u) {
                    if (aborting(bars)) break;
                    if (ptx::globaltimer() - idle_since > kTimeoutNs) {
                        set_abort(bars, p.status, kSiteMma);
                        break;
                    }
                }
            }
            // All MMAs of this CTA complete before TMEM is released.
            ptx::mma_commit(b_final);
            wait_phase(b_final, 0, bars, p.status, kSiteDrain, true);
        }
    } else {
        // ------------------------------------------- softmax / exchange / epilogue
        const int quarter = warp & 3;
        const int h = quarter * 32 + lane;
        const uint32_t trow = tmem + (uint32_t(quarter * 32) << 16);
        const bool live_head = h < N;
        const uint16_t* qrow = p.q + (size_t(b) * N + h) * kD;

        // q dims 0..447 -> TMEM (A operand), dims 448..575 -> shared memory.
        {
#pragma unroll 1
            for (int c = 0; c < kQTmemBlocks; ++c) {
                uint32_t r[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = 0u;
                if (live_head) {
                    const uint4* src = reinterpret_cast<const uint4*>(qrow + 64 * c);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint4 v = __ldg(src + i);
                        r[4 * i + 0] = v.x;
                        r[4 * i + 1] = v.y;
                        r[4 * i + 2] = v.z;
                        r[4 * i + 3] = v.w;
                    }
                }
                ptx::tmem_st32(trow + kTmemQ + uint32_t(c * 32), r);
            }
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
                unsigned char* row = smem + kOffQS + kb * 16384 + h * 128;
                const uint4* src = reinterpret_cast<const uint4*>(qrow + 64 * (kQTmemBlocks + kb));
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 v = make_uint4(0, 0, 0, 0);
                    if (live_head) v = __ldg(src + c);
                    *reinterpret_cast<uint4*>(row + ((c ^ (h & 7)) * 16)) = v;
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(b_qready);
        }

        float* small = reinterpret_cast<float*>(smem + kOffSmall);   // [buf][rank][3][128]
        float m_ref = -INFINITY;   // integer valued or -inf, log2 units
        float l_sum = 0.f;         // sum of fp32 weights at scale m_ref (for the LSE)
        float l_bf = 0.f;          // sum of the bf16 weights the MMA used (for O)
        uint32_t sync_phase = 0;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            const int buf = j & 1;
            // 1. Scores of this CTA's 32 tokens.
            ok = wait_phase(b_sfull, j & 1, bars, p.status, kSiteSFull);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            ptx::tc_fence_after();
            float x[32];
            {
                uint32_t r[32];
                ptx::tmem_ld32(trow + kTmemS, r);
#pragma unroll
                for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(r[i]);
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(b_sempty);

            // 2. Mask, local max, this CTA's base and weights.
            const int valid_page = min(kTile, t_hi - (t_lo + j * kTile));
            const int valid_own = max(0, min(kHalf, valid_page - kHalf * int(rank)));
            float mx = -INFINITY;
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                x[t] = t < valid_own ? x[t] * p.scale_log2 : -INFINITY;
                mx = fmaxf(mx, x[t]);
            }
            float base = m_ref;
            if (mx != -INFINITY && (m_ref == -INFINITY || mx > m_ref + kRescaleThreshold))
                base = ceilf(mx);
            uint32_t pk[16];
            float rs = 0.f, rs_bf = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float a = base == -INFINITY ? 0.f : ptx::ex2(x[2 * i] - base);
                const float c = base == -INFINITY ? 0.f : ptx::ex2(x[2 * i + 1] - base);
                rs += a + c;
                pk[i] = pack_bf16x2(a, c);
                rs_bf += __uint_as_float(pk[i] << 16) + __uint_as_float(pk[i] & 0xffff0000u);
            }

            // 3. Both CTAs finished the P.V that last read this buffer; my
            //    earlier copies have read their sources.
            ok = wait_phase(b_pfree + 8 * buf, ((j >> 1) & 1) ^ 1, bars, p.status, kSitePFree);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            if (h == 0) ptx::bulk_wait_read_all();
            ptx::mbar_arrive(b_smsync);
            ok = wait_phase(b_smsync, sync_phase++ & 1, bars, p.status, kSiteSmSync);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }

            // 4. Publish this CTA's half: P row (SW64), base and row sums.
            unsigned char* pbuf = smem + kOffP + buf * 2 * kPHalfBytes;
            unsigned char* prow_own = pbuf + rank * kPHalfBytes + h * 64;
            unsigned char* prow_peer = pbuf + peer * kPHalfBytes + h * 64;
#pragma unroll
            for (int c = 0; c < 4; ++c)
                *reinterpret_cast<uint4*>(prow_own + ((c ^ ((h >> 1) & 3)) * 16)) =
                    make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            float* mine = small + (buf * 2 + int(rank)) * 384;
            const float* theirs = small + (buf * 2 + int(peer)) * 384;
            mine[h] = base;
            mine[128 + h] = rs;
            mine[256 + h] = rs_bf;
            // Rows past the sequence end in the last page may hold anything
            // (even NaN): zero their value columns so that 0 * V stays 0.
            if (valid_page < kTile) {
                unsigned char* st = smem + kOffStages + (j % kStages) * kStageBytes;
#pragma unroll 1
                for (int r = 0; r < 2; ++r) {
                    const int valid_r = max(0, min(kHalf, valid_page - kHalf * r));
                    const int rows = kHalf - valid_r;
                    unsigned char* reg = st + pv_box(rank, r) * kBoxBytes;
                    for (int idx = h; idx < rows * 32; idx += 128) {
                        const int row = valid_r + idx / 32;
                        const int box = (idx / 8) & 3;
                        const int ch = idx & 7;
                        *reinterpret_cast<uint4*>(reg + box * kBoxBytes + row * 128 + ch * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(b_smsync);
            ok = wait_phase(b_smsync, sync_phase++ & 1, bars, p.status, kSiteSmSync);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            if (h == 0) {
                const uint32_t precv = b_precv + 8 * buf;
                ptx::mbar_arrive_expect_tx(precv, uint32_t(kPHalfBytes + kSmallBytes));
                const uint32_t precv_peer = ptx::mapa(precv, peer);
                const uint32_t src_p = ptx::smem_addr(pbuf + rank * kPHalfBytes);
                const uint32_t src_s = ptx::smem_addr(mine);
                ptx::bulk_copy_to_cluster(ptx::mapa(src_p, peer), src_p, kPHalfBytes, precv_peer);
                ptx::bulk_copy_to_cluster(ptx::mapa(src_s, peer), src_s, kSmallBytes, precv_peer);
                ptx::bulk_commit_group();
            }

            // 5. The other half arrives; agree on the new reference max.
            ok = wait_phase(b_precv + 8 * buf, (j >> 1) & 1, bars, p.status, kSitePRecv);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            const float base_peer = theirs[h];
            const float rs_peer = theirs[128 + h];
            const float rs_bf_peer = theirs[256 + h];
            const float b0 = rank == 0 ? base : base_peer;
            const float b1 = rank == 0 ? base_peer : base;
            const float m_new = fmaxf(b0, b1);
            const float f0 = b0 == -INFINITY ? 0.f : ptx::pow2i(int(b0 - m_new));
            const float f1 = b1 == -INFINITY ? 0.f : ptx::pow2i(int(b1 - m_new));
            const float alpha = m_ref == -INFINITY ? 0.f : ptx::pow2i(int(m_ref - m_new));
            const float r0 = rank == 0 ? rs : rs_peer;
            const float r1 = rank == 0 ? rs_peer : rs;
            const float q0 = rank == 0 ? rs_bf : rs_bf_peer;
            const float q1 = rank == 0 ? rs_bf_peer : rs_bf;
            l_sum = l_sum * alpha + r0 * f0 + r1 * f1;
            l_bf = l_bf * alpha + q0 * f0 + q1 * f1;
            const float f_own = rank == 0 ? f0 : f1;
            const float f_peer = rank == 0 ? f1 : f0;
            if (f_own != 1.f) scale_p_row(prow_own, f_own);
            if (f_peer != 1.f) scale_p_row(prow_peer, f_peer);
            m_ref = m_new;

            // 6. Rescale O when the reference moved (O holds P.V of earlier tiles).
            if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
                ok = wait_phase(b_pvdone, (j - 1) & 1, bars, p.status, kSitePvDone);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                ptx::tc_fence_after();
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
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(b_pfull + 8 * buf);
        }
        if (h == 0) ptx::bulk_wait_read_all();

        // Epilogue: O / l -> bf16 output, or the fp32 split partial.
        if (ok && ntiles > 0) {
            ok = wait_phase(b_pvdone, (ntiles - 1) & 1, bars, p.status, kSitePvDone);
            ok = __all_sync(0xffffffffu, ok);
            ptx::tc_fence_after();
        }
        if (ok && aligned_ok) {
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
                    float4* dst =
                        reinterpret_cast<float4*>(p.o_part + (row * S + split) * kLkv + col);
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
    const cuuint32_t box[2] = {64, kHalf};
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
