// Tensor-core decode kernel for sm_103a (MLA_KERNEL_TC): tcgen05 MMAs with
// TMEM accumulators and TMA page loads.
//
// What it computes is the absorbed ("forward_mqa") MLA decode of the vLLM
// mla_attention API docs, module docstring, "Data-Movement Friendly
// Approach": for one request and one split of its cached tokens, every head
// attends to every token with K = the 576-wide latent entry and V = its first
// 512 columns. The design is this file's own.
//
// Work is cut into segments (tokens [t_lo, t_hi) of one request): a CTA
// pair, two CTAs launched as a cluster so that they run side by side, walks
// its segments in order (the page-balanced schedule: the requests its range
// of work units touches; the split schedule: a contiguous run of (request,
// split) items). CTA c owns the value columns [256c, 256c+256) of O;
// everything else it does on its own, with no traffic between the two:
//   * Scores: the full tile S = Q K^T for all (up to) 128 heads and the 64
//     tokens of a page, tcgen05.mma M=128, N=64, K=16 (36 steps). An MMA with
//     N = 32 costs the tensor pipe about as much as one with N = 64 (so
//     splitting a page's tokens between the CTAs would save no tensor time),
//     and splitting its dims needs the partial scores exchanged, which costs
//     more than it saves; so the score tile is computed in both CTAs, which
//     keeps the softmax local. q's dims 0..255 are the A operand in TMEM,
//     dims 256..575 in shared memory.
//   * Each page is TMA-loaded by both CTAs (the second read of a page is
//     served from L2; pulling pages into L2 ahead of the loads measured
//     slower). Its 64-column blocks go to two page rings: this CTA's four
//     value blocks to a V ring (kept until the P.V MMA of the page), the five
//     other blocks to a K ring (released once the page's score MMAs finish).
//   * Softmax: 128 threads, one per head (= TMEM lane), fp32, base 2 with the
//     scale folded into the weights' FMA; the reference max moves only when a
//     page raises it by more than 8 (log2), so the O rescale (a TMEM
//     read-modify-write) is rare. The bf16 weights P overwrite the page's
//     scores in TMEM; O is normalised by the sum of those rounded weights and
//     the LSE keeps the fp32 sum.
//   * O_c[128 x 256] += P[128 x 64] V_c[64 x 256]: P the A operand in TMEM,
//     V read MN-major from the V ring.
// Two score buffers in TMEM let the score MMAs of the next page run while the
// softmax works on the current one.
//
// Warp roles: 0 = K-ring loads (and the next q's L2 prefetch), 6 = V-ring loads,
// 1 = score MMAs (one elected lane per segment), 2-5 = softmax, P.V MMAs, O
// correction and epilogue. The two rings have their own producers, so a
// page's K blocks never wait behind the previous page's V slot; the softmax
// warp that finishes a page last issues its P.V MMAs, with no hand-off to
// another warp. An issuing thread blocks until the tensor pipe takes each
// MMA, so the score lane keeps its own instructions few (operand descriptors
// come from a table built once; four MMAs per asm statement) and tests the
// barriers it will need inside those statements, waiting only when a test
// found the phase pending. Every wait is bounded: on expiry the kernel
// records MLA_ERR_TIMEOUT, lets each role leave its loop, waits (bounded) for
// its own loads and MMAs, frees TMEM and returns. A block id outside the pool
// is recorded and loaded from negative rows, which TMA fills with zeros.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <climits>
#include <cmath>

#include "mla_device.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace {

constexpr int kThreads = 224;                  // 7 warps
constexpr int kThreadsFp8 = 352;               // fp8 cache: + 4 warps that widen pages to f16
constexpr int kFp8BlockBytes = 64 * 64;        // 64 rows x 64 E4M3 columns = 4 KB
constexpr int kTile = 64;                      // tokens per page
constexpr int kBlockBytes = kTile * 128;       // 64 rows x 64 bf16 columns = 8 KB
constexpr int kKPerPage = 5;                   // K-ring blocks per page
constexpr int kVBytes = 4 * kBlockBytes;       // a page's four value blocks: 32 KB
constexpr int kKBytes = kKPerPage * kBlockBytes;   // a page's five K-ring blocks: 40 KB
constexpr int kQPrefetchPages = 1;             // next request's q pulled into L2 this many pages early

constexpr int kOffQS = 0;                      // q dims 256..575: 5 x [128 x 64] bf16, SW128
constexpr int kOffV = 5 * 16384;               // V ring: 2 pages
constexpr int kOffK = kOffV + 2 * kVBytes;     // K ring: 2 pages
constexpr int kOffBar = kOffK + 2 * kKBytes;   // 229,376
constexpr int kOffPfx = kOffBar + 256;         // page offsets of the balanced schedule
// UMMA descriptors of every score-MMA operand, built once by the score warp:
// q's five shared-memory blocks (4 K-steps each), then per ring slot the
// five K-ring and four value blocks (4 K-steps each).
constexpr int kDescA = 5 * 4;
constexpr int kDescSlot = 9 * 4;
constexpr int kOffDesc = kOffPfx + (kMaxBalancedBatch + 4) * 4;
constexpr int kSmemBytes = kOffDesc + (kDescA + 2 * kDescSlot) * 8;   // base is 1 KB aligned
static_assert(kOffDesc % 16 == 0, "descriptor table alignment");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemQ = 0;     // 128 columns: q dims 0..255 as bf16 pairs (A operand)
constexpr uint32_t kTmemS = 128;   // two 64-column score buffers; P (32 columns) overwrites S
constexpr uint32_t kTmemO = 256;   // 256 fp32 columns of O
constexpr int kQTmemBlocks = 4;    // 64-dim blocks of q held in TMEM

// A waiting thread sleeps in mbarrier.try_wait until the phase completes (or
// this long), so waiting warps take no issue slots from the working ones.
constexpr uint32_t kSuspendNs = 20000;
constexpr int kSoftmaxSpin = 256;   // polls of s_full before the softmax warps sleep
constexpr float kLn2 = 0.693147180559945309f;
constexpr float kRescaleThreshold = 8.0f;         // log2 units

// Barriers. Page j uses ring slot j & 1 everywhere; each barrier of a pair
// completes once per page of its parity, so a wait has at most one phase
// pending.
struct TcBars {
    uint64_t vfull[2];    // TMA: value blocks landed
    uint64_t vempty[2];   // P.V MMA done with them
    uint64_t kfull[2];    // TMA: K-ring blocks landed
    uint64_t kempty[2];   // score MMAs done with them
    uint64_t s_full[2];   // score MMAs of the page complete
    uint64_t p_free[2];   // P.V MMA complete: score buffer free, O current
    uint64_t q_ready;     // q staged (128 arrivals)
    uint64_t q_staged;    // q dims 0..255 copied to the staging area (128 arrivals)
    uint64_t q_read;      // staging area read into TMEM (128 arrivals)
    uint64_t final_qk;    // drain of the score warp's MMAs
    uint64_t final_sm[4]; // drain of each softmax warp's P.V MMAs
    uint64_t kstaged[2];  // fp8 cache: TMA: the K-ring blocks' codes landed
    uint64_t vstaged[2];  // fp8 cache: TMA: the value blocks' codes landed
    uint32_t p_count[2];  // softmax warps done with the pages of each parity
    uint32_t tmem_base;
    int32_t abort;
};
static_assert(sizeof(TcBars) <= 256, "barrier block too large");

enum WaitSite : int32_t {
    kSiteVEmpty = 1, kSiteKEmpty, kSiteSFull, kSiteSFree, kSitePvDone, kSiteQReady,
    kSiteDrain, kSiteKFull, kSiteVFull, kSiteStaged
};

__device__ __forceinline__ bool aborting(TcBars* bars) {
    return *reinterpret_cast<volatile int32_t*>(&bars->abort) != 0;
}

__device__ __forceinline__ void set_abort(TcBars* bars, int32_t* status, int32_t site) {
    *reinterpret_cast<volatile int32_t*>(&bars->abort) = 1;
    record_error(status, MLA_ERR_TIMEOUT, site);
}

// Bounded wait on a local mbarrier phase (at most `limit_ns`). Returns false
// when the kernel is aborting (another role timed out) or when this wait
// expires. The score warp waits with the call's limit and the roles that
// depend on it (the loaders, the softmax warps) with twice that, so that
// when something stops, the wait nearest the cause is the one recorded.
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, TcBars* bars,
                                       int32_t* status, int32_t site, bool ignore_abort,
                                       uint64_t limit_ns) {
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
        for (int i = 0; i < 4; ++i)
            if (ptx::mbar_try_wait_sleep(bar, parity, kSuspendNs)) return true;
        if (!ignore_abort && aborting(bars)) return false;
        if (ptx::globaltimer() - t0 > limit_ns) {
            set_abort(bars, status, site);
            return false;
        }
    }
}

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, TcBars* bars,
                                           int32_t* status, int32_t site, uint64_t limit_ns,
                                           bool ignore_abort = false) {
    if (ptx::mbar_test_wait(bar, parity)) return true;
    return wait_slow(bar, parity, bars, status, site, ignore_abort, limit_ns);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// The two 16-bit weights of a packed pair, as the MMA reads them.
template <bool kF16>
__device__ __forceinline__ float2 unpack_x2(uint32_t w) {
    if constexpr (kF16) {
        return __half22float2(*reinterpret_cast<const __half2*>(&w));
    } else {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
}

// Two bf16 q values (one 32-bit word) as two f16 (exact for |q| <= 65504;
// `big` is set when a value lies beyond that).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w, bool& big) {
    const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xffff0000u);
    big = big || !(fabsf(lo) <= 65504.f) || !(fabsf(hi) <= 65504.f);
    return pack_f16x2(lo, hi);
}

// The 64-column block kb (dims 64kb..64kb+63) of a page is one of this CTA's
// value blocks when kb is in [4c, 4c+4); the five others go to the K ring,
// in ascending kb (position pos = 0..4).
__host__ __device__ constexpr int k_block(int rank, int pos) {
    return rank == 0 ? pos + 4 : (pos < 4 ? pos : 8);
}

// ------------------------------------------------------------ work segments
// A CTA pair works through one or more segments: tokens [t_lo, t_hi) of a
// request. In the split schedule the B*S items (b, split), b-major, are cut
// into one contiguous run per CTA pair and each item is a segment; the
// page-balanced schedule gives a pair the requests its page range touches
// (the page offsets pfx[b] = pages of requests 0..b-1 are in shared memory).
struct Segment {
    int b;
    int L;             // the request's length (multi-token rows end before it)
    int t_lo, t_hi;
    int prow0;         // partial row of head 0, or -1: write out / lse directly
    int prow_stride;   // partial rows from one head to the next
};

struct SegmentWalk {
    int next_b;        // balanced: next request to look at
    int64_t g0, g1;    // balanced: the pair's unit range; split: its item range
    bool first;        // balanced: no segment returned yet
};

__device__ __forceinline__ SegmentWalk walk_begin(const DecodeParams& p, const int32_t* pfx,
                                                  int pair) {
    SegmentWalk w{0, 0, 0, true};
    if (p.sched_pairs == 0) {
        const int64_t items = int64_t(p.batch) * p.num_splits;
        const int64_t pairs = int64_t(gridDim.x >> 1);
        w.g0 = pair * items / pairs;
        w.g1 = (pair + 1) * items / pairs;
    } else {
        const int64_t total = pfx[p.batch];
        if (total > 0) {
            w.g0 = pair_begin(pair, p.sched_pairs, total);
            w.g1 = pair_begin(pair + 1, p.sched_pairs, total);
        }
        // The first request whose pages reach past g0.
        int lo = 0, hi = p.batch;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (pfx[mid + 1] > w.g0)
                hi = mid;
            else
                lo = mid + 1;
        }
        w.next_b = lo;
    }
    return w;
}

__device__ __forceinline__ bool walk_next(const DecodeParams& p, const int32_t* pfx, int pair,
                                          SegmentWalk& w, Segment& s) {
    if (p.sched_pairs == 0) {
        if (w.g0 >= w.g1) return false;
        const int S = p.num_splits;
        const int64_t item = w.g0++;
        const int split = int(item % S);
        s.b = int(item / S);
        s.L = checked_seq_len(p, s.b);
        split_range(s.L, S, split, &s.t_lo, &s.t_hi);
        s.prow0 = S == 1 ? -1 : s.b * p.num_heads * S + split;
        s.prow_stride = S;
        return true;
    }
    while (w.next_b < p.batch && pfx[w.next_b] < w.g1) {
        const int b = w.next_b++;
        if (pfx[b + 1] == pfx[b]) continue;   // no pages: the merge writes this request
        // The request's pages occupy units [pb, pe), after its fixed cost.
        const int64_t pb = pfx[b] + kSegmentCostPages, pe = pfx[b + 1];
        const int64_t lo = pb > w.g0 ? pb : w.g0;
        const int64_t hi = pe < w.g1 ? pe : w.g1;
        if (lo >= hi) continue;   // only the fixed cost falls in this range
        s.b = b;
        s.L = p.seq_lens[b];
        s.t_lo = int(lo - pb) * kPageSize;
        s.t_hi = min(p.seq_lens[b], int(hi - pb) * kPageSize);
        s.prow0 = (lo == pb && hi == pe) ? -1 : (w.first ? 2 * pair : 2 * pair + 1) * p.num_heads;
        s.prow_stride = 1;
        w.first = false;
        return true;
    }
    return false;
}

__device__ __forceinline__ int seg_pages(const Segment& s) {
    return (s.t_hi - s.t_lo + kTile - 1) / kTile;
}

// ------------------------------------------------------------ MMA issue
// The score warp blocks on its barriers in a suspended wait (not a spin that
// would take issue slots from the softmax warps), runs its loop in lockstep
// and issues every tcgen05 op from one elected lane; a page's score MMAs are
// unrolled at compile time (a template on the CTA rank), so every operand is
// a warp-uniform base plus a constant and the issue keeps up with the pipe.

struct MmaWarpArgs {
    uint32_t tmem, sbase;
    TcBars* bars;
    int32_t* status;
    unsigned char* smem;
    uint64_t limit_ns;   // the score warp's wait limit
};

// Slow path of warp_wait, out of line. Called by the whole warp; returns
// lane 0's answer.
__device__ __noinline__ int warp_wait_slow(uint32_t bar, uint32_t parity, TcBars* bars,
                                           int32_t* status, int32_t site, uint64_t limit_ns) {
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (__shfl_sync(0xffffffffu, ptx::mbar_try_wait_sleep(bar, parity, kSuspendNs) ? 1 : 0,
                        0) != 0)
            return 1;
        if ((it & 3u) == 0u) {
            int stop = aborting(bars) ? 1 : 0;
            if (!stop && ptx::globaltimer() - t0 > limit_ns) stop = 2;
            stop = __shfl_sync(0xffffffffu, stop, 0);
            if (stop != 0) {
                if (stop == 2 && (threadIdx.x & 31) == 0) set_abort(bars, status, site);
                return 0;
            }
        }
    }
}

// Bounded wait with one answer for the whole warp (lane 0's). Returns false
// when the kernel is aborting or this wait expires (then it records the
// timeout).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const MmaWarpArgs& a,
                                          int32_t site) {
    if (__shfl_sync(0xffffffffu, ptx::mbar_test_wait(bar, parity) ? 1 : 0, 0) != 0) return true;
    return __shfl_sync(0xffffffffu,
                       warp_wait_slow(bar, parity, a.bars, a.status, site, a.limit_ns), 0) != 0;
}

// Every tcgen05 op this warp issued completes before the CTA frees TMEM.
__device__ __forceinline__ void warp_drain(uint32_t bar, const MmaWarpArgs& a) {
    if (ptx::elect_one()) ptx::mma_commit(bar);
    __syncwarp();
    if ((threadIdx.x & 31) == 0) wait_phase(bar, 0, a.bars, a.status, kSiteDrain, a.limit_ns, true);
    __syncwarp();
}

__device__ __forceinline__ uint64_t desc_kmajor(uint32_t addr) {
    return ptx::desc_sw128(addr, 16, 1024);    // K-major SW128: 8-row groups 1 KB apart
}
__device__ __forceinline__ uint64_t desc_vmn(uint32_t addr) {
    return ptx::desc_sw128(addr, kBlockBytes, 1024);   // MN-major: 64-col blocks, 8-token groups
}

// Four score MMAs (K = 64 dims) of dim block KB against the 64 x 64 block
// whose four K-step descriptors are at bdesc (q's shared-memory blocks' at
// desc). Called by one elected lane. With bar != 0 the
// block also tests the mbarrier phase (bar, parity) without blocking, before
// its first MMA, and reads the answer after its fourth (returned).
template <int KB, bool kF16>
__device__ __forceinline__ uint32_t score_block(uint32_t d, uint32_t tmem, const uint64_t* desc,
                                                const uint64_t* bdesc, bool first,
                                                uint32_t bar = 0, uint32_t parity = 0) {
    constexpr uint32_t idesc_qk =
        kF16 ? ptx::idesc_f16_f32(kTile, false) : ptx::idesc_bf16_f32(kTile, false);
    const uint32_t acc0 = first ? 0u : 1u;
    const ulonglong2 b01 = *reinterpret_cast<const ulonglong2*>(bdesc);
    const ulonglong2 b23 = *reinterpret_cast<const ulonglong2*>(bdesc + 2);
    const uint64_t bd[4] = {b01.x, b01.y, b23.x, b23.y};
    if (KB < kQTmemBlocks) {
        const uint32_t at = tmem + kTmemQ + uint32_t(KB * 32);
        if (bar != 0)
            return ptx::mma4_ts_probe(d, at, at + 8, at + 16, at + 24, bd[0], bd[1], bd[2], bd[3],
                                      idesc_qk, acc0, bar, parity);
        ptx::mma4_ts(d, at, at + 8, at + 16, at + 24, bd[0], bd[1], bd[2], bd[3], idesc_qk, acc0);
    } else {
        const uint64_t* ad4 = desc + (KB - kQTmemBlocks) * 4;
        const ulonglong2 a01 = *reinterpret_cast<const ulonglong2*>(ad4);
        const ulonglong2 a23 = *reinterpret_cast<const ulonglong2*>(ad4 + 2);
        const uint64_t ad[4] = {a01.x, a01.y, a23.x, a23.y};
        if (bar != 0)
            return ptx::mma4_ss_probe(d, ad[0], ad[1], ad[2], ad[3], bd[0], bd[1], bd[2], bd[3],
                                      idesc_qk, acc0, bar, parity);
        ptx::mma4_ss(d, ad[0], ad[1], ad[2], ad[3], bd[0], bd[1], bd[2], bd[3], idesc_qk, acc0);
    }
    return 1u;
}

// S = Q K^T for every page: the five K-ring blocks, then the four value
// blocks. CTA 0's K-ring blocks are dims 256..575 (q from shared memory) and
// its value blocks dims 0..255 (q from TMEM); CTA 1's K-ring blocks are dims
// 0..255 (TMEM) and 512..575 (shared memory), its value blocks dims 256..511
// (shared memory). Pages are numbered across segments (jg) for the rings;
// each segment waits for its own q.
template <int RANK, bool kF16>
__device__ __forceinline__ void score_warp(const MmaWarpArgs& a, const uint32_t* b,
                                           const DecodeParams& p, const int32_t* pfx, int pair) {
    const uint32_t b_kfull = b[0], b_kempty = b[1], b_vfull = b[2], b_sfull = b[3],
                   b_pfree = b[4], b_qready = b[5], b_final = b[6];
    const uint32_t tmem = a.tmem;
    // The descriptor table (the operands' shared-memory addresses never
    // change): lanes fill it, the elected lane reads it after __syncwarp.
    uint64_t* desc = reinterpret_cast<uint64_t*>(a.smem + kOffDesc);
    for (int i = int(threadIdx.x & 31); i < kDescA + 2 * kDescSlot; i += 32) {
        uint32_t off;
        if (i < kDescA) {
            off = uint32_t(kOffQS + (i >> 2) * 16384 + (i & 3) * 32);
        } else {
            const int e = i - kDescA, sl = e / kDescSlot, r = e % kDescSlot;
            const int pos = r >> 2, kk = r & 3;
            off = pos < kKPerPage
                      ? uint32_t(kOffK + sl * kKBytes + pos * kBlockBytes + kk * 32)
                      : uint32_t(kOffV + sl * kVBytes + (pos - kKPerPage) * kBlockBytes + kk * 32);
        }
        desc[i] = desc_kmajor(a.sbase + off);
    }
    __syncwarp();
    SegmentWalk walk = walk_begin(p, pfx, pair);
    Segment sg;
    int jg = 0;
    int nseg = 0;   // q stagings waited for so far (one q_ready phase each)
    int q_b = -1;   // request whose q is staged
    bool ok = true;
    while (ok && walk_next(p, pfx, pair, walk, sg)) {
        const int ntiles = seg_pages(sg);
        if (ntiles == 0) continue;
        // A new request's q (consecutive splits of one request share it).
        if (sg.b != q_b) {
            ok = warp_wait(b_qready, uint32_t(nseg++) & 1u, a, kSiteQReady);
            if (!ok) break;
            q_b = sg.b;
        }
        // One elected lane issues the whole segment. Each barrier it needs
        // is first probed inside an earlier MMA (the probe's latency passes
        // while the lane waits for the pipe), and it only waits when the
        // probe found the phase still pending.
        const int jg0 = jg;
        if (ptx::elect_one()) {
            // This page's score buffer and K-ring blocks, found free / landed
            // by probes during the previous page.
            bool pf_ready = false, kf_ready = false;
            for (int j = 0; j < ntiles; ++j) {
                const int jc = jg0 + j;
                const int sl = jc & 1;
                const uint32_t ph = uint32_t(jc >> 1) & 1u;
                // The score buffer is free once the P.V MMA of page jc-2 has read P.
                if (jc >= 2 && !pf_ready &&
                    !wait_phase(b_pfree + 8 * sl, ph ^ 1u, a.bars, a.status, kSiteSFree,
                                a.limit_ns))
                    break;
                if (!kf_ready &&
                    !wait_phase(b_kfull + 8 * sl, ph, a.bars, a.status, kSiteKFull, a.limit_ns))
                    break;
                ptx::tc_fence_after();
                const uint32_t d = tmem + kTmemS + uint32_t(sl * 64);
                const uint64_t* bk = desc + kDescA + sl * kDescSlot;   // K-ring blocks
                const uint64_t* bv = bk + kKPerPage * 4;               // value blocks
                const uint32_t b_vf = b_vfull + 8 * sl;
                // Page jn (the next one; it may lie in the next segment or not
                // exist, and then the answers are not used): its K-ring blocks
                // are probed early (they landed long ago), its score buffer as
                // late as possible (the P.V of page jc-1 finishes about now).
                const int jn = jc + 1;
                const uint32_t phn = uint32_t(jn >> 1) & 1u;
                score_block<k_block(RANK, 0), kF16>(d, tmem, desc, bk + 0, true);
                const uint32_t nk = score_block<k_block(RANK, 1), kF16>(
                    d, tmem, desc, bk + 4, false, b_kfull + 8 * (jn & 1), phn);
                score_block<k_block(RANK, 2), kF16>(d, tmem, desc, bk + 8, false);
                const uint32_t vr = score_block<k_block(RANK, 3), kF16>(
                    d, tmem, desc, bk + 12, false, b_vf, ph);
                score_block<k_block(RANK, 4), kF16>(d, tmem, desc, bk + 16, false);
                ptx::mma_commit(b_kempty + 8 * sl);
                if (!vr && !wait_phase(b_vf, ph, a.bars, a.status, kSiteVFull, a.limit_ns)) break;
                score_block<4 * RANK + 0, kF16>(d, tmem, desc, bv + 0, false);
                score_block<4 * RANK + 1, kF16>(d, tmem, desc, bv + 4, false);
                score_block<4 * RANK + 2, kF16>(d, tmem, desc, bv + 8, false);
                const uint32_t nf = score_block<4 * RANK + 3, kF16>(
                    d, tmem, desc, bv + 12, false, b_pfree + 8 * (jn & 1), phn ^ 1u);
                ptx::mma_commit(b_sfull + 8 * sl);
                const bool more = j + 1 < ntiles;
                pf_ready = more && nf != 0;
                kf_ready = more && nk != 0;
            }
        }
        __syncwarp();
        jg = jg0 + ntiles;
        if (aborting(a.bars)) ok = false;
    }
    warp_drain(b_final, a);
}

// O += P V for page np: P the A operand in TMEM, V (MN-major) from the V
// ring. Issued by one elected lane of the softmax warp that finished the page
// last; the commits release the V slot and the score buffer.
template <bool kF16>
__device__ __forceinline__ void issue_pv(uint32_t tmem, uint32_t sbase, int np, bool accumulate,
                                         uint32_t b_vempty, uint32_t b_pfree) {
    constexpr uint32_t idesc_pv =
        kF16 ? ptx::idesc_f16_f32(256, true) : ptx::idesc_bf16_f32(256, true);
    const int sl = np & 1;
    const uint32_t pcol = tmem + kTmemS + uint32_t(sl * 64);
    const uint32_t vb = sbase + uint32_t(kOffV + sl * kVBytes);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        ptx::mma_ts(tmem + kTmemO, pcol + uint32_t(kk * 8), desc_vmn(vb + uint32_t(kk * 2048)),
                    idesc_pv, (accumulate || kk > 0) ? 1u : 0u);
    ptx::mma_commit(b_vempty + 8 * sl);
    ptx::mma_commit(b_pfree + 8 * sl);
}


// ------------------------------------------------------------ page loaders
// Loader dump (test hook): the rows of a page as this CTA received them, from
// a ring slot of 64 x 64 bf16 blocks in the 128-byte swizzled layout (16-byte
// chunk c of row r at r * 128 + (c ^ (r % 8)) * 16), to
// p.dump[rank, b, t0 + r, :].
__device__ void dump_slot(const DecodeParams& p, const unsigned char* slot, bool k_ring,
                          uint32_t rank, int b, int t0, int rows) {
    const int nblk = k_ring ? kKPerPage : 4;
    for (int k = 0; k < nblk; ++k) {
        const int col0 = k_ring ? 64 * k_block(int(rank), k) : 256 * int(rank) + 64 * k;
        const unsigned char* blk = slot + k * kBlockBytes;
        for (int r = 0; r < rows && t0 + r < p.dump_max_tokens; ++r) {
            uint4* dst = reinterpret_cast<uint4*>(
                p.dump + ((size_t(rank) * p.batch + b) * p.dump_max_tokens + t0 + r) * kD + col0);
#pragma unroll
            for (int c = 0; c < 8; ++c)
                dst[c] = *reinterpret_cast<const uint4*>(blk + r * 128 + ((c ^ (r & 7)) * 16));
        }
    }
}

// One of the two page loaders (K ring or V ring), run by one thread. For
// every page of the pair's segments it waits for its ring slot to be free,
// then TMA-loads the page's blocks for this ring: box 64 columns x 64 rows of
// the tensor map over the cache viewed as [num_blocks * 64, 576], at row
// y = block * 64 (block = block_table[b, page]). With kDump the loader runs
// alone (no consumers free the slots): it waits for each page to land and
// copies it out with dump_slot. With kFp8 the tensor map is over the E4M3
// codes (64 x 64 one-byte boxes, unswizzled) and the boxes land in the upper
// half of the slot, which the converter warps widen in place to f16
// (b_full is then the barrier the converters wait on).
template <bool kDump, bool kFp8>
__device__ __forceinline__ void page_loader(const DecodeParams& p, const CUtensorMap* tmap,
                                            const int32_t* pfx, int pair, uint32_t rank,
                                            bool k_ring, TcBars* bars, unsigned char* smem,
                                            uint32_t sbase, uint32_t b_full, uint32_t b_empty,
                                            uint64_t limit_ns) {
    const int N = p.num_heads;
    const int slot_bytes = k_ring ? kKBytes : kVBytes;
    // bytes that land per page: the slot (bf16), or its upper half (E4M3)
    const int bytes = kFp8 ? slot_bytes / 2 : slot_bytes;
    const int box_bytes = kFp8 ? kFp8BlockBytes : kBlockBytes;
    const int off0 = k_ring ? kOffK : kOffV;
    const uint32_t dst0 = sbase + uint32_t(off0 + (kFp8 ? slot_bytes / 2 : 0));
    // Test hook: CTA 0 withholds its first K-ring load, so the score warp's
    // wait for it runs out.
    const bool withhold =
        !kDump && k_ring && blockIdx.x == 0 && (p.debug & kDebugWithholdLoad) != 0;
    SegmentWalk walk = walk_begin(p, pfx, pair);
    Segment sg;
    int jg = 0;   // pages issued so far, across segments
    bool ok = true;
    while (ok && walk_next(p, pfx, pair, walk, sg)) {
        const int ntiles = seg_pages(sg);
        const int page0 = sg.t_lo / kTile;
        const int32_t* table = p.block_table + size_t(sg.b) * p.max_blocks;
        // q of the next segment's request into L2 (half per CTA) a few pages
        // before this segment ends (earlier, the page stream would evict
        // it), so that staging it is short.
        int q_next = -1;
        if (k_ring && !kDump) {
            SegmentWalk peek = walk;
            Segment nx;
            if (walk_next(p, pfx, pair, peek, nx)) q_next = nx.b;
        }
        auto prefetch_q = [&]() {
            if (q_next < 0) return;
            const uint32_t qbytes = uint32_t(N) * kD * 2;   // a multiple of 16
            const unsigned char* qb =
                reinterpret_cast<const unsigned char*>(p.q + size_t(io_row(p, q_next)) * N * kD);
            const uint32_t half = (qbytes / 2) & ~15u;
            ptx::prefetch_l2(qb + rank * half, rank == 0 ? half : qbytes - half);
        };
        if (ntiles <= kQPrefetchPages) prefetch_q();
        int next = ntiles > 0 ? table[page0] : 0;
        for (int j = 0; j < ntiles; ++j, ++jg) {
            const int blk = next;
            if (j + 1 < ntiles) next = table[page0 + j + 1];
            if (j + kQPrefetchPages == ntiles) prefetch_q();
            int32_t y;
            if (blk >= 0 && int64_t(blk) < p.num_blocks) {
                y = blk * kTile;
            } else {
                if (k_ring) record_error(p.status, MLA_ERR_BAD_BLOCK_ID, blk);
                y = -kTile;   // wholly outside the tensor: TMA writes zeros
            }
            const int sl = jg & 1;
            if (!kDump && !wait_phase(b_empty + 8 * sl, (uint32_t(jg >> 1) & 1u) ^ 1u, bars,
                                      p.status, k_ring ? kSiteKEmpty : kSiteVEmpty, limit_ns)) {
                ok = false;
                break;
            }
            if (withhold && jg == 0) continue;
            ptx::mbar_arrive_expect_tx(b_full + 8 * sl, uint32_t(bytes));
            const uint32_t dst = dst0 + uint32_t(sl * slot_bytes);
            if (k_ring) {
                // The five K-ring blocks, in score order.
                for (int pos = 0; pos < kKPerPage; ++pos)
                    ptx::tma_load_2d(dst + uint32_t(pos * box_bytes), tmap,
                                     64 * k_block(int(rank), pos), y, b_full + 8 * sl);
            } else {
                // This CTA's four value blocks.
                for (int k = 0; k < 4; ++k)
                    ptx::tma_load_2d(dst + uint32_t(k * box_bytes), tmap,
                                     256 * int(rank) + 64 * k, y, b_full + 8 * sl);
            }
            if constexpr (kDump) {
                if (!wait_phase(b_full + 8 * sl, uint32_t(jg >> 1) & 1u, bars, p.status,
                                kSiteDrain, limit_ns, true)) {
                    ok = false;
                    ++jg;   // issued: the drain below waits for it once more
                    break;
                }
                const int t0 = sg.t_lo + j * kTile;
                dump_slot(p, smem + off0 + sl * slot_bytes, k_ring, rank, sg.b, t0,
                          min(kTile, sg.t_hi - t0));
            }
        }
    }
    // Every issued load lands before the CTA may exit.
    for (int j = jg > 2 ? jg - 2 : 0; j < jg; ++j) {
        if (withhold && j == 0) continue;
        wait_phase(b_full + 8 * (j & 1), uint32_t(j >> 1) & 1u, bars, p.status, kSiteDrain,
                   limit_ns, true);
    }
}

// fp8 cache: widen a page's E4M3 codes to f16 in place. The loader put the
// ring's blocks of codes (64 rows x 64 bytes each, unswizzled) in the upper
// half of the slot; block k's f16 copy goes to the k-th 8 KB of the slot in
// the 128-byte swizzled layout the MMAs read. Block k's f16 bytes overlap
// only the codes of blocks <= k, so the 64 converter threads of the ring
// read a whole block, meet at a named barrier, then write it. The
// conversion is exact (every E4M3 value is an f16 value). Each thread then
// makes its writes visible to the tensor cores and arrives on b_full (64
// arrivals per page).
template <bool kKRing>
__device__ __forceinline__ void page_converter(const DecodeParams& p, const int32_t* pfx,
                                               int pair, TcBars* bars, unsigned char* smem,
                                               uint32_t b_staged, uint32_t b_full, int ct,
                                               uint64_t limit_ns) {
    constexpr int nblk = kKRing ? kKPerPage : 4;
    constexpr int slot_bytes = kKRing ? kKBytes : kVBytes;
    constexpr uint32_t bar_id = kKRing ? 1u : 2u;
    unsigned char* ring = smem + (kKRing ? kOffK : kOffV);
    SegmentWalk walk = walk_begin(p, pfx, pair);
    Segment sg;
    int jg = 0;
    bool ok = true;
    while (ok && walk_next(p, pfx, pair, walk, sg)) {
        const int ntiles = seg_pages(sg);
        for (int j = 0; j < ntiles; ++j, ++jg) {
            const int sl = jg & 1;
            const bool landed = wait_phase(b_staged + 8 * sl, uint32_t(jg >> 1) & 1u, bars,
                                           p.status, kSiteStaged, limit_ns);
            // One decision for all 64 threads: the named barriers below need
            // every one of them.
            if (ptx::named_barrier_or(bar_id, 64, !landed || aborting(bars))) {
                ok = false;
                break;
            }
            unsigned char* slot = ring + sl * slot_bytes;
            const unsigned char* codes = slot + slot_bytes / 2;
#pragma unroll 1
            for (int blk = 0; blk < nblk; ++blk) {
                uint4 v[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int i = ct + 64 * k;          // 256 chunks of 16 codes
                    v[k] = *reinterpret_cast<const uint4*>(codes + blk * kFp8BlockBytes +
                                                           (i >> 2) * 64 + (i & 3) * 16);
                }
                ptx::named_barrier_sync(bar_id, 64);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int i = ct + 64 * k;
                    const int r = i >> 2, cc = i & 3;
                    const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
                    uint32_t h[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(
                            __nv_fp8x2_storage_t(w[e] & 0xffffu), __NV_E4M3);
                        const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(
                            __nv_fp8x2_storage_t(w[e] >> 16), __NV_E4M3);
                        h[2 * e] = uint32_t(lo.x) | (uint32_t(lo.y) << 16);
                        h[2 * e + 1] = uint32_t(hi.x) | (uint32_t(hi.y) << 16);
                    }
                    unsigned char* row = slot + blk * kBlockBytes + r * 128;
                    *reinterpret_cast<uint4*>(row + (((2 * cc) ^ (r & 7)) * 16)) =
                        make_uint4(h[0], h[1], h[2], h[3]);
                    *reinterpret_cast<uint4*>(row + (((2 * cc + 1) ^ (r & 7)) * 16)) =
                        make_uint4(h[4], h[5], h[6], h[7]);
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(b_full + 8 * sl);
        }
    }
}

template <bool kDump, bool kFp8>
__global__ void __launch_bounds__(kFp8 ? kThreadsFp8 : kThreads, 1)
mla_decode_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmap) {
    extern __shared__ __align__(1024) unsigned char smem[];
    TcBars* bars = reinterpret_cast<TcBars*>(smem + kOffBar);
    int32_t* pfx = reinterpret_cast<int32_t*>(smem + kOffPfx);
    const uint32_t sbase = ptx::smem_addr(smem);
    // The page-balanced merge is launched as a programmatic dependent of this
    // kernel: it may start on SMs this grid has left, and waits for each
    // request's partial rows through counters (never for the whole grid).
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const int N = p.num_heads;
    const int pair = blockIdx.x >> 1;

    // Swizzled TMA boxes and UMMA descriptors assume a 1 KB aligned base.
    const bool aligned_ok = (sbase & 1023u) == 0u;

    const uint32_t b_vfull = ptx::smem_addr(&bars->vfull[0]);
    const uint32_t b_vempty = ptx::smem_addr(&bars->vempty[0]);
    const uint32_t b_kfull = ptx::smem_addr(&bars->kfull[0]);
    const uint32_t b_kempty = ptx::smem_addr(&bars->kempty[0]);
    const uint32_t b_sfull = ptx::smem_addr(&bars->s_full[0]);
    const uint32_t b_pfree = ptx::smem_addr(&bars->p_free[0]);
    const uint32_t b_qready = ptx::smem_addr(&bars->q_ready);
    const uint32_t b_qstaged = ptx::smem_addr(&bars->q_staged);
    const uint32_t b_qread = ptx::smem_addr(&bars->q_read);
    const uint32_t b_final_qk = ptx::smem_addr(&bars->final_qk);
    const uint32_t b_final_sm = ptx::smem_addr(&bars->final_sm[0]);
    const uint32_t b_kstaged = ptx::smem_addr(&bars->kstaged[0]);
    const uint32_t b_vstaged = ptx::smem_addr(&bars->vstaged[0]);
    const uint32_t a_pcount = ptx::smem_addr(&bars->p_count[0]);

    if (warp == 0) {
        if (lane == 0) {
            if (!aligned_ok) record_error(p.status, MLA_ERR_UNSUPPORTED, int32_t(sbase));
            // A slot is full after the TMA landed (bf16), or after the 64
            // converter threads of its ring widened it (fp8).
            const uint32_t full_count = kFp8 ? 64u : 1u;
            for (int i = 0; i < 2; ++i) {
                ptx::mbar_init(b_vfull + 8 * i, full_count);
                ptx::mbar_init(b_vempty + 8 * i, 1);
                ptx::mbar_init(b_kfull + 8 * i, full_count);
                ptx::mbar_init(b_kempty + 8 * i, 1);
                ptx::mbar_init(b_kstaged + 8 * i, 1);
                ptx::mbar_init(b_vstaged + 8 * i, 1);
                ptx::mbar_init(b_sfull + 8 * i, 1);
                ptx::mbar_init(b_pfree + 8 * i, 1);
                bars->p_count[i] = 0;
            }
            ptx::mbar_init(b_qready, 128);
            ptx::mbar_init(b_qstaged, 128);
            ptx::mbar_init(b_qread, 128);
            ptx::mbar_init(b_final_qk, 1);
            for (int i = 0; i < 4; ++i) ptx::mbar_init(b_final_sm + 8 * i, 1);
            bars->abort = 0;
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        if (p.sched_pairs > 0) {
            // Unit offsets of the balanced schedule: pfx[b] = work units of
            // requests 0..b-1 (a request with an invalid length has none).
            int carry = 0;
            for (int base = 0; base < p.batch; base += 128) {
                int pg[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int i = base + 32 * k + lane;
                    pg[k] = i < p.batch ? work_units(pages_of(checked_seq_len(p, i))) : 0;
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    int v = pg[k];
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int n = __shfl_up_sync(0xffffffffu, v, o);
                        if (lane >= o) v += n;
                    }
                    const int i = base + 32 * k + lane;
                    if (i < p.batch) pfx[i + 1] = carry + v;
                    carry += __shfl_sync(0xffffffffu, v, 31);
                }
            }
            if (lane == 0) pfx[0] = 0;
        }
    }
    if (!kDump && warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(&bars->tmem_base), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = kDump ? 0u : bars->tmem_base;
    const uint64_t lim_score = p.timeout_ns;       // the score warp's waits
    const uint64_t lim_dep = 2 * p.timeout_ns;     // the roles that depend on it
    const MmaWarpArgs margs{tmem, sbase, bars, p.status, smem, lim_score};

    if (!aligned_ok) {
        // nothing runs; the error is recorded
    } else if (warp == 0 || warp == 6) {
        // ------------------------------------------------------ TMA producers
        const uint32_t b_land = kFp8 ? (warp == 0 ? b_kstaged : b_vstaged)
                                     : (warp == 0 ? b_kfull : b_vfull);
        if (lane == 0)
            page_loader<kDump, kFp8>(p, &tmap, pfx, pair, rank, warp == 0, bars, smem, sbase,
                                     b_land, warp == 0 ? b_kempty : b_vempty, lim_dep);
    } else if (kDump) {
        // loader dump: only the loaders run
    } else if (kFp8 && warp >= 7) {
        // fp8 cache: warps 7-8 widen the K-ring blocks, 9-10 the value blocks
        if (warp < 9)
            page_converter<true>(p, pfx, pair, bars, smem, b_kstaged, b_kfull,
                                 (warp - 7) * 32 + lane, lim_dep);
        else
            page_converter<false>(p, pfx, pair, bars, smem, b_vstaged, b_vfull,
                                  (warp - 9) * 32 + lane, lim_dep);
    } else if (warp == 1) {
        // ------------------------------------------------------ score MMAs
        const uint32_t bq[7] = {b_kfull, b_kempty, b_vfull, b_sfull, b_pfree, b_qready, b_final_qk};
        if (rank == 0)
            score_warp<0, kFp8>(margs, bq, p, pfx, pair);
        else
            score_warp<1, kFp8>(margs, bq, p, pfx, pair);
    } else {
        // ------------------------------- softmax / P.V issue / correction / epilogue
        const int quarter = warp & 3;
        const int h = quarter * 32 + lane;
        const uint32_t trow = tmem + (uint32_t(quarter * 32) << 16);
        const bool live_head = h < N;
        const int shift = row_shift(p, h);   // multi-token rows: tokens past this row's end
        bool issued_pv = false;
        bool ok = true;
        // q of request qb, copied with coalesced 16-byte cp.async (a warp
        // copies whole rows): dims 0..255 first into the q area as a staging
        // copy (row r at 512 r, chunk c at (c ^ r % 32) * 16: conflict-free
        // row reads), from which each thread moves its own row to TMEM; then
        // dims 256..575 into the q area in the score MMAs' SW128 layout. Rows
        // of padded heads are zero-filled. Called once every score MMA that
        // read the previous q has completed. Returns false if a wait expired.
        int nstage = 0;
        bool q_big = false;   // fp8 cache: a q entry beyond the f16 range was seen
        auto stage_q = [&](int qb) -> bool {
            const uint16_t* qbase = p.q + size_t(io_row(p, qb)) * N * kD;
            const uint32_t ph = uint32_t(nstage++) & 1u;
            const int t = tid - 64;   // 0..127 over the four softmax warps
#pragma unroll 4
            for (int k = 0; k < 32; ++k) {
                const int i = t + 128 * k;   // 128 rows x 32 chunks
                const int r = i >> 5, c = i & 31;
                const bool live = r < N;
                ptx::cp_async16(sbase + uint32_t(kOffQS + r * 512 + ((c ^ (r & 31)) * 16)),
                                qbase + (live ? size_t(r) * kD + 8 * c : 0), live ? 16u : 0u);
            }
            ptx::cp_async_wait_all();
            ptx::mbar_arrive(b_qstaged);
            if (!wait_phase(b_qstaged, ph, bars, p.status, kSiteQReady, lim_dep)) return false;
#pragma unroll 1
            for (int blk = 0; blk < kQTmemBlocks; ++blk) {
                uint32_t r32[32];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int c = 8 * blk + i;
                    const uint4 v = *reinterpret_cast<const uint4*>(
                        smem + kOffQS + h * 512 + ((c ^ (h & 31)) * 16));
                    r32[4 * i + 0] = v.x;
                    r32[4 * i + 1] = v.y;
                    r32[4 * i + 2] = v.z;
                    r32[4 * i + 3] = v.w;
                }
                if constexpr (kFp8) {
                    // f16 operands: q widened exactly (bf16 -> f16)
#pragma unroll
                    for (int i = 0; i < 32; ++i) r32[i] = bf16x2_to_f16x2(r32[i], q_big);
                }
                ptx::tmem_st32(trow + kTmemQ + uint32_t(blk * 32), r32);
            }
            ptx::mbar_arrive(b_qread);
            if (!wait_phase(b_qread, ph, bars, p.status, kSiteQReady, lim_dep)) return false;
#pragma unroll 4
            for (int k = 0; k < 40; ++k) {
                const int i = t + 128 * k;   // 128 rows x 40 chunks (dims 256..575)
                const int r = i / 40, c = i - 40 * (i / 40);
                const int kb = c >> 3, cc = c & 7;
                const bool live = r < N;
                ptx::cp_async16(
                    sbase + uint32_t(kOffQS + kb * 16384 + r * 128 + ((cc ^ (r & 7)) * 16)),
                    qbase + (live ? size_t(r) * kD + 256 + 8 * c : 0), live ? 16u : 0u);
            }
            ptx::cp_async_wait_all();
            if constexpr (kFp8) {
                // Each thread widens the chunks it copied, in place.
#pragma unroll 4
                for (int k = 0; k < 40; ++k) {
                    const int i = t + 128 * k;
                    const int r = i / 40, c = i - 40 * (i / 40);
                    const int kb = c >> 3, cc = c & 7;
                    uint4* a = reinterpret_cast<uint4*>(smem + kOffQS + kb * 16384 + r * 128 +
                                                        ((cc ^ (r & 7)) * 16));
                    const uint4 v = *a;
                    *a = make_uint4(bf16x2_to_f16x2(v.x, q_big), bf16x2_to_f16x2(v.y, q_big),
                                    bf16x2_to_f16x2(v.z, q_big), bf16x2_to_f16x2(v.w, q_big));
                }
                if (q_big) record_error(p.status, MLA_ERR_RANGE, qb);
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(b_qready);
            return true;
        };
        SegmentWalk walk = walk_begin(p, pfx, pair);
        Segment sg, nx;
        bool have = walk_next(p, pfx, pair, walk, sg);
        int staged_b = -1;   // request whose q is staged
        if (have && seg_pages(sg) > 0) {
            ok = __all_sync(0xffffffffu, stage_q(sg.b));
            staged_b = sg.b;
        }
        int jg = 0;   // pages done so far, across segments
        while (ok && have) {
            const int ntiles = seg_pages(sg);
            // The next segment, looked up now so that its global loads are
            // done by the time this segment ends.
            const bool have_next = walk_next(p, pfx, pair, walk, nx);
            float m_ref = -INFINITY;   // log2 units
            float l_sum = 0.f;         // sum of fp32 weights (for the LSE)
            float l_bf = 0.f;          // sum of the bf16 weights the MMA used (for O)
            const int jg0 = jg;
            for (int j = 0; j < ntiles; ++j, ++jg) {
                const int sl = jg & 1;
                // Poll briefly before sleeping: the scores are usually a few
                // hundred cycles away and a poll wakes sooner than a
                // suspended thread.
                ok = false;
                for (int sp = 0; sp < kSoftmaxSpin && !ok; ++sp)
                    ok = ptx::mbar_test_wait(b_sfull + 8 * sl, uint32_t(jg >> 1) & 1u);
                if (!ok)
                    ok = wait_phase(b_sfull + 8 * sl, uint32_t(jg >> 1) & 1u, bars, p.status,
                                    kSiteSFull, lim_dep);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                ptx::tc_fence_after();
                // The page's 64 raw scores of this head. The scale (log2
                // units) is applied inside the weights' FMA below, so the
                // page maximum of the scaled scores is the scale times the
                // raw maximum (the raw minimum for a negative scale; the host
                // never passes 0). Tokens past the sequence end get the raw
                // score that scales to -inf.
                const uint32_t sbuf = trow + kTmemS + uint32_t(sl * 64);
                const int valid = min(kTile, sg.t_hi - (sg.t_lo + j * kTile));
                // This row's visible tokens on the page (fewer for an earlier
                // query token of a causal multi-token block; possibly none).
                const int valid_row =
                    shift == 0 ? valid
                               : min(valid, sg.L - shift - (sg.t_lo + j * kTile));
                const float sc = p.scale_log2;
                float x[64];
                {
                    uint32_t r[64];
                    ptx::tmem_ld64(sbuf, r);
#pragma unroll
                    for (int i = 0; i < 64; ++i) x[i] = __uint_as_float(r[i]);
                }
                if (valid_row < kTile) {
                    const float masked = sc > 0.f ? -INFINITY : INFINITY;
#pragma unroll
                    for (int i = 0; i < 64; ++i) x[i] = i < valid_row ? x[i] : masked;
                }
                float mx;
                if (sc > 0.f) {
                    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int i = 0; i < 64; i += 2)
                        m4[(i >> 1) & 3] = ptx::fmax3(m4[(i >> 1) & 3], x[i], x[i + 1]);
                    mx = ptx::fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
                } else {
                    float m4[4] = {INFINITY, INFINITY, INFINITY, INFINITY};
#pragma unroll
                    for (int i = 0; i < 64; i += 2)
                        m4[(i >> 1) & 3] = ptx::fmin3(m4[(i >> 1) & 3], x[i], x[i + 1]);
                    mx = ptx::fmin3(m4[0], m4[1], fminf(m4[2], m4[3]));
                }
                const float m_new = fmaxf(m_ref, mx * sc);
                const bool rescale = m_new > m_ref + kRescaleThreshold;
                float alpha = 1.f;
                if (rescale) {
                    alpha = ptx::ex2(m_ref - m_new);
                    m_ref = m_new;
                }

                // Weights: P row of this head, 64 tokens as bf16 pairs, written
                // over the first 32 columns of the score buffer (all read
                // above). Masked tokens (x = -inf) get 0.
                // The weights go to TMEM first; their two sums are formed
                // after the P.V hand-off below, off the path from these
                // scores to the MMA that frees their buffer (x keeps the
                // fp32 weights, pk the rounded ones).
                uint32_t pk[32];
                {
                    // A row that has seen no token yet keeps m_ref = -inf:
                    // its weights are exp2(-inf) = 0, not NaN.
                    const float mneg = m_ref == -INFINITY ? 0.f : -m_ref;
                    const float2 negm2 = make_float2(mneg, mneg);
                    const float2 sc2 = make_float2(sc, sc);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float2 d = __ffma2_rn(make_float2(x[2 * i], x[2 * i + 1]), sc2, negm2);
                        x[2 * i] = ptx::ex2(d.x);
                        x[2 * i + 1] = ptx::ex2(d.y);
                        pk[i] = kFp8 ? pack_f16x2(x[2 * i], x[2 * i + 1])
                                     : pack_bf16x2(x[2 * i], x[2 * i + 1]);
                    }
                    ptx::tmem_st32(sbuf, pk);
                }

                // O rescale once the P.V of the previous page is done.
                if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
                    ok = wait_phase(b_pfree + 8 * ((jg - 1) & 1), uint32_t((jg - 1) >> 1) & 1u, bars,
                                    p.status, kSitePvDone, lim_dep);
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
                // Rows past the sequence end in the last page may hold anything
                // (even NaN): zero their value columns so that 0 * V stays 0.
                if (valid < kTile) {
                    unsigned char* vs = smem + kOffV + sl * kVBytes;
                    const int rows = kTile - valid;
                    for (int idx = h; idx < rows * 32; idx += 128) {
                        const int row = valid + idx / 32;
                        const int blk = (idx / 8) & 3;
                        const int ch = idx & 7;
                        *reinterpret_cast<uint4*>(vs + blk * kBlockBytes + row * 128 + ch * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    ptx::fence_proxy_async_smem();
                }
                // The fourth softmax warp to finish page jg issues its P.V MMAs
                // (the first page of a segment starts O afresh).
                ptx::tc_fence_before();
                __syncwarp();
                uint32_t done_before = 0;
                if (lane == 0) done_before = ptx::atom_add_acq_rel_shared(a_pcount + 4 * sl, 1u);
                done_before = __shfl_sync(0xffffffffu, done_before, 0);
                if (done_before == 4u * uint32_t(jg >> 1) + 3u) {
                    ptx::tc_fence_after();
                    if (ptx::elect_one())
                        issue_pv<kFp8>(tmem, sbase, jg, j > 0, b_vempty, b_pfree);
                    __syncwarp();
                    issued_pv = true;
                }
                {
                    float2 ls2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                    float2 lb2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        ls2[i & 1] = __fadd2_rn(ls2[i & 1], make_float2(x[2 * i], x[2 * i + 1]));
                        lb2[i & 1] = __fadd2_rn(lb2[i & 1], unpack_x2<kFp8>(pk[i]));
                    }
                    const float2 ls = __fadd2_rn(ls2[0], ls2[1]);
                    const float2 lb = __fadd2_rn(lb2[0], lb2[1]);
                    l_sum = l_sum * alpha + (ls.x + ls.y);
                    l_bf = l_bf * alpha + (lb.x + lb.y);
                }
            }
            if (!ok) break;

            // q of the next segment goes in now, ahead of this epilogue: the
            // score MMAs of this segment (the only readers of q) are complete
            // (this warp saw their last s_full), and the score warp can start
            // the next segment while the output is written.
            if (have_next && seg_pages(nx) > 0 && nx.b != staged_b) {
                ok = __all_sync(0xffffffffu, stage_q(nx.b));
                if (!ok) break;
                staged_b = nx.b;
            }

            // Epilogue: O / l -> bf16 output, or the fp32 partial row.
            if (ntiles > 0) {
                // The commit after the segment's last P.V covers every
                // earlier one too.
                const int jl = jg0 + ntiles - 1;
                ok = wait_phase(b_pfree + 8 * (jl & 1), uint32_t(jl >> 1) & 1u, bars, p.status,
                                kSitePvDone, lim_dep);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                ptx::tc_fence_after();
            }
            float inv = l_bf > 0.f ? 1.f / l_bf : 0.f;
            if constexpr (kFp8) inv *= p.v_scale;   // the cache codes' per-tensor scale
            const float lse = l_sum > 0.f ? (m_ref + log2f(l_sum)) * kLn2 : -INFINITY;
            const size_t row = size_t(io_row(p, sg.b)) * N + h;
            const bool out32 = (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0u;
            const size_t prow = size_t(sg.prow0) + size_t(h) * sg.prow_stride;
            // An empty split's partial row is never read (its LSE of -inf
            // gives it weight 0 in the merge): only its LSE is written.
            const int cend = (ntiles == 0 && sg.prow0 >= 0) ? 0 : 256;
#pragma unroll 1
            for (int c = 0; c < cend; c += 32) {
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
                } else if (sg.prow0 < 0) {
                    // bf16 row: 32-byte stores when `out` allows them.
                    uint16_t* dst = p.out + row * kLkv + col;
                    uint32_t v[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        v[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv,
                                           __uint_as_float(o[2 * i + 1]) * inv);
                    if (out32) {
                        ptx::st_global_v8(dst, *reinterpret_cast<const uint32_t(*)[8]>(v));
                        ptx::st_global_v8(dst + 16, *reinterpret_cast<const uint32_t(*)[8]>(v + 8));
                    } else {
                        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            d4[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                    }
                } else if (p.part_bf16) {
                    // bf16 split partial row (workspace rows 1 KB apart).
                    uint16_t* dst = reinterpret_cast<uint16_t*>(p.o_part) + prow * kLkv + col;
                    uint32_t v[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        v[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv,
                                           __uint_as_float(o[2 * i + 1]) * inv);
                    ptx::st_global_v8(dst, *reinterpret_cast<const uint32_t(*)[8]>(v));
                    ptx::st_global_v8(dst + 16, *reinterpret_cast<const uint32_t(*)[8]>(v + 8));
                } else {
                    // fp32 partial row (workspace: 256-byte aligned rows).
                    float* dst = p.o_part + prow * kLkv + col;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint32_t v[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            v[k] = __float_as_uint(__uint_as_float(o[8 * i + k]) * inv);
                        ptx::st_global_v8(dst + 8 * i, v);
                    }
                }
            }
            if (rank == 0 && live_head) {
                if (sg.prow0 < 0) {
                    if (p.lse != nullptr) p.lse[row] = lse;
                } else {
                    p.lse_part[prow] = lse;
                }
            }
            if (p.sched_pairs > 0 && sg.prow0 >= 0) {
                // This warp's part of a partial row set is written: count it
                // for the merge, which may already be running on SMs that
                // other CTAs have left (it waits for kPieceArrivals per piece).
                __threadfence();
                __syncwarp();
                if (lane == 0) atomicAdd(p.counters + kReadyWord + sg.b, 1);
            }
            // The next segment's first P.V overwrites O: every softmax warp
            // has read it by then, since that P.V waits for all four warps
            // to finish the segment's first page, which comes after this.
            sg = nx;
            have = have_next;
        }
        // Every P.V MMA this warp issued completes before TMEM is freed.
        if (issued_pv) warp_drain(b_final_sm + 8 * quarter, margs);
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (!kDump && warp == 1) ptx::tmem_dealloc(tmem, kTmemCols);
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

namespace {

template <bool kDump, bool kFp8>
int launch_tc(const DecodeParams& p, int grid_ctas, void* stream) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = get_encoder();
    if (encode == nullptr) return int(cudaErrorNotSupported);
    // The cache viewed as [num_blocks * 64, 576]: bf16 with 128-byte swizzled
    // 64 x 64 boxes, or E4M3 codes with unswizzled 64 x 64 one-byte boxes.
    CUtensorMap tmap;
    const cuuint64_t dims[2] = {cuuint64_t(kD), cuuint64_t(p.num_blocks) * kTile};
    const cuuint64_t strides[1] = {cuuint64_t(kD) * (kFp8 ? 1 : 2)};
    const cuuint32_t box[2] = {64, kTile};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(&tmap,
                        kFp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                        const_cast<uint16_t*>(p.cache), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        kFp8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return int(cudaErrorInvalidValue);
    cudaError_t e = cudaFuncSetAttribute(mla_decode_tc_kernel<kDump, kFp8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return int(e);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid_ctas), 1, 1);
    cfg.blockDim = dim3(kFp8 ? kThreadsFp8 : kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;   // the two CTAs of an item run together
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, mla_decode_tc_kernel<kDump, kFp8>, p, tmap);
    return int(e);
}

}  // namespace

int launch_decode_tc(const DecodeParams& p, int grid_ctas, void* stream) {
    return launch_tc<false, false>(p, grid_ctas, stream);
}

int launch_decode_tc_loader_dump(const DecodeParams& p, int grid_ctas, void* stream) {
    return launch_tc<true, false>(p, grid_ctas, stream);
}

int launch_decode_tc_fp8(const DecodeParams& p, int grid_ctas, void* stream) {
    return launch_tc<false, true>(p, grid_ctas, stream);
}

}  // namespace mla
