// Inline-PTX wrappers for the sm_103a tensor-core decode kernel: mbarriers,
// cluster shared memory, TMA tile loads, and tcgen05 (TMEM allocation, MMA,
// commit, TMEM loads/stores). Each wrapper is one documented PTX instruction
// (or a load/store immediately followed by its wait).
#pragma once

#include <cstdint>

namespace mla {
namespace ptx {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// 16-byte global -> shared copy, bypassing L1; reads src_bytes (0 or 16) and
// zero-fills the rest. Completed by cp_async_wait_all.
__device__ __forceinline__ void cp_async16(uint32_t dst_smem, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst_smem), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Hint: pull `bytes` (a multiple of 16) at `p` (16-byte aligned) into L2.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Acquire-release add on a shared-memory word (CTA scope); returns the old
// value. Orders the caller's earlier writes (and, with tcgen05 fences around
// it, its TMEM stores) before a later acquirer's reads.
__device__ __forceinline__ uint32_t atom_add_acq_rel_shared(uint32_t addr, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "r"(addr), "r"(v)
                 : "memory");
    return old;
}

// One active lane of a converged warp (the same lane each time for the same
// set of active lanes). tcgen05.mma issued under this predicate keeps its
// operands in the warp-uniform datapath.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile(
        "{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(pred));
    return pred != 0;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Non-blocking test of a phase.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Same, but the thread may sleep in hardware for up to `suspend_ns` while
// the phase is pending (it wakes as soon as the phase completes).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t suspend_ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(suspend_ns)
        : "memory");
    return ok != 0;
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int32_t x, int32_t y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// 32-byte global store (the address must be 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* dst, const uint32_t (&v)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(v[0]),
                 "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Four MMAs into one accumulator, the first with accumulate flag acc0 and
// the others accumulating (A from TMEM at a0..a3, or from shared memory
// through descriptors a0..a3; B descriptors b0..b3).
__device__ __forceinline__ void mma4_ts(uint32_t d, uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint64_t b0, uint64_t b1, uint64_t b2,
                                        uint64_t b3, uint32_t idesc, uint32_t acc0) {
    asm volatile(
        "{\n .reg .pred p;\n"
        " setp.ne.b32 p, %9, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %5, %8, p;\n"
        " setp.eq.b32 p, %9, %9;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %6, %8, p;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %7, %8, p;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], %10, %8, p;\n}\n"
        ::"r"(d), "r"(a0), "r"(a1), "r"(a2), "r"(a3), "l"(b0), "l"(b1), "l"(b2), "r"(idesc),
          "r"(acc0), "l"(b3)
        : "memory");
}

__device__ __forceinline__ void mma4_ss(uint32_t d, uint64_t a0, uint64_t a1, uint64_t a2,
                                        uint64_t a3, uint64_t b0, uint64_t b1, uint64_t b2,
                                        uint64_t b3, uint32_t idesc, uint32_t acc0) {
    asm volatile(
        "{\n .reg .pred p;\n"
        " setp.ne.b32 p, %9, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %5, %8, p;\n"
        " setp.eq.b32 p, %9, %9;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %6, %8, p;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %7, %8, p;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %10, %8, p;\n}\n"
        ::"r"(d), "l"(a0), "l"(a1), "l"(a2), "l"(a3), "l"(b0), "l"(b1), "l"(b2), "r"(idesc),
          "r"(acc0), "l"(b3)
        : "memory");
}

// Four MMAs into one accumulator (A from TMEM at a0..a3, or from shared
// memory through descriptors a0..a3; B descriptors b0..b3), the first with
// accumulate flag acc0, the others accumulating; an mbarrier phase is tested
// before the first and the answer read after the fourth, so the test's
// latency passes while the MMAs issue. Returns 1 if the phase with `parity`
// has completed.
__device__ __forceinline__ uint32_t mma4_ts_probe(uint32_t d, uint32_t a0, uint32_t a1, uint32_t a2,
                                                  uint32_t a3, uint64_t b0, uint64_t b1, uint64_t b2,
                                                  uint64_t b3, uint32_t idesc, uint32_t acc0,
                                                  uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p, q;\n"
        " mbarrier.test_wait.parity.shared::cta.b64 q, [%11], %12;\n"
        " setp.ne.b32 p, %10, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%1], [%2], %6, %9, p;\n"
        " setp.eq.b32 p, %10, %10;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%1], [%3], %7, %9, p;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%1], [%4], %8, %9, p;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%1], [%5], %13, %9, p;\n"
        " selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(done)
        : "r"(d), "r"(a0), "r"(a1), "r"(a2), "r"(a3), "l"(b0), "l"(b1), "l"(b2), "r"(idesc),
          "r"(acc0), "r"(bar), "r"(parity), "l"(b3)
        : "memory");
    return done;
}

__device__ __forceinline__ uint32_t mma4_ss_probe(uint32_t d, uint64_t a0, uint64_t a1, uint64_t a2,
                                                  uint64_t a3, uint64_t b0, uint64_t b1, uint64_t b2,
                                                  uint64_t b3, uint32_t idesc, uint32_t acc0,
                                                  uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p, q;\n"
        " mbarrier.test_wait.parity.shared::cta.b64 q, [%11], %12;\n"
        " setp.ne.b32 p, %10, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%1], %2, %6, %9, p;\n"
        " setp.eq.b32 p, %10, %10;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%1], %3, %7, %9, p;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%1], %4, %8, %9, p;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%1], %5, %13, %9, p;\n"
        " selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(done)
        : "r"(d), "l"(a0), "l"(a1), "l"(a2), "l"(a3), "l"(b0), "l"(b1), "l"(b2), "r"(idesc),
          "r"(acc0), "r"(bar), "r"(parity), "l"(b3)
        : "memory");
    return done;
}

// Arrive once on a local mbarrier when every prior tcgen05 op of this thread completes.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns; thread i of the warp gets lane
// (base lane + i). Waits for the load before returning.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns from registers; waits for the store.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// 32 lanes x 64 consecutive 32-bit columns; thread i of the warp gets lane
// (base lane + i). Waits for the load before returning.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr)
        : "memory");
}

// Maximum / minimum of three floats in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float fmin3(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ------------------------------------------------------- UMMA descriptors

// Shared-memory matrix descriptor (version 1) for a 128-byte-swizzled layout.
//   K-major operand: 8-row groups of 128-byte rows, `sbo` bytes apart.
//   MN-major operand: `lbo` = byte stride between 64-element column blocks,
//                     `sbo` = byte stride between 8-row groups along K.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= uint64_t((saddr & 0x3FFFFu) >> 4);
    d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
    d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
    d |= uint64_t(1) << 46;
    d |= uint64_t(2) << 61;   // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B, M = 128.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int n, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           (uint32_t(n >> 3) << 17) | (uint32_t(128 >> 4) << 24);
}

// The same with f16 A and B (format field 0 for both operands).
__host__ __device__ constexpr uint32_t idesc_f16_f32(int n, bool b_mn_major) {
    return (1u << 4) | ((b_mn_major ? 1u : 0u) << 16) | (uint32_t(n >> 3) << 17) |
           (uint32_t(128 >> 4) << 24);
}

// Named barrier over `count` threads (a multiple of 32) of the CTA.
__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// The same barrier, returning the OR of `v` over the `count` threads (one
// answer for all of them).
__device__ __forceinline__ bool named_barrier_or(uint32_t id, uint32_t count, bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %3, 0;\n"
        " bar.red.or.pred q, %1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"(id), "r"(count), "r"(v ? 1u : 0u)
        : "memory");
    return r != 0;
}

}  // namespace ptx
}  // namespace mla
