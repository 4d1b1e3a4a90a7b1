// sm100.cuh -- thin inline-PTX wrappers for the Blackwell (sm_100 family, built for
// sm_103a) features the tensor-core kernels use: tcgen05 MMA / tensor memory, mbarriers,
// TMA bulk and tensor copies, cp.async, and bounded waits that report instead of hanging.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "internal.cuh"

namespace lsh {
namespace sm100 {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// ------------------------------------------------------------------ descriptors

// Shared-memory matrix descriptor of tcgen05.mma.  `addr` is a shared-window byte
// address; lbo/sbo are byte strides (leading / stride dimension); swizzle 2 = 128-byte
// swizzle.  Bits 46-47 hold the descriptor version (1 on sm_100).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swizzle = 2) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFF) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)swizzle << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma.kind::f16: bf16 x bf16 -> fp32, M x N, with the
// A / B operands K-major (0) or MN-major (1).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// The same for kind::f16 with fp16 A and B (operand format fields 0 instead of 1); the
// two operands always share one type.
__host__ __device__ constexpr uint32_t idesc_16(int M, int N, int a_mn, int b_mn, bool f16) {
    return f16 ? (idesc_bf16(M, N, a_mn, b_mn) & ~((1u << 7) | (1u << 10)))
               : idesc_bf16(M, N, a_mn, b_mn);
}

// Byte offset of element (row, k) of a K-major tile with 128-byte swizzle: 64 bf16 of K
// per 128-byte row, blocks of `rows` rows per 64-wide K block, 8-row atoms of 1 KB.
__host__ __device__ __forceinline__ uint32_t kmajor_sw128_off(int row, int k, int rows) {
    const int kb = k >> 6, kk = k & 63;
    return (uint32_t)(kb * rows * 128 + row * 128 + ((((kk >> 3) ^ (row & 7))) << 4) + (kk & 7) * 2);
}

// ------------------------------------------------------------------ tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// MMA issue.  Every wrapper below is executed by a whole, converged warp: one lane is
// elected inside the instruction sequence and issues.  (Issuing from a lane-divergent
// branch instead, e.g. under `if (lane == 0)`, measured about half the issue rate on
// sm_103a: ~256 cycles per M=128 instruction against ~123 from a converged warp, which
// reaches the full dense bf16 rate at N=256.)
//
// D (tmem) (+)= A (smem) * B (smem)
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p, e;\n\t.reg .b32 r;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "elect.sync r|e, 0xffffffff;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}
// D (tmem) (+)= A (tmem, packed 16-bit pairs) * B (smem)
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p, e;\n\t.reg .b32 r;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "elect.sync r|e, 0xffffffff;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}
// Arrive once on an mbarrier when every tcgen05 op the warp's elected lane issued so far
// completes (whole warp; the elected lane is the one that issued the MMAs).
__device__ __forceinline__ void mma_commit(uint32_t mbar) {
    asm volatile("{\n\t.reg .pred e;\n\t.reg .b32 r;\n\telect.sync r|e, 0xffffffff;\n\t"
                 "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
                 :: "r"(mbar) : "memory");
}

#define LSH_R32(p) "=r"(p[0]), "=r"(p[1]), "=r"(p[2]), "=r"(p[3]), "=r"(p[4]), "=r"(p[5]), \
    "=r"(p[6]), "=r"(p[7]), "=r"(p[8]), "=r"(p[9]), "=r"(p[10]), "=r"(p[11]), "=r"(p[12]), \
    "=r"(p[13]), "=r"(p[14]), "=r"(p[15]), "=r"(p[16]), "=r"(p[17]), "=r"(p[18]), "=r"(p[19]), \
    "=r"(p[20]), "=r"(p[21]), "=r"(p[22]), "=r"(p[23]), "=r"(p[24]), "=r"(p[25]), "=r"(p[26]), \
    "=r"(p[27]), "=r"(p[28]), "=r"(p[29]), "=r"(p[30]), "=r"(p[31])

// 32 consecutive fp32 columns of this thread's tensor-memory lane (warp-collective).
// Completion needs tmem_wait_ld().
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,"
                 "%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31},"
                 " [%32];"
                 : LSH_R32(r) : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
#define LSH_RW32(p) "+r"(p[0]), "+r"(p[1]), "+r"(p[2]), "+r"(p[3]), "+r"(p[4]), "+r"(p[5]), \
    "+r"(p[6]), "+r"(p[7]), "+r"(p[8]), "+r"(p[9]), "+r"(p[10]), "+r"(p[11]), "+r"(p[12]), \
    "+r"(p[13]), "+r"(p[14]), "+r"(p[15]), "+r"(p[16]), "+r"(p[17]), "+r"(p[18]), "+r"(p[19]), \
    "+r"(p[20]), "+r"(p[21]), "+r"(p[22]), "+r"(p[23]), "+r"(p[24]), "+r"(p[25]), "+r"(p[26]), \
    "+r"(p[27]), "+r"(p[28]), "+r"(p[29]), "+r"(p[30]), "+r"(p[31])
// tcgen05.wait::ld that also ties the destination registers of the loads it waits for:
// the compiler sees them as written here, so no use of them is scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" : LSH_RW32(r) :: "memory");
}
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32], uint32_t (&s)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" : LSH_RW32(r) :: "memory");
    asm volatile("" : LSH_RW32(s) :: "memory");
}
// 16 consecutive fp32 columns of this thread's lane (warp-collective); completion needs
// tmem_wait_ld16 (or any tcgen05.wait::ld).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,"
                 "%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
}
// tcgen05.wait::ld that ties the 16 destination registers (no use moves above it).
__device__ __forceinline__ void tmem_wait_ld16(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]) :: "memory");
}
// Ties 16 registers filled by a tcgen05.ld already waited for (by a wait that tied
// other registers): no use of them moves above this point.
__device__ __forceinline__ void tmem_tie16(uint32_t (&r)[16]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]) :: "memory");
}
// 8 consecutive 32-bit columns into this thread's lane.  Completion needs tmem_wait_st().
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
                    "r"(r[6]), "r"(r[7]) : "memory");
}
// 16 consecutive 32-bit columns into this thread's lane.  Completion needs tmem_wait_st().
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,"
                 "%11,%12,%13,%14,%15,%16};"
                 :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
                    "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
                    "r"(r[13]), "r"(r[14]), "r"(r[15]) : "memory");
}
// 16 zero columns into this thread's lane.
__device__ __forceinline__ void tmem_st16_zero(uint32_t taddr) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,"
                 "%1,%1,%1,%1,%1,%1};" :: "r"(taddr), "r"(0u) : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ mbarriers

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
// try_wait with a suspend-time hint: a thread whose phase is not complete yet is parked
// (up to `ns` nanoseconds, woken when the phase completes) instead of re-polling, so
// waiting roles do not take issue slots from the warps doing the arithmetic.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity), "r"(ns) : "memory");
    return ok != 0;
}
// Arrive on `bar` once all cp.async copies this thread issued so far have landed.
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait.  Every wait in the tensor-core kernels goes through this: after
// kWaitLimitNs without progress (or as soon as another role of the CTA gave up), it
// records `where` in the workspace status block, raises the CTA's abort flag and returns
// false, so the kernel winds down instead of hanging.
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s; legitimate waits are microseconds

__device__ __forceinline__ void report(StatusBlock *st, volatile int *abort_flag, int where) {
    *abort_flag = 1;
    if (st && atomicCAS(&st->code, 0, 1) == 0) st->detail = where;
}

#ifdef LSH_WAIT_PROF
// Profiling build only: cycles spent in each wait, summed over threads, by wait code.
extern __device__ unsigned long long g_wait_cycles[4096];
extern __device__ unsigned long long g_wait_count[4096];
#endif

// Profiling build only: time spans inside compute loops (summed per warp by lane 0).
#ifdef LSH_WAIT_PROF
#define LSH_SPAN_BEGIN(v) const long long v = clock64()
#define LSH_SPAN_END(v, code)                                                          \
    do {                                                                               \
        if ((threadIdx.x & 31) == 0) {                                                 \
            atomicAdd(&::lsh::sm100::g_wait_cycles[(code) & 4095],                     \
                      (unsigned long long)(clock64() - (v)));                          \
            atomicAdd(&::lsh::sm100::g_wait_count[(code) & 4095], 1ull);               \
        }                                                                              \
    } while (0)
#else
#define LSH_SPAN_BEGIN(v) do {} while (0)
#define LSH_SPAN_END(v, code) do {} while (0)
#endif

static __device__ __noinline__ bool wait_impl(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                       StatusBlock *st, int where) {
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_sleep(bar, parity, 20000)) return true;
        if ((it & 7) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > kWaitLimitNs) {
                report(st, abort_flag, where);
                return false;
            }
        }
    }
}

static __device__ __forceinline__ bool wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                            StatusBlock *st, int where) {
#ifdef LSH_WAIT_PROF
    const long long c0 = clock64();
    const bool ok = mbar_try_wait(bar, parity) || wait_impl(bar, parity, abort_flag, st, where);
    if ((threadIdx.x & 31) == 0) {
        atomicAdd(&g_wait_cycles[where & 4095], (unsigned long long)(clock64() - c0));
        atomicAdd(&g_wait_count[where & 4095], 1ull);
    }
    return ok;
#else
    // Fast path inline: a phase that is already complete costs no call (a call would
    // also make the caller's loads in flight land before it).
    if (mbar_try_wait(bar, parity)) return true;
    return wait_impl(bar, parity, abort_flag, st, where);
#endif
}

// Bounded wait by a whole warp, with a warp-uniform answer (false if any lane gave up).
static __device__ __forceinline__ bool wait_w(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                              StatusBlock *st, int where) {
    return __all_sync(0xffffffffu, wait(bar, parity, abort_flag, st, where));
}

// ------------------------------------------------------------------ copies

// 1-D bulk copy global -> shared, completing `bytes` transactions on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
// 2-D tensor-map tile copy global -> shared (coordinates: x = innermost element, y = row).
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3}], [%4];"
                 :: "r"(smem_u32(dst)), "l"((uint64_t)map), "r"(x), "r"(y), "r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" :: "l"((uint64_t)map) : "memory");
}
// 16-byte asynchronous copy global -> shared (L2 only, bypassing L1).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(dst), "l"(src) : "memory");
}
// 4-byte asynchronous copy global -> shared (both 4-byte aligned).
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(threads) : "memory");
}

}  // namespace sm100

// Host side: encode a 2-D bf16 tensor map (rows x cols, row-major) with a box of
// box_cols x box_rows and 128-byte swizzle.  Returns false when the driver entry point
// is unavailable or the encoding fails.
bool make_tmap_2d_bf16(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                       uint32_t box_cols, uint32_t box_rows);

}  // namespace lsh
