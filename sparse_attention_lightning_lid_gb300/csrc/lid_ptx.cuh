// lid_ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarrier, TMA,
// tcgen05 (tensor-memory allocation, MMA, commit, loads) and named barriers.
// Every wait on an mbarrier is bounded: it gives up after about a second of
// SM clock, records an error code and sets a CTA-wide abort flag.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lid {

// Device-side error word, read by lid_device_error(). Each translation unit
// that includes this header (lid_api.cu, lid_attn.cu) is its own device
// module with its own copy; lid_device_error reads both.
__device__ int g_dev_error = 0;

constexpr long long kWaitLimitCycles = 1ll << 31;  // default limit of a wait: ~1 s at 2 GHz

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// A waiting thread may be suspended until the phase completes, for at most
// this long per try (so the bounded waits below still check their limit):
// it then takes no issue slots from the warps that do the work.
constexpr uint32_t kSuspendHintNs = 20000;

__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(addr), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of `bar` to complete. Returns false (and sets the
// abort flag and the device error word) if it has not after `limit` cycles,
// or if another role of the CTA already aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int err_code,
                                          long long limit = kWaitLimitCycles) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(a, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort_flag) return false;
            if (clock64() - t0 > limit) {
                *abort_flag = 1;
                atomicCAS(&g_dev_error, 0, err_code);
                return false;
            }
        }
    }
}

// -------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 2D tiled load of one box into shared memory, completing tx bytes on `bar`.
// x is the innermost coordinate in elements; the caller keeps x * 2 bytes a
// multiple of 16.
__device__ __forceinline__ void tma_load_2d(void *dst, const void *tmap, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// 1D bulk copy global -> shared (both 16-byte aligned, bytes a multiple of 16),
// completing tx bytes on `bar`.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (f16 or bf16 in, f32 accumulate)
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Same with 8-bit operands (kind::f8f6f4; the instruction descriptor names
// both as E4M3), K = 32 per instruction.
__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Four MMAs over one 128-byte column chunk of a K-major 128-byte-swizzled
// pair of operands: K steps at 0, 32, 64 and 96 bytes into the rows (the
// descriptors' address field advances by 2 per 32 bytes). The first MMA
// accumulates only if first_acc != 0, the other three always. One asm block,
// so the issuing thread spends as few instructions as possible per MMA: the
// warp shares its scheduler with the busy epilogue warps, and each issue slot
// it waits for leaves the tensor pipe idle.
// (STEP: the descriptors' advance from one MMA to the next, in 16-byte units:
// 2 for the next 32 bytes of a K-major row; other layouts pass their own.)
template <bool F8, int STEP = 2>
__device__ __forceinline__ void umma_quad(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t first_acc) {
    if constexpr (F8) {
        asm volatile(
            "{\n\t.reg .pred p, q;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
            "setp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 q, %3, %3;\n\t"
            "add.s64 a1, %1, %5;\n\tadd.s64 b1, %2, %5;\n\t"
            "add.s64 a2, %1, %6;\n\tadd.s64 b2, %2, %6;\n\t"
            "add.s64 a3, %1, %7;\n\tadd.s64 b3, %2, %7;\n\t"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a1, b1, %3, q;\n\t"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a2, b2, %3, q;\n\t"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a3, b3, %3, q;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(first_acc), "n"(STEP), "n"(2 * STEP), "n"(3 * STEP)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p, q;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
            "setp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 q, %3, %3;\n\t"
            "add.s64 a1, %1, %5;\n\tadd.s64 b1, %2, %5;\n\t"
            "add.s64 a2, %1, %6;\n\tadd.s64 b2, %2, %6;\n\t"
            "add.s64 a3, %1, %7;\n\tadd.s64 b3, %2, %7;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, q;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, q;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, q;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(first_acc), "n"(STEP), "n"(2 * STEP), "n"(3 * STEP)
            : "memory");
    }
}

// Arrive once on `bar` when every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// The same wait, naming the registers of the load it completes as in/out
// operands: their uses cannot be scheduled above it.
__device__ __forceinline__ void tmem_wait_ld_dep8(uint32_t *r) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7])
                 :
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_ld_dep16(uint32_t *r) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15])
                 :
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_ld_dep32(uint32_t *r) {
    tmem_wait_ld_dep16(r);
    asm volatile(""
                 : "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]),
                   "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}
template <int W>
__device__ __forceinline__ void tmem_wait_ld_dep(uint32_t *r) {
    static_assert(W == 8 || W == 16 || W == 32, "8, 16 or 32 registers");
    if constexpr (W == 8) tmem_wait_ld_dep8(r);
    else if constexpr (W == 16) tmem_wait_ld_dep16(r);
    else tmem_wait_ld_dep32(r);
}

// 32 lanes x 32 bits, N consecutive columns: thread i of the warp gets lane
// (base lane + i), columns [col, col + N).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t *r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

template <int W>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t *r) {
    if constexpr (W == 8) tmem_ld8(taddr, r);
    else if constexpr (W == 16) tmem_ld16(taddr, r);
    else tmem_ld32(taddr, r);
}

// Shared-memory matrix descriptor for a K-major operand stored as 128-byte
// rows with the 128-byte swizzle (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B): 8-row atoms of 1024 bytes, so the stride
// between row groups is 1024 bytes; the leading offset is unused for this
// layout; bits 46-47 carry the descriptor version 1; bits 61-63 = 2 select
// the 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;             // leading byte offset 16 B (ignored)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;     // stride byte offset
    d |= static_cast<uint64_t>(1) << 46;             // version
    d |= static_cast<uint64_t>(2) << 61;             // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16 or kind::f8f6f4, f32 accumulator, both
// operands K-major. ab_format: kind::f16: 0 = f16, 1 = bf16; kind::f8f6f4:
// 0 = E4M3.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, int ab_format) {
    return (1u << 4)                                   // D format f32
           | (static_cast<uint32_t>(ab_format) << 7)   // A format
           | (static_cast<uint32_t>(ab_format) << 10)  // B format
           | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// ------------------------------------------------------ packed f32 pairs
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ float sum_f32x2(uint64_t v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return lo + hi;
}

// two independent fp32 fused multiply-adds (round to nearest) in one instruction
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// --------------------------------------------------------- named barriers
__device__ __forceinline__ void named_bar(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Barrier that also returns, to every participating thread, the OR of `pred`
// over all of them (so a decision taken on it is uniform across the group).
__device__ __forceinline__ bool named_bar_or(int id, int nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

}  // namespace lid
