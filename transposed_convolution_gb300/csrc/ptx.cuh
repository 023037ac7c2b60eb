// ptx.cuh -- inline-PTX wrappers for sm_103a: mbarriers, TMA tile loads, tcgen05
// (TMEM allocation, MMA, commit, loads) and the shared-memory matrix descriptors.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace ctr {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint: a thread whose phase is not yet complete may sleep up
// to hint_ns (waking as soon as the phase completes) instead of returning at once, so a
// waiting role spends few issue slots while others work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity,
                                                    uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Suspend-time hint of the bounded waits (nanoseconds): long against the time a phase
// takes to complete, short against any wait limit.
constexpr uint32_t kWaitHintNs = 20000;

// Wait until the phase of `bar` with the given parity has completed.  Bounded: gives up
// once limit_ns nanoseconds of global time have passed (at once when limit_ns is 0 and the
// phase is not complete on the first poll), or as soon as *abort becomes non-zero (abort
// may be null).  Returns true when the phase completed.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                          const volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    if (limit_ns == 0) return false;
    const uint64_t t0 = globaltimer_ns();
    const uint32_t hint = limit_ns < kWaitHintNs ? (uint32_t)limit_ns : kWaitHintNs;
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, hint)) return true;
        if (abort && *abort) return false;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// ---------------------------------------------------------------- warp-wide issue loops
// A role that issues tcgen05 instructions runs its loop on all 32 lanes of its warp, so that
// every value the loop computes (stage, descriptors, TMEM addresses) is warp-uniform, and one
// lane picked by elect.sync issues each instruction.  Measured on GB300 with streaming
// operands: about 74 cycles per 128x128x16 bf16 MMA this way against about 95 when lane 0
// alone runs the loop.  Every lane must reach each elect_one() of the loop (no lane-dependent
// exits), which the warp-wide wait and abort test below keep true.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b32 l;\n\t"
        "elect.sync l|p, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

// mbar_wait run by every lane of a warp; true on all lanes only when it succeeded on all.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                               const volatile int *abort) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, limit_ns, abort));
}

// *abort as seen by any lane of the warp (the same answer on every lane).
__device__ __forceinline__ bool abort_warp(const volatile int *abort) {
    return __any_sync(0xffffffffu, *abort != 0);
}

// ---------------------------------------------------------------- programmatic dependent launch
// Wait until the grids this one depends on (the previous kernels of the stream, when this one
// was launched with programmatic stream serialization) have completed and their memory is
// visible; a no-op otherwise.  Every kernel calls it before its first global memory access.
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Let the next kernel of the stream be scheduled now (it still waits for this grid's
// completion before touching memory).
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load of one box into shared memory, completing on `bar` (complete_tx bytes).
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
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

// D[tmem] (+)= A[smem] * B[smem]^T, cta_group::1.  kind::f16 (bf16 or fp16 operands, both the
// same) or kind::tf32.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far completes.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 TMEM lanes x 32 consecutive 32-bit columns: thread i of the warp receives lane
// (taddr.lane + i), columns taddr.col .. taddr.col + 31.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
        "[%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
          "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
          "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
          "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
          "=r"(v[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// The same wait, with the registers of the load it completes as in/out operands: the
// compiler then cannot move any use of them above the wait (a plain wait has no register
// dependence on the load).  Used when another load is still in flight while earlier values
// are consumed.
__device__ __forceinline__ void tmem_wait_ld_regs(uint32_t (&v)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]),
                   "+r"(v[6]), "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]),
                   "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15]), "+r"(v[16]),
                   "+r"(v[17]), "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]),
                   "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]), "+r"(v[26]),
                   "+r"(v[27]), "+r"(v[28]), "+r"(v[29]), "+r"(v[30]), "+r"(v[31])
                 :
                 : "memory");
}

// The store counterpart: thread i of the warp writes lane (taddr.lane + i), columns
// taddr.col .. taddr.col + 31.
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
          "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]),
          "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]),
          "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]),
          "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format) of a K-major operand tile whose rows are
// RowBytes (128 or 64) wide and stored with the swizzle of that width, as TMA writes them
// with CU_TENSOR_MAP_SWIZZLE_128B / _64B: 8-row groups 8 * RowBytes apart.  Fields: start
// address >> 4 in bits 0-13, leading byte offset >> 4 in 16-29 (unused for swizzled K-major
// layouts, 1), stride byte offset >> 4 in 32-45, the fixed value 1 in bits 46-47, base
// offset 0, and the layout type in bits 61-63 (2 = 128-byte swizzle, 4 = 64-byte swizzle).
// The tile base must be aligned to the swizzle pattern's repeat (8 rows); stepping along K
// inside a row adds the byte offset to the start address.
template <int RowBytes>
__device__ __forceinline__ uint64_t sdesc_k(uint32_t smem_addr) {
    static_assert(RowBytes == 128 || RowBytes == 64, "128- or 64-byte swizzled rows");
    constexpr uint64_t kLayout = RowBytes == 128 ? 2 : 4;
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;
    d |= static_cast<uint64_t>((8 * RowBytes) >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= kLayout << 61;
    return d;
}

// Instruction descriptor for kind::f16 / kind::tf32 with an fp32 accumulator, both operands
// K-major, dense: D format (1 = f32) in bits 4-5, A format in 7-9, B format in 10-12
// (f16 kind: 0 = fp16, 1 = bf16; tf32 kind: 2 = tf32), N >> 3 in bits 17-22, M >> 4 in
// bits 24-28.  A and B always have the same format.
__host__ __device__ constexpr uint32_t idesc_f32acc(uint32_t ab_format, int M, int N) {
    return (1u << 4) | (ab_format << 7) | (ab_format << 10) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
constexpr uint32_t kFmtF16 = 0;
constexpr uint32_t kFmtBF16 = 1;
constexpr uint32_t kFmtTF32 = 2;

// Round an fp32 value to tf32 (10 explicit mantissa bits), to nearest with ties away from
// zero; the result is an fp32 bit pattern whose low 13 bits are zero.
__device__ __forceinline__ float to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// fp32 operands on the tensor cores.  A value v is split into hi = tf32(v), which the
// kind::tf32 MMA reads from the first operand plane, and lo = v - hi (exact in fp32).  The
// second plane holds, per K element, one 32-bit word of two bf16 halves, bf16(hi) and
// bf16(lo), read by one kind::f16 MMA of twice the K: the input operand's word has bf16(hi)
// in its low half (the lower K index), the weight's has bf16(lo) there, so the products
// pair crosswise and the MMA adds hi_x * lo_w + lo_x * hi_w.  The dropped lo_x * lo_w is
// below 2^-22 of x * w, each cross product is off by at most about 2^-18 of it (two bf16
// roundings of a term below 2^-11 of it), and the three products of the 3xTF32 split (hi *
// hi, hi * lo, lo * hi in tf32) take one tf32 and one bf16 MMA here.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo_half, float hi_half) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi_half), "f"(lo_half));
    return r;
}
// Input operand: returns tf32(v) and sets the cross word (bf16(hi) low, bf16(lo) high).
__device__ __forceinline__ float split_x(float v, uint32_t &cross) {
    const float hi = to_tf32(v);
    cross = bf16x2_rn(hi, v - hi);
    return hi;
}
// Weight operand: returns tf32(v) and sets the cross word (bf16(lo) low, bf16(hi) high).
__device__ __forceinline__ float split_w(float v, uint32_t &cross) {
    const float hi = to_tf32(v);
    cross = bf16x2_rn(v - hi, hi);
    return hi;
}

}  // namespace ptx
}  // namespace ctr
