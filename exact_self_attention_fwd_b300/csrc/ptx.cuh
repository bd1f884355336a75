// Inline-PTX wrappers for the sm_103a attention kernel: mbarriers, TMA tensor
// copies, tcgen05 (tensor memory allocation, MMA, commit, loads and stores) and
// a few scalar helpers. Every wrapper is a single documented PTX instruction (or a
// short fixed sequence of them); nothing here is derived from compiled code.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace attn {
namespace ptx {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (TMA, tensor core).
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// true once the phase with the given parity has completed
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_try_wait, but a thread that finds the phase incomplete may sleep until it
// completes or until about `hint_ns` nanoseconds pass, instead of spinning.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------ warp-uniform issue
// The producer and MMA roles run their loops on all 32 lanes of a warp with identical
// values, so that every operand below is warp-uniform; each of these wrappers issues its
// instruction from one lane, chosen by elect.sync inside the same asm statement.

__device__ __forceinline__ void mbar_arrive_expect_tx_elect(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;\n\t}"
        ::"r"(bar), "r"(bytes) : "memory");
}

// contiguous copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from
// global to shared memory, completing on `bar`; issued by one elected lane
__device__ __forceinline__ void bulk_load_elect(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n\t}"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// 3-D tiled tensor copy global -> shared, completing bytes on an mbarrier
__device__ __forceinline__ void tma_load_3d_elect(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                                  int x, int y, int z) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];\n\t}"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// D[tmem] (+)= A[tmem] B[smem desc] with e4m3 operands (kind::f8f6f4, K = 32), one MMA
__device__ __forceinline__ void mma_ts_elect_f8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Four MMAs issued from one asm statement by one elected lane: the k-th MMA uses the
// descriptors advanced by k x STEP in their start-address field (bits 0-13, in 16-byte
// units). Shared-memory addresses stay below 2^18 bytes, so the field never carries
// into bit 14 and a 32-bit add on the low word advances it. The first MMA accumulates
// when acc0 != 0, the others always accumulate. F8: kind::f8f6f4 (e4m3) instead of
// kind::f16.
//   mma_ss4: A and B from shared memory (descriptors), the same STEP for both.
//   mma_ts4: A from tensor memory (column address advanced by ACOLS per MMA), B from
//            shared memory advanced by STEP.
template <uint32_t STEP, bool F8 = false>
__device__ __forceinline__ void mma_ss4_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t acc0) {
    if constexpr (F8) {
        asm volatile(
            "{\n\t.reg .pred e, p, t;\n\t.reg .b32 alo, ahi, blo, bhi, x, y;\n\t.reg .b64 a, b;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "setp.eq.b32 t, %4, %4;\n\t"
            "mov.b64 {alo, ahi}, %1;\n\t"
            "mov.b64 {blo, bhi}, %2;\n\t"
            "elect.sync _|e, 0xffffffff;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t"
            "add.u32 x, alo, %5;\n\tadd.u32 y, blo, %5;\n\tmov.b64 a, {x, ahi};\n\tmov.b64 b, {y, bhi};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a, b, %3, t;\n\t"
            "add.u32 x, alo, %6;\n\tadd.u32 y, blo, %6;\n\tmov.b64 a, {x, ahi};\n\tmov.b64 b, {y, bhi};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a, b, %3, t;\n\t"
            "add.u32 x, alo, %7;\n\tadd.u32 y, blo, %7;\n\tmov.b64 a, {x, ahi};\n\tmov.b64 b, {y, bhi};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a, b, %3, t;\n\t}"
            ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc0), "n"(STEP), "n"(2 * STEP), "n"(3 * STEP)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred e, p, t;\n\t.reg .b32 alo, ahi, blo, bhi, x, y;\n\t.reg .b64 a, b;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "setp.eq.b32 t, %4, %4;\n\t"
            "mov.b64 {alo, ahi}, %1;\n\t"
            "mov.b64 {blo, bhi}, %2;\n\t"
            "elect.sync _|e, 0xffffffff;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
            "add.u32 x, alo, %5;\n\tadd.u32 y, blo, %5;\n\tmov.b64 a, {x, ahi};\n\tmov.b64 b, {y, bhi};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t"
            "add.u32 x, alo, %6;\n\tadd.u32 y, blo, %6;\n\tmov.b64 a, {x, ahi};\n\tmov.b64 b, {y, bhi};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t"
            "add.u32 x, alo, %7;\n\tadd.u32 y, blo, %7;\n\tmov.b64 a, {x, ahi};\n\tmov.b64 b, {y, bhi};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t}"
            ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc0), "n"(STEP), "n"(2 * STEP), "n"(3 * STEP)
            : "memory");
    }
}

template <uint32_t ACOLS, uint32_t STEP, bool F8 = false>
__device__ __forceinline__ void mma_ts4_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                              uint32_t acc0) {
    if constexpr (F8) {
        asm volatile(
            "{\n\t.reg .pred e, p, t;\n\t.reg .b32 blo, bhi, x, y;\n\t.reg .b64 b;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "setp.eq.b32 t, %4, %4;\n\t"
            "mov.b64 {blo, bhi}, %2;\n\t"
            "elect.sync _|e, 0xffffffff;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t"
            "add.u32 x, %1, %5;\n\tadd.u32 y, blo, %8;\n\tmov.b64 b, {y, bhi};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [x], b, %3, t;\n\t"
            "add.u32 x, %1, %6;\n\tadd.u32 y, blo, %9;\n\tmov.b64 b, {y, bhi};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [x], b, %3, t;\n\t"
            "add.u32 x, %1, %7;\n\tadd.u32 y, blo, %10;\n\tmov.b64 b, {y, bhi};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [x], b, %3, t;\n\t}"
            ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc0), "n"(ACOLS), "n"(2 * ACOLS),
              "n"(3 * ACOLS), "n"(STEP), "n"(2 * STEP), "n"(3 * STEP)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred e, p, t;\n\t.reg .b32 blo, bhi, x, y;\n\t.reg .b64 b;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "setp.eq.b32 t, %4, %4;\n\t"
            "mov.b64 {blo, bhi}, %2;\n\t"
            "elect.sync _|e, 0xffffffff;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
            "add.u32 x, %1, %5;\n\tadd.u32 y, blo, %8;\n\tmov.b64 b, {y, bhi};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [x], b, %3, t;\n\t"
            "add.u32 x, %1, %6;\n\tadd.u32 y, blo, %9;\n\tmov.b64 b, {y, bhi};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [x], b, %3, t;\n\t"
            "add.u32 x, %1, %7;\n\tadd.u32 y, blo, %10;\n\tmov.b64 b, {y, bhi};\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [x], b, %3, t;\n\t}"
            ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc0), "n"(ACOLS), "n"(2 * ACOLS),
              "n"(3 * ACOLS), "n"(STEP), "n"(2 * STEP), "n"(3 * STEP)
            : "memory");
    }
}

__device__ __forceinline__ void mma_commit_elect(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
        ::"r"(bar) : "memory");
}

// ------------------------------------------------------------------ tcgen05
// Tensor-memory allocation (whole warp), result address written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
                 : "memory");
    return v;
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 32 columns of 32-bit: thread i of the warp gets lane (base+i), 32 columns.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
          "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
          "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]),
          "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
          "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
          "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
          "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ register split
// Per-warpgroup register budget changes (all four warps of a warpgroup execute them).
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ------------------------------------------------------------------ descriptors
// Shared-memory matrix descriptor for a 128-byte-swizzled operand (tcgen05 format):
// start address, leading- and stride-dimension byte offsets (all >> 4), descriptor
// version 1 at bit 46, base offset 0 (tiles are 1024-byte aligned), layout type
// SWIZZLE_128B (= 2) in bits 61..63.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor, kind::f16 with bf16 A and B, fp32 accumulator.
// Bits: [4,6) D format (1 = f32), [7,10) A format (1 = bf16), [10,13) B format
// (1 = bf16), 15 A major (0 = K), 16 B major (1 = MN), [17,23) N >> 3, [24,29) M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor, kind::f8f6f4 with e4m3 A and B (format code 0), fp32 accumulator;
// the same bit layout as above.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N, bool b_mn_major) {
    return (1u << 4) | (0u << 7) | (0u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ------------------------------------------------------------------ scalar helpers
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// v, or the bit pattern of -inf when off > span (unsigned), as one predicated select
__device__ __forceinline__ uint32_t mask_above(uint32_t v, uint32_t off, uint32_t span) {
    uint32_t r;
    asm("{\n\t.reg .pred p;\n\t"
        "setp.gt.u32 p, %1, %2;\n\t"
        "selp.b32 %0, 0xFF800000, %3, p;\n\t}"
        : "=r"(r) : "r"(off), "r"(span), "r"(v));
    return r;
}

// max of three floats in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// acc += the two bf16 halves of `packed` (each widened exactly to fp32): acc_lo gets
// the low half, acc_hi the high half
__device__ __forceinline__ void add_bf16x2_halves(float &acc_lo, float &acc_hi, uint32_t packed) {
    asm("{\n\t.reg .b16 l, h;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "add.rn.f32.bf16 %0, l, %0;\n\t"
        "add.rn.f32.bf16 %1, h, %1;\n\t}"
        : "+f"(acc_lo), "+f"(acc_hi)
        : "r"(packed));
}

// four floats -> four e4m3 codes (round to nearest even, saturating at 448), x0 in the
// lowest byte
__device__ __forceinline__ uint32_t pack_e4m3x4(float x0, float x1, float x2, float x3) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(x1), "f"(x0));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(x3), "f"(x2));
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// acc_a += value of the low two e4m3 codes of `w`, acc_b += the high two (each code
// widened exactly, through f16)
__device__ __forceinline__ void add_e4m3x4(float &acc_a, float &acc_b, uint32_t w) {
    asm("{\n\t.reg .b16 l, h;\n\t.reg .b32 fl, fh;\n\t.reg .b16 a0, a1, b0, b1;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 fl, l;\n\t"
        "cvt.rn.f16x2.e4m3x2 fh, h;\n\t"
        "mov.b32 {a0, a1}, fl;\n\t"
        "mov.b32 {b0, b1}, fh;\n\t"
        "add.rn.f32.f16 %0, a0, %0;\n\t"
        "add.rn.f32.f16 %0, a1, %0;\n\t"
        "add.rn.f32.f16 %1, b0, %1;\n\t"
        "add.rn.f32.f16 %1, b1, %1;\n\t}"
        : "+f"(acc_a), "+f"(acc_b)
        : "r"(w));
}

__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// two floats -> packed bf16x2 (round to nearest even), `lo` in the low half
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

}  // namespace ptx
}  // namespace attn
