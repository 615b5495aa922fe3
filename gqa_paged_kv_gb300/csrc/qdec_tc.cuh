// qdec_tc.cuh -- inline PTX for the 5th-generation tensor core (tcgen05) used
// by the prefill attention: tensor-memory allocation, shared-memory matrix
// descriptors, the f16-kind MMA, commits to mbarriers, and loads/stores of
// the accumulators.  Not part of the ABI.
#pragma once

#include "qdec_internal.h"

namespace qdec {
namespace tc {

// Tensor-memory columns: allocated by one whole warp, address written to
// shared memory `slot`; the allocation permit is given up at once so that
// another CTA on the SM may allocate.
static __device__ __forceinline__ void alloc(uint32_t slot, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                 "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
static __device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
                 : "memory");
}
static __device__ __forceinline__ void fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
static __device__ __forceinline__ void fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Matrix descriptors of operands in the 128-byte swizzled layouts (atoms of
// 8 rows x 128 bytes, 1024 bytes, starting on 1024-byte boundaries).  Bits:
// start address >> 4 (0-13), leading byte offset >> 4 (16-29), stride byte
// offset >> 4 (32-45), descriptor version 1 (46-47), swizzle mode 2 = 128 B
// (61-63).
//   K-major (rows of the M or N dimension, 64 elements of K per 128-byte
//   row): stride = 1024 between 8-row groups; the leading offset is unused
//   within one 128-byte row (16).  A K step of 16 elements adds 32 bytes.
//   MN-major (rows of the K dimension, 64 elements of M or N per 128-byte
//   row): stride = distance between 8-row groups of K, leading offset =
//   distance between 64-element blocks of M or N.
static __device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo,
                                                      uint32_t sbo) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3fffu) |
           (static_cast<uint64_t>((lbo >> 4) & 0x3fffu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3fffu) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor of kind::f16 with bf16 A and B, fp32 D: D format
// (bits 4-5 = 1), A and B bf16 (7-9 = 1, 10-12 = 1), A and B major-ness
// (bit 15: A MN-major, bit 16: B MN-major), N >> 3 (17-22), M >> 4 (24-28).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn_major ? (1u << 16) : 0u) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// The same with f16 A and B (bits 7-9 = 0, 10-12 = 0).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool b_mn_major) {
    return (1u << 4) | (b_mn_major ? (1u << 16) : 0u) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// D (+)= A B, one K = 16 step, issued by one thread (A: M x 16 from adesc,
// B: 16 x N from bdesc).
static __device__ __forceinline__ void mma(uint32_t dtmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dtmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate ? 1 : 0)
        : "memory");
}
// D (+)= A B with A read from tensor memory (a_tmem: lane = row of A, each
// 32-bit column two consecutive K elements, the lower half first) and B from
// shared memory; one K = 16 step (8 columns of A).
static __device__ __forceinline__ void mma_ts(uint32_t dtmem, uint32_t a_tmem, uint64_t bdesc,
                                              uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(dtmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate ? 1 : 0)
        : "memory");
}
// One arrival on `bar` once every tcgen05 operation this thread issued so
// far has completed.
static __device__ __forceinline__ void commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::
                     "r"(bar)
                 : "memory");
}

// 32 consecutive fp32 columns of the 32 lanes this warp may access (warp
// w % 4: lanes 32 (w % 4) .. +31); taddr carries the lane base in bits 16-31.
static __device__ __forceinline__ void ld32(uint32_t (&v)[32], uint32_t taddr) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
          "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
          "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
}
static __device__ __forceinline__ void wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
static __device__ __forceinline__ void st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
        "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
        "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}
static __device__ __forceinline__ void wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

}  // namespace tc
}  // namespace qdec
