// qdec_ptx.cuh -- inline PTX wrappers shared by the kernel translation units
// of libqdec (mbarriers, matrix loads and products, programmatic launch,
// cluster barriers and distributed shared memory).  Not part of the ABI.
#pragma once

#include "qdec_internal.h"

namespace qdec {

static __device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// 2^x by the hardware's approximation (one instruction; relative error
// about 2^-22, far below the 16-bit rounding of the weights it feeds;
// 2^-inf = 0; results below 2^-126 flush to zero).
static __device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// The four E4M3 codes of `four_codes` (byte i = code i) as two f16 pairs:
// lo = codes 0, 1 and hi = codes 2, 3 (the lower code in the lower half);
// two conversion instructions on the word's halves, exact.
static __device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t four_codes, uint32_t &lo,
                                                        uint32_t &hi) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(four_codes));
}
// Two E4M3 codes (the low 16 bits of `two_codes`, the low byte first) as an
// f16 pair (low byte -> low half): one conversion instruction; exact, since
// every E4M3 value is an f16 value (NaN stays NaN).
static __device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
    uint32_t d;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(static_cast<unsigned short>(two_codes)));
    return d;
}
// E4M3 codes of lo and hi (nearest-even, saturated to +-448; NaN stays NaN)
// as two bytes, lo in the low byte: one conversion instruction.
static __device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
    unsigned short d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    return d;
}
static __device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
static __device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
static __device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
static __device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
static __device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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
// Wait for a barrier phase; give up after kWaitTimeoutCycles SM cycles (about
// two seconds) or when another thread of the CTA has already given up.  Never
// spins without bound.  The budget is counted with clock64(), which is
// monotonic on the SM the thread runs on (the global nanosecond timer is
// not: it can step backwards, which would end a wait at once).
static __device__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                  long long budget = kWaitTimeoutCycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > budget) return false;
    }
}
static __device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Plain bulk copy global -> shared (16-byte aligned addresses and size),
// counted on the transaction barrier `bar`.
static __device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                                 uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}
static __device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
static __device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
// D += A (16x16 bf16, row) * B (16x8 bf16, col), fp32 accumulate.
static __device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
static __device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
static __device__ __forceinline__ void launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Split cluster barrier: every thread of every CTA of the cluster arrives,
// then waits for all arrivals.
static __device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
static __device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}
static __device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}
static __device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// Generic address of the same shared-memory location in CTA `rank` of this
// cluster (distributed shared memory).
static __device__ __forceinline__ float *cluster_peer(float *ptr, int rank) {
    uint64_t r;
    asm volatile("mapa.u64 %0, %1, %2;"
                 : "=l"(r)
                 : "l"(reinterpret_cast<uint64_t>(ptr)), "r"(rank));
    return reinterpret_cast<float *>(r);
}

}  // namespace qdec
