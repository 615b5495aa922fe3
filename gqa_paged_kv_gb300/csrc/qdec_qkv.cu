// qdec_qkv.cu -- the merged QKV projection fused with steps 1-3 (RMSNorm,
// NeoX RoPE, paged append), on sm_103a.
//
// The projection is one matrix W [(Hq + 2 Hkv) * D][hidden] (article "扔掉
// vLLM！从零构建 Qwen3-8B 推理引擎" (news.rkmt.cn), section 4.4.3: the q, k and v
// projections merged into one; rows: the query heads, then the key heads,
// then the value heads), applied to every sequence's hidden state x [B][hidden].
// Its epilogue keeps each head's 128 outputs unrounded (fp32) into the norm,
// the rotation and the append: query heads go to q_rot (fp32, unscaled, the
// input of qdec_attn_decode / qdec_attn_split), key heads are rounded once to
// bf16 after the rotation and value heads once as they are, into slot
// seq_lens[b] - 1 (into an FP8 pool: those bf16 rows divided by the slot's
// scales and rounded to E4M3).
//
// Layout: a cluster of 4 CTAs per output head splits the hidden dimension:
// CTA r computes all 128 dims of the head for up to 64 batch rows over its
// quarter of the 64-element blocks of hidden, so it streams a quarter of the
// head's weight and of x.  The weight is packed once (qdec_qkv_pack_weights)
// into the order the projection reads it: per (head, block of 64 hidden
// elements) 16 KiB, four 4 KiB sub-blocks of 32 rows (sub-block i: dims
// 16i .. 16i+15, then 64+16i .. 64+16i+15), each 128-byte row already
// swizzled for conflict-free matrix loads; a CTA's share is one contiguous
// run.  One producer warp streams stages of one 16 KiB block (one bulk copy)
// and the matching box of x (the batch rounded up to 16 rows, at most 64; rows
// past B read as zero, TMA) into a ring of about 96 KiB.  Both land in the
// K-major 128-byte-swizzled layout the 5th-generation tensor core reads from
// shared memory: one thread issues, per stage, four tcgen05.mma of kind f16
// (bf16 operands, M = 128 head dims, N = the R batch rows, K = 16) that
// accumulate D [128][R] in fp32 in tensor memory, and commits them to the
// stage's empty barrier, so the stage is refilled as soon as they have read it.
// Once the MMAs have completed, the four consumer warps read D out of tensor
// memory (warp w: lanes 32w .. 32w+31) into a partial-sum tile in shared
// memory, and after one cluster barrier every CTA pushes to CTA q (one bulk
// shared-to-shared copy each, counted on q's transaction barrier) the rows q
// owns: rows q R/4 .. (q+1) R/4 - 1 of the R.  The owner adds the four partials in rank order, so each row's 128
// dims are complete in one CTA: the RMSNorm sum of squares, the rotation and
// the writes need nothing from the peers.  The epilogue's lookups (append
// slot, norm weights, rotation table) are made before the main loop.
#include "qdec_internal.h"
#include "qdec_ptx.cuh"
#include "qdec.h"

#include <math.h>

#include <algorithm>
#include <mutex>

namespace qdec {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kQkvCluster = 4;                              // CTAs per output head
constexpr int kQkvRows = 4 * 16;                            // batch rows per CTA
constexpr int kQkvChunk = 64;                               // hidden elements per block
constexpr int kQkvMaxStages = 16;
constexpr int kQkvSub = 32 * kQkvChunk * 2;                 // one 32-row sub-block, 4 KiB
constexpr int kQkvBlock = kQkvCluster * kQkvSub;            // one head's block, 16 KiB
constexpr int kQkvRingBytes = 96 * 1024;
constexpr int kQkvPartStride = kHeadDim + 8;                // floats per row of the partials
constexpr int kQkvSliceMax = kQkvRows / kQkvCluster * kQkvPartStride * 4;  // rows one CTA owns
constexpr int kQkvRecvOff = 36 * 1024;                      // receive area in the ring
constexpr int kQkvRingUse = kQkvRecvOff + kQkvCluster * kQkvSliceMax;
constexpr int kQkvTmemCols = 64;                           // fp32 accumulator columns (N <= 64)
// after the ring: barriers full[16], empty[16], recv, mma-done, the abort
// flag, the tensor-memory address
constexpr int kQkvTailBytes = 2 * kQkvMaxStages * 8 + 8 + 8 + 8 + 8;
static_assert(kQkvRows * kQkvPartStride * 4 <= kQkvRecvOff, "partials end before the receive area");
// a stage: [boxes packed blocks of 16 KiB][boxes x boxes of rows x 64], each
// piece starting on a 1024-byte boundary (rows % 16 == 0)
__host__ __device__ constexpr int qkv_stage_bytes(int rows, int boxes) {
    return boxes * (kQkvBlock + rows * kQkvChunk * 2);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Bulk copy of `bytes` from this CTA's shared memory to the same-offset-mapped
// address `dst` of a peer (shared::cluster), counted on the peer's barrier.
__device__ __forceinline__ void bulk_push(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, "
        "[%3];" ::"r"(dst),
        "r"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ uint32_t cluster_addr(uint32_t local, int rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

// Address of row r, 16-byte chunk c of a 128-byte-swizzled box at `base`.
__device__ __forceinline__ uint32_t swz(uint32_t base, int r, int c) {
    return base + r * 128 + ((c ^ (r & 7)) << 4);
}

// ---- 5th-generation tensor core (tcgen05) wrappers.  The accumulator D
// lives in tensor memory (lane = row of D, one 32-bit column per fp32
// element); A and B are read from shared memory through matrix descriptors.
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t cols) {  // whole warp
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                 "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {  // whole warp
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzled layout (8-row x 128-byte atoms, 1024 bytes apart; the atoms must
// start on 1024-byte boundaries): start address >> 4 in bits 0-13, leading
// byte offset (unused for this layout; 16 bytes) >> 4 in bits 16-29, stride
// byte offset 1024 >> 4 in bits 32-45, descriptor version 1 in bits 46-47,
// layout 2 (128-byte swizzle) in bits 61-63.  Stepping K by 16 elements adds
// 32 bytes to the start address.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3fffu) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}
// Instruction descriptor of kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
// (bits 7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 in bits
// 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t f16_idesc(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}
// D (+)= A B^T for one K = 16 step, issued by one thread
__device__ __forceinline__ void tc_mma(uint32_t dtmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dtmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate ? 1 : 0)
        : "memory");
}
// arrive (once) on `bar` when every tcgen05 operation this thread issued so
// far has completed
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
// 16 consecutive columns of this warp's 32 lanes (lane l: row 32 (warp % 4) + l)
__device__ __forceinline__ void tmem_ld16(uint32_t (&v)[16], uint32_t taddr) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void flag_error(int32_t *err, int bits) {
    if (err) atomicOr(err, bits);
}

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t v) {  // exact: bf16 -> fp32
    return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
           (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
}

// Four dims d0 .. d0+3 (a) and d0+64 .. d0+67 (c) of a key or value row into
// its slot at element offset `slot`: bf16 (nearest-even) into the bf16 pool,
// or, with an FP8 pool, the E4M3 codes of those bf16 values divided by the
// slot's scale kv_scale[si] (fp32 division, nearest-even, saturating) --
// slot / (16 * 128) is page * 2 Hkv + head, the K scale's index.
__device__ __forceinline__ void store_row4(const Params &p, int64_t slot, int d0,
                                           const float *a, const float *c, int64_t si) {
    const uint2 lo = make_uint2(pack2_bf16(a[0], a[1]), pack2_bf16(a[2], a[3]));
    const uint2 hi = make_uint2(pack2_bf16(c[0], c[1]), pack2_bf16(c[2], c[3]));
    if (p.pool8 == nullptr) {
        *reinterpret_cast<uint2 *>(p.pool + slot + d0) = lo;
        *reinterpret_cast<uint2 *>(p.pool + slot + d0 + 64) = hi;
        return;
    }
    const float s = p.kv_scale[si];
    auto codes = [s](uint2 v) {  // four bf16 -> four E4M3 codes, low dim first
        const float2 f0 = make_float2(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u));
        const float2 f1 = make_float2(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
        const uint32_t c0 = f32x2_to_e4m3x2(__fdiv_rn(f0.x, s), __fdiv_rn(f0.y, s));
        const uint32_t c1 = f32x2_to_e4m3x2(__fdiv_rn(f1.x, s), __fdiv_rn(f1.y, s));
        return (c0 & 0xffffu) | (c1 << 16);
    };
    *reinterpret_cast<uint32_t *>(p.pool8 + slot + d0) = codes(lo);
    *reinterpret_cast<uint32_t *>(p.pool8 + slot + d0 + 64) = codes(hi);
}


// kTc: the contraction on the 5th-generation tensor core (tcgen05, operands
// read from shared memory, the accumulator in tensor memory); otherwise on
// mma.sync with the accumulators in registers, which has the shorter fixed
// cost per launch and is used when the batch fits one 16-row tile (where the
// weight stream, not the arithmetic, sets the time).
template <bool kTc>
__global__ void __launch_bounds__(kThreads, 2)
    qkv_append_kernel(const __grid_constant__ CUtensorMap x_map, const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int head = blockIdx.x / kQkvCluster, rank = blockIdx.x % kQkvCluster;
    const int row0 = blockIdx.y * kQkvRows;
    const int NB = p.qkv_boxes;
    const int R = p.qkv_rows;
    const int NS = p.qkv_stages;
    const int stage_bytes = qkv_stage_bytes(R, NB);
    // this CTA's 64-element blocks of hidden: [kb0, kb1), in stages of NB
    const int nk = p.hidden / kQkvChunk;
    const int kb0 = rank * nk / kQkvCluster, kb1 = (rank + 1) * nk / kQkvCluster;
    const int nchunks = (kb1 - kb0) / max(NB, 1);
    uint8_t *tail = sm + NS * stage_bytes;
    const uint32_t full0 = smem_u32(tail);
    const uint32_t empty0 = full0 + kQkvMaxStages * 8;
    const uint32_t recv_bar = empty0 + kQkvMaxStages * 8;
    const uint32_t done_bar = recv_bar + 8;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tail + 2 * kQkvMaxStages * 8 + 16);
    volatile uint32_t *tmem_slot =
        reinterpret_cast<volatile uint32_t *>(tail + 2 * kQkvMaxStages * 8 + 24);
    if (NS < 1 || NS > kQkvMaxStages || R < 16 || R > kQkvRows || R % 16 != 0 || NB < 1 ||
        NB > 2 || p.hidden % kQkvChunk != 0 || (kb1 - kb0) % NB != 0 ||
        NS * stage_bytes < kQkvRingUse) {
        if (tid == 0) flag_error(p.err, QDEC_FLAG_BAD_INDEX);
        return;  // uniform over the cluster: every CTA sees the same parameters
    }

    if (p.pdl && tid == 0) launch_dependents();  // the next kernel waits for our completion
    // The producer thread sets up the barriers and at once sends the weight
    // (which no kernel writes) of the first stages, before any dependency
    // wait, with their boxes of x unless the launch overlaps the previous
    // kernel; warp 0 meanwhile allocates the tensor memory.
    const __nv_bfloat16 *wsrc =
        p.w_packed + (static_cast<int64_t>(head) * nk + kb0) * (kQkvBlock / 2);
    const int pre = min(NS, nchunks);
    if (warp == kConsumerWarps && lane == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full0 + 8 * s, 1);
            // tcgen05: the commit of the stage's MMAs; mma.sync: every consumer warp
            mbar_init(empty0 + 8 * s, kTc ? 1 : kConsumerWarps);
        }
        mbar_init(recv_bar, 1);
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        for (int c = 0; c < pre; ++c) {
            if (p.withhold_first && c == 0) continue;  // test hook: stage 0 never lands
            const uint32_t full = full0 + 8 * c;
            mbar_arrive_expect_tx(full, stage_bytes);
            bulk_load(smem_u32(sm + c * stage_bytes),
                      wsrc + static_cast<int64_t>(c) * NB * (kQkvBlock / 2), NB * kQkvBlock, full);
            for (int j = 0; j < NB && !p.pdl; ++j)
                tma_load_2d(smem_u32(sm + c * stage_bytes) + NB * kQkvBlock + j * R * kQkvChunk * 2,
                            &x_map, (kb0 + c * NB + j) * kQkvChunk, row0, full);
        }
    }
    if (kTc && warp == 0) tmem_alloc(smem_u32(const_cast<uint32_t *>(tmem_slot)), kQkvTmemCols);
    if (kTc) tc_fence_before();
    __syncthreads();
    if (kTc) tc_fence_after();
    const uint32_t tmem = kTc ? *tmem_slot : 0u;  // lane 0, the first allocated column

    // The partial sums [64 rows][128 + 8] fp32 overwrite the ring once every
    // stage is consumed; CTA q owns rows q R/4 .. (q+1) R/4 - 1 (a contiguous
    // slice of part) and receives the peers' slices of them at
    // recv + sender * kQkvSliceMax.
    float *part = reinterpret_cast<float *>(sm);
    const int R4 = R / kQkvCluster;
    const uint32_t slice_bytes = R4 * kQkvPartStride * 4;
    const uint32_t recv = smem_u32(sm + kQkvRecvOff);
    if (warp == kConsumerWarps) {
        // ------------------------------------------------ TMA producer --
        if (lane == 0) {
            // the remaining hidden states only after the dependency wait
            if (p.pdl) grid_dependency_wait();
            for (int c = 0; c < nchunks; ++c) {
                const int s = c % NS;
                const uint32_t full = full0 + 8 * s;
                const uint32_t dst = smem_u32(sm + s * stage_bytes);
                if (c >= pre) {
                    if (c >= NS &&
                        !mbar_wait_bounded(empty0 + 8 * s, ((c / NS) - 1) & 1, abort_flag,
                                           p.wait_cycles)) {
                        *abort_flag = 1;
                        flag_error(p.err, QDEC_FLAG_TIMEOUT);
                        break;
                    }
                    mbar_arrive_expect_tx(full, stage_bytes);
                    bulk_load(dst, wsrc + static_cast<int64_t>(c) * NB * (kQkvBlock / 2),
                              NB * kQkvBlock, full);
                }
                const bool send_x = (c >= pre || p.pdl) && !(p.withhold_first && c == 0);
                for (int j = 0; j < NB && send_x; ++j)
                    tma_load_2d(dst + NB * kQkvBlock + j * R * kQkvChunk * 2, &x_map,
                                (kb0 + c * NB + j) * kQkvChunk, row0, full);
            }
        }
        __syncwarp();
        cluster_sync_all();  // partials in place, every ring free
    } else {
        // ------------------------------------------- consumer warps --
        // kTc: thread 0 issues the tensor-core MMAs: per stage, D [128 dims]
        // [R rows] += W_block [128][64] x_box [R][64]^T in four K = 16 steps,
        // committed to the stage's empty barrier; all four warps then read D.
        // Otherwise every warp takes every stage with mma.sync (see below).
        if (p.pdl) grid_dependency_wait();  // the tables, q_rot and the pool of earlier kernels

        // ---- the epilogue's inputs, fetched while the weight streams.  Thread
        // tid takes rows rs and rs + 8 (rs = tid / 16) of this CTA's R/4 and
        // the rotate-half pairs 4 (tid % 16) .. +3: dims d0 .. d0+3 and
        // d0+64 .. d0+67.  slot: the append slot (-1: skip the row).
        const int rs = tid >> 4, d0 = 4 * (tid & 15);
        const int Hq = p.Hq, Hkv = p.Hkv;
        const int kind = head < Hq ? 0 : (head < Hq + Hkv ? 1 : 2);  // q, k or v head
        const int kvh = kind == 1 ? head - Hq : head - Hq - Hkv;
        int64_t slot[2] = {-1, -1};
        float4 cs[2][2];  // (c_hi, s_hi) of pairs d0 .. d0+3 per row: {c0 s0 c1 s1}, {c2 s2 c3 s3}
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            cs[h][0] = cs[h][1] = make_float4(0.f, 0.f, 0.f, 0.f);
            const int i = rs + 8 * h, b = row0 + rank * R4 + i;
            if (i >= R4 || b >= p.B) continue;
            const int L = p.seq_lens[b];
            if (L < 1 || L > p.max_blocks * kPageSize) {
                if ((tid & 15) == 0 && head == 0) flag_error(p.err, QDEC_FLAG_BAD_SEQLEN);
                continue;
            }
            if (kind != 2) {
                const RopeEntry *e = p.rope + static_cast<int64_t>(b) * kRotPairs + d0;
                cs[h][0] = make_float4(e[0].c_hi, e[0].s_hi, e[1].c_hi, e[1].s_hi);
                cs[h][1] = make_float4(e[2].c_hi, e[2].s_hi, e[3].c_hi, e[3].s_hi);
            }
            if (kind == 0) {
                slot[h] = 0;
                continue;
            }
            const int page =
                p.block_table[static_cast<int64_t>(b) * p.max_blocks + (L - 1) / kPageSize];
            if (page < 0 || page >= p.num_pages) {
                if ((tid & 15) == 0 && kvh == 0 && kind == 1) flag_error(p.err, QDEC_FLAG_BAD_PAGE);
                continue;
            }
            slot[h] =
                ((static_cast<int64_t>(page) * 2 * Hkv + kvh) * kPageSize + (L - 1) % kPageSize) *
                kHeadDim;
        }
        uint2 wn1 = make_uint2(0u, 0u), wn2 = make_uint2(0u, 0u);  // norm weights, bf16 pairs
        if (kind != 2) {
            const __nv_bfloat16 *wn = kind == 0 ? p.w_q : p.w_k;
            wn1 = *reinterpret_cast<const uint2 *>(wn + d0);
            wn2 = *reinterpret_cast<const uint2 *>(wn + d0 + 64);
        }

        bool aborted = false;
        if constexpr (kTc) {
            if (tid == 0) {
                const uint32_t idesc = f16_idesc(kHeadDim, R);
                for (int c = 0; c < nchunks; ++c) {
                    const int s = c % NS;
                    if (!mbar_wait_bounded(full0 + 8 * s, (c / NS) & 1, abort_flag, p.wait_cycles)) {
                        *abort_flag = 1;
                        flag_error(p.err, QDEC_FLAG_TIMEOUT);
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sb = smem_u32(sm + s * stage_bytes);
                    for (int j = 0; j < NB; ++j) {
                        const uint32_t wb = sb + j * kQkvBlock;
                        const uint32_t xb = sb + NB * kQkvBlock + j * R * kQkvChunk * 2;
#pragma unroll
                        for (int kk = 0; kk < kQkvChunk / 16; ++kk)
                            tc_mma(tmem, sw128_desc(wb + 32 * kk), sw128_desc(xb + 32 * kk), idesc,
                                   c > 0 || j > 0 || kk > 0);
                    }
                    tc_commit(empty0 + 8 * s);  // the stage may be refilled once these are done
                }
                tc_commit(done_bar);  // every MMA issued above has completed
            }
            __syncwarp();
            // wait for the MMAs whatever happened: tensor memory is released below
            {
                volatile int never = 0;
                if (!mbar_wait_bounded(done_bar, 0, &never, p.wait_cycles)) {
                    aborted = true;
                    if (lane == 0) {
                        *abort_flag = 1;
                        flag_error(p.err, QDEC_FLAG_TIMEOUT);
                    }
                }
            }
            aborted = aborted || *abort_flag;
            tc_fence_after();
            // D row 32 warp + lane (part column) for batch rows 0 .. R-1 -> part
            // [row][column]; the ring is free (every stage's MMAs completed)
            for (int c0 = 0; c0 < R; c0 += 16) {
                uint32_t v[16];
                tmem_ld16(v, tmem + (static_cast<uint32_t>(32 * warp) << 16) + c0);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    part[(c0 + e) * kQkvPartStride + 32 * warp + lane] =
                        nchunks > 0 && !aborted ? __uint_as_float(v[e]) : 0.f;
            }
            tc_fence_before();
            asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
            if (warp == 0) {
                tc_fence_after();
                tmem_dealloc(tmem, kQkvTmemCols);
            }
        } else {
            // RT 16-row tiles x CG column groups (RT * CG <= 4): warp w takes
            // tile w / CG and sub-blocks [(w % CG) * 4 / CG, +4 / CG) of every
            // block, i.e. NT = 16 / CG n-tiles of 8 columns
            const int g = lane >> 2, t = lane & 3;
            const int RT = R / 16;
            const int CG = RT == 1 ? 4 : (RT == 2 ? 2 : 1);
            const int NT = 16 / CG;
            const int rt = warp / CG, sb0 = (warp % CG) * (4 / CG);
            const bool live = rt < RT && row0 + 16 * rt < p.B;
            float acc[16][4];
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
            const int mi = lane >> 3, r8 = lane & 7;
            const int arow = 16 * rt + (mi & 1) * 8 + r8;  // x row this lane addresses
            const int brow = (mi >> 1) * 8 + r8;            // W row within a 16-row half sub-block
            for (int c = 0; c < nchunks; ++c) {
                const int s = c % NS;
                const bool ok = mbar_wait_bounded(full0 + 8 * s, (c / NS) & 1, abort_flag,
                                                  p.wait_cycles);
                if (!ok) {
                    if (lane == 0) {
                        *abort_flag = 1;
                        flag_error(p.err, QDEC_FLAG_TIMEOUT);
                    }
                    aborted = true;
                    break;
                }
                for (int j = 0; j < NB && live; ++j) {
                    const uint32_t sb = smem_u32(sm + s * stage_bytes);
                    const uint32_t wb = sb + j * kQkvBlock + sb0 * kQkvSub;
                    const uint32_t xb = sb + NB * kQkvBlock + j * R * kQkvChunk * 2;
#pragma unroll
                    for (int kk = 0; kk < kQkvChunk / 16; ++kk) {
                        uint32_t a[4];
                        ldmatrix_x4(a, swz(xb, arow, 2 * kk + (mi >> 1)));
#pragma unroll
                        for (int pr = 0; pr < 8; ++pr) {  // n-tile pairs: 16 W rows each
                            if (2 * pr >= NT) break;
                            uint32_t b[4];
                            // pair pr: sub-block pr / 2, rows 16 (pr % 2) ..
                            ldmatrix_x4(b, swz(wb + (pr >> 1) * kQkvSub, 16 * (pr & 1) + brow,
                                               2 * kk + (mi & 1)));
                            mma_bf16(acc[2 * pr], a, b[0], b[1]);
                            mma_bf16(acc[2 * pr + 1], a, b[2], b[3]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty0 + 8 * s);
            }
            // every stage is consumed (no copy is landing in the ring): the
            // partials go to part[row][column], column = 32 * sub-block + row of it
            asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
            if (live && !aborted) {
#pragma unroll
                for (int nt = 0; nt < 16; ++nt) {
                    if (nt >= NT) break;
                    const int col = 32 * sb0 + 8 * nt + 2 * t;
                    float *r0 = part + (16 * rt + g) * kQkvPartStride + col;
                    *reinterpret_cast<float2 *>(r0) = make_float2(acc[nt][0], acc[nt][1]);
                    *reinterpret_cast<float2 *>(r0 + 8 * kQkvPartStride) =
                        make_float2(acc[nt][2], acc[nt][3]);
                }
            }
        }
        fence_proxy_async_smem();  // the partials are read next by bulk copies
        cluster_sync_all();        // every CTA's partials are in place, every ring is free

        // push slice q of the partials to CTA q (one bulk copy each)
        if (tid == 0) {
            mbar_arrive_expect_tx(recv_bar, (kQkvCluster - 1) * slice_bytes);
#pragma unroll
            for (int q = 0; q < kQkvCluster; ++q) {
                if (q == rank) continue;
                bulk_push(cluster_addr(recv + rank * kQkvSliceMax, q),
                          smem_u32(part + q * R4 * kQkvPartStride), slice_bytes,
                          cluster_addr(recv_bar, q));
            }
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
        // every peer pushes after the barrier whatever happened before it, so
        // wait for the bytes even after an abort: this CTA's memory must
        // outlive the copies into it (bounded all the same)
        volatile int never = 0;
        const bool got = mbar_wait_bounded(recv_bar, 0, &never, p.wait_cycles);
        if (!got && tid == 0) {
            *abort_flag = 1;
            flag_error(p.err, QDEC_FLAG_TIMEOUT);
        }

        // the owned rows: the four CTAs' partials added in rank order, then
        // RMSNorm over the 128 dims (16 threads per row), RoPE, write
        const float2 w01 = bf16x2_to_float2(wn1.x), w23 = bf16x2_to_float2(wn1.y);
        const float2 w45 = bf16x2_to_float2(wn2.x), w67 = bf16x2_to_float2(wn2.y);
        const float wv[8] = {w01.x, w01.y, w23.x, w23.y, w45.x, w45.y, w67.x, w67.y};
        // part column of dim d < 64: 32 (d / 16) + d % 16; of dim 64 + d: that + 16
        const int clo = 32 * (d0 >> 4) + (d0 & 15);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int i = rs + 8 * h;
            if (i >= R4) break;  // uniform over each half-warp (16 threads per row)
            float y[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = 0.f;
#pragma unroll
            for (int q = 0; q < kQkvCluster; ++q) {
                const float *src = q == rank ? part + (rank * R4 + i) * kQkvPartStride
                                             : reinterpret_cast<const float *>(
                                                   sm + kQkvRecvOff + q * kQkvSliceMax) +
                                                   i * kQkvPartStride;
                const float4 lo = *reinterpret_cast<const float4 *>(src + clo);
                const float4 hi = *reinterpret_cast<const float4 *>(src + clo + 16);
                y[0] += lo.x; y[1] += lo.y; y[2] += lo.z; y[3] += lo.w;
                y[4] += hi.x; y[5] += hi.y; y[6] += hi.z; y[7] += hi.w;
            }
            float sq = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) sq += y[e] * y[e];
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) sq += __shfl_xor_sync(kFull, sq, o);
            const int b = row0 + rank * R4 + i;
            if (aborted || *abort_flag || slot[h] < 0) continue;
            const int64_t kslot = slot[h];
            if (kind == 2) {
                const int64_t vslot = kslot + static_cast<int64_t>(Hkv) * kPageSize * kHeadDim;
                store_row4(p, vslot, d0, y, y + 4, (kslot >> 11) + Hkv);
                continue;
            }
            const float rn = rsqrtf(sq * (1.0f / kHeadDim) + p.eps);
            const float c[4] = {cs[h][0].x, cs[h][0].z, cs[h][1].x, cs[h][1].z};
            const float sn[4] = {cs[h][0].y, cs[h][0].w, cs[h][1].y, cs[h][1].w};
            float o1[4], o2[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float n1 = y[e] * rn * wv[e], n2 = y[4 + e] * rn * wv[4 + e];
                o1[e] = n1 * c[e] - n2 * sn[e];
                o2[e] = n2 * c[e] + n1 * sn[e];
            }
            if (kind == 0) {
                float *dst = p.q_rot_out + (static_cast<int64_t>(b) * Hq + head) * kHeadDim;
                *reinterpret_cast<float4 *>(dst + d0) = make_float4(o1[0], o1[1], o1[2], o1[3]);
                *reinterpret_cast<float4 *>(dst + d0 + 64) = make_float4(o2[0], o2[1], o2[2], o2[3]);
            } else {
                store_row4(p, kslot, d0, o1, o2, kslot >> 11);
            }
        }
        // the pushed slices must be read out before this CTA's memory is released
        if (tid == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    }
    __syncthreads();
    // a wait that gave up may leave copies in flight: let them land (bounded)
    if (tid == 0 && *abort_flag) {
        volatile int never = 0;
        const int first = nchunks > NS ? nchunks - NS : 0;
        for (int c = first; c < nchunks; ++c)
            mbar_wait_bounded(full0 + 8 * (c % NS), (c / NS) & 1, &never, p.wait_cycles);
    }
}

// Packing: destination 16-byte unit u lies in block u / 1024 (16 KiB, block
// index = head * (hidden / 64) + k-block), sub-block (u / 256) % 4, row
// (u / 8) % 32 of the sub-block, position u % 8, which holds source chunk
// (u % 8) ^ (row % 8) of that row (the 128-byte swizzle).  Sub-block i rows
// 0-15 are weight rows head * 128 + 16 i + row, rows 16-31 are
// head * 128 + 64 + 16 i + row - 16.
__global__ void qkv_pack_kernel(const __nv_bfloat16 *w, __nv_bfloat16 *wp, int rows, int hidden) {
    const int64_t total = static_cast<int64_t>(rows) * hidden / 8;
    const int nk = hidden / kQkvChunk;
    for (int64_t u = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; u < total;
         u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t block = u / 1024;
        const int sub = static_cast<int>((u / 256) % 4);
        const int rho = static_cast<int>((u / 8) % 32), pos = static_cast<int>(u % 8);
        const int q = pos ^ (rho & 7);
        const int kb = static_cast<int>(block % nk);
        const int head = static_cast<int>(block / nk);
        const int row = head * kHeadDim + (rho < 16 ? 16 * sub + rho : 64 + 16 * sub + rho - 16);
        const uint4 v = *reinterpret_cast<const uint4 *>(
            w + static_cast<int64_t>(row) * hidden + kb * kQkvChunk + q * 8);
        *reinterpret_cast<uint4 *>(wp + u * 8) = v;
    }
}

std::mutex g_qkv_mu;
bool g_qkv_smem_set[64];
constexpr int kQkvSmemMax = kQkvRingBytes + kQkvTailBytes + 1024;

}  // namespace

void qkv_geometry(int B, int hidden, int &rows, int &boxes, int &stages) {
    (void)hidden;
    rows = B >= kQkvRows ? kQkvRows : (B + 15) / 16 * 16;
    boxes = 1;
    stages = kQkvRingBytes / qkv_stage_bytes(rows, boxes);
    if (stages > kQkvMaxStages) stages = kQkvMaxStages;
}

cudaError_t launch_qkv_pack(const __nv_bfloat16 *w, __nv_bfloat16 *w_packed, int rows,
                            int hidden, cudaStream_t s) {
    const int64_t units = static_cast<int64_t>(rows) * hidden / 8;
    const int threads = 256;
    const int blocks = static_cast<int>(std::min<int64_t>((units + threads - 1) / threads, 4096));
    qkv_pack_kernel<<<blocks, threads, 0, s>>>(w, w_packed, rows, hidden);
    return cudaGetLastError();
}

cudaError_t launch_qkv_append(const Params &p, const CUtensorMap &x_map, cudaStream_t s) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 63;
    {
        std::lock_guard<std::mutex> lock(g_qkv_mu);
        if (!g_qkv_smem_set[dev]) {
            cudaError_t e = cudaFuncSetAttribute(
                qkv_append_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kQkvSmemMax);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(qkv_append_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kQkvSmemMax);
            if (e != cudaSuccess) return e;
            g_qkv_smem_set[dev] = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((p.Hq + 2 * p.Hkv) * kQkvCluster, (p.B + kQkvRows - 1) / kQkvRows);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes =
        p.qkv_stages * qkv_stage_bytes(p.qkv_rows, p.qkv_boxes) + kQkvTailBytes + 1024;
    cfg.stream = s;
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = kQkvCluster;
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    int na = 1;
    if (p.pdl) {
        attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    // one 16-row tile: mma.sync; larger batches: tcgen05
    return p.qkv_rows <= 16 ? cudaLaunchKernelEx(&cfg, qkv_append_kernel<false>, x_map, p)
                            : cudaLaunchKernelEx(&cfg, qkv_append_kernel<true>, x_map, p);
}

}  // namespace qdec
