// qdec_prefill.cu -- chunked prefill over the paged pool, on sm_103a.
//
// A chunk of n_b new tokens per sequence (packed rows qo_indptr[b] ..
// qo_indptr[b+1]-1; they become tokens L_b - n_b .. L_b - 1 of the sequence,
// L_b = seq_lens[b] counted after the chunk):
//
// prefill_append_kernel -- steps 1-3 for every chunk token: RMSNorm and NeoX
//   RoPE (at positions[row]) of its query rows into q_rot (fp32) and of its
//   key rows, then bf16(k_rot) and v into slot L_b - n_b + j of the pool.
//   One CTA per token (the angles taken once), one warp per KV head.
//
// prefill_attention_kernel -- causal paged attention of the chunk (article
//   "扔掉 vLLM！从零构建 Qwen3-8B 推理引擎" (news.rkmt.cn), section 4.4.1:
//   FlashAttention-2 prefill, the queries in blocks that each see only the
//   keys at or before them, never forming the whole score matrix).  One CTA
//   per (sequence, KV head, block of 16 chunk tokens), the blocks with the
//   most keys first.  A producer warp streams the sequence's page tiles (K
//   and V of one page and KV head, 8 KiB, one TMA box) up to the block's last
//   query into a ring; each of the four consumer warps owns one query head
//   of the group for the block's 16 tokens and, per tile, forms S = Q K^T
//   with mma.sync (q as bf16 hi + lo, ~16-bit mantissa), masks keys after
//   each query, keeps the online softmax in fp32 (log2 units) and adds
//   P V with P taken straight from the score accumulators as bf16.
//
// Over an FP8 (E4M3) pool the append stores codes, each row element divided
// by its (page, plane, head) scale in fp32 and rounded to nearest-even with
// saturation (the decode step's rule), and the attention brings each page
// tile as codes plus its two scales, converts the codes to bf16 in shared
// memory (exact: every E4M3 value is a bf16 value), multiplies the scores by
// the K scale and folds the V scale into the weights of the value product.
#include "qdec_internal.h"
#include "qdec_ptx.cuh"
#include "qdec_ff.cuh"
#include "qdec_tc.cuh"
#include "qdec.h"

#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>

#include <mutex>

namespace qdec {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kPfRows = 16;                 // chunk tokens per work unit (one m16 tile)
constexpr int kPfStages = 8;                // page tiles in flight per CTA
// shared memory: [ring of page tiles][FP8: scale windows of every slot, two
// converted bf16 tiles][full[8], empty[8], slot_ok[8], the abort flag, the unit]
template <bool kFp8>
__host__ __device__ constexpr int pf_ring_bytes() {
    return kPfStages * (kFp8 ? kFp8TileBytes : kTileBytes);
}
template <bool kFp8>
__host__ __device__ constexpr int pf_extra_bytes() {
    return kFp8 ? kPfStages * kFp8SlotExtra + 2 * kTileBytes : 0;
}
// the tail: full and empty barriers (128 B), slot_ok (32 B), misc (16 B, then
// 16 B unused), the FP8 conversion barriers (32 B), the slot scale indices
// (32 B); plus up to 1 KiB lost aligning the base
constexpr int kPfTailBytes = 2 * kPfStages * 8 + kPfStages * 4 + 32 + 32 + kPfStages * 4;
static_assert(kPfTailBytes == 256, "tail layout");
template <bool kFp8>
__host__ __device__ constexpr int pf_smem_bytes() {
    return pf_ring_bytes<kFp8>() + pf_extra_bytes<kFp8>() + kPfTailBytes + 1024;
}

__device__ __forceinline__ void flag_error(int32_t *err, int bits) {
    if (err) atomicOr(err, bits);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
           (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
}

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t v) {  // exact: bf16 -> fp32
    return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// The sequence b with qo[b] <= r < qo[b+1] when qo is a valid layout (binary
// search; always in [0, B)).
__device__ int seq_of_row(const int32_t *qo, int B, int r) {
    int lo = 0, hi = B;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (qo[mid] <= r)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// Whether sequence b's chunk is well formed: 0 <= n <= L <= max_blocks * P,
// L >= 1, rows inside [0, T).
__device__ __forceinline__ bool chunk_ok(const Params &p, int b, int &n, int &L) {
    const int q0 = p.qo_indptr[b], q1 = p.qo_indptr[b + 1];
    n = q1 - q0;
    L = p.seq_lens[b];
    return q0 >= 0 && q1 <= p.T && n >= 0 && L >= 1 && L <= p.max_blocks * kPageSize && n <= L;
}

// ------------------------------------------------------------------ append --
// One CTA per chunk row, 256 threads: the 64 angles of the row's position are
// taken once (double sincos) into shared memory; warp w then handles KV head
// w (and w + 8, ...): its four query rows in fp32 (q_rot's tolerance is
// absolute), its key row in float-float arithmetic rounded once to bf16 (the
// decode append's rule: the nearest-even bf16 of the exact value), and the
// copy of its value row.
constexpr int kPfAppendThreads = 256;

// E4M3 codes of a / s and b / s (fp32 division, one rounding each, then
// nearest-even with saturation to +-448), a in the low byte.
__device__ __forceinline__ uint16_t quantize_pair_e4m3(float a, float b, float s) {
    return static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(
        make_float2(__fdiv_rn(a, s), __fdiv_rn(b, s)), __NV_SATFINITE, __NV_E4M3));
}

template <bool kFp8>
__global__ void __launch_bounds__(kPfAppendThreads) prefill_append_kernel(
    const __grid_constant__ Params p) {
    __shared__ double cs_d[kRotPairs], sn_d[kRotPairs];
    const int r = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = seq_of_row(p.qo_indptr, p.B, r);
    int n, L;
    if (!chunk_ok(p, b, n, L) || r < p.qo_indptr[b] || r >= p.qo_indptr[b + 1]) {
        if (threadIdx.x == 0) flag_error(p.err, QDEC_FLAG_BAD_SEQLEN);
        return;  // uniform over the CTA
    }
    const int t = L - n + (r - p.qo_indptr[b]);  // token index in the sequence
    if (threadIdx.x < kRotPairs)  // angle i: positions[r] * theta^(-2i/D)
        sincos(static_cast<double>(p.positions[r]) * p.inv_freq[threadIdx.x], &sn_d[threadIdx.x],
               &cs_d[threadIdx.x]);
    __syncthreads();
    // this lane's rotate-half pairs i = 2 lane, 2 lane + 1: dims i and i + 64
    const double c0 = cs_d[2 * lane], c1 = cs_d[2 * lane + 1];
    const double s0 = sn_d[2 * lane], s1 = sn_d[2 * lane + 1];
    const float fc0 = static_cast<float>(c0), fc1 = static_cast<float>(c1);
    const float fs0 = static_cast<float>(s0), fs1 = static_cast<float>(s1);
    // RMSNorm (eps inside the root) of one 128-dim row; x w is exact in fp32
    // (a product of two bf16).  Returns the root; n holds x w for dims
    // 2 lane, 2 lane + 1, 64 + 2 lane, 64 + 2 lane + 1.
    auto norm = [&](const __nv_bfloat16 *x, const __nv_bfloat16 *w, float (&nv)[4]) {
        const float2 a = __bfloat1622float2(reinterpret_cast<const __nv_bfloat162 *>(x)[lane]);
        const float2 c = __bfloat1622float2(reinterpret_cast<const __nv_bfloat162 *>(x + 64)[lane]);
        const float ss = warp_sum(a.x * a.x + a.y * a.y + c.x * c.x + c.y * c.y);
        const float2 wa = __bfloat1622float2(reinterpret_cast<const __nv_bfloat162 *>(w)[lane]);
        const float2 wc = __bfloat1622float2(reinterpret_cast<const __nv_bfloat162 *>(w + 64)[lane]);
        nv[0] = a.x * wa.x;
        nv[1] = a.y * wa.y;
        nv[2] = c.x * wc.x;
        nv[3] = c.y * wc.y;
        return rsqrtf(ss * (1.0f / kHeadDim) + p.eps);
    };
    for (int g = warp; g < p.Hkv; g += kPfAppendThreads / 32) {
#pragma unroll
        for (int j = 0; j < kGroup; ++j) {  // unrolled: the four rows' loads overlap
            const int h = g * kGroup + j;
            float nv[4];
            const float rn = norm(p.q + static_cast<int64_t>(r) * p.q_stride + h * kHeadDim,
                                  p.w_q, nv);
            const float n1a = nv[0] * rn, n1b = nv[1] * rn, n2a = nv[2] * rn, n2b = nv[3] * rn;
            float *dst = p.q_rot_out + (static_cast<int64_t>(r) * p.Hq + h) * kHeadDim;
            reinterpret_cast<float2 *>(dst)[lane] =
                make_float2(n1a * fc0 - n2a * fs0, n1b * fc1 - n2b * fs1);
            reinterpret_cast<float2 *>(dst + 64)[lane] =
                make_float2(n2a * fc0 + n1a * fs0, n2b * fc1 + n1b * fs1);
        }
        const int page = p.block_table[static_cast<int64_t>(b) * p.max_blocks + t / kPageSize];
        if (page < 0 || page >= p.num_pages) {
            if (lane == 0) flag_error(p.err, QDEC_FLAG_BAD_PAGE);
            continue;
        }
        const int64_t slot =
            ((static_cast<int64_t>(page) * 2 * p.Hkv + g) * kPageSize + t % kPageSize) * kHeadDim;
        // the key: norm and rotation in float-float, one rounding to bf16
        const __nv_bfloat16 *krow = p.k + static_cast<int64_t>(r) * p.k_stride + g * kHeadDim;
        const RopeEntry e0 = {fc0, static_cast<float>(c0 - static_cast<double>(fc0)), fs0,
                              static_cast<float>(s0 - static_cast<double>(fs0))};
        const RopeEntry e1 = {fc1, static_cast<float>(c1 - static_cast<double>(fc1)), fs1,
                              static_cast<float>(s1 - static_cast<double>(fs1))};
        __nv_bfloat16 kb[4];
        key_row(p.eps, reinterpret_cast<const __nv_bfloat162 *>(krow)[lane],
                reinterpret_cast<const __nv_bfloat162 *>(krow + 64)[lane],
                reinterpret_cast<const __nv_bfloat162 *>(p.w_k)[lane],
                reinterpret_cast<const __nv_bfloat162 *>(p.w_k + 64)[lane], e0, e1, kb);
        const uint32_t k01 = static_cast<uint32_t>(__bfloat16_as_ushort(kb[0])) |
                             (static_cast<uint32_t>(__bfloat16_as_ushort(kb[1])) << 16);
        const uint32_t k23 = static_cast<uint32_t>(__bfloat16_as_ushort(kb[2])) |
                             (static_cast<uint32_t>(__bfloat16_as_ushort(kb[3])) << 16);
        const uint32_t *vs = reinterpret_cast<const uint32_t *>(
            p.v + static_cast<int64_t>(r) * p.v_stride + g * kHeadDim);
        const uint32_t v01 = vs[lane], v23 = vs[32 + lane];
        const int64_t vslot = slot + static_cast<int64_t>(p.Hkv) * kPageSize * kHeadDim;
        if constexpr (kFp8) {
            // the bf16 rows the bf16 pool would hold, divided by the scales
            const int64_t si = static_cast<int64_t>(page) * 2 * p.Hkv + g;
            const float sk = p.kv_scale[si], sv = p.kv_scale[si + p.Hkv];
            const float2 ka = bf16x2_to_float2(k01), kc = bf16x2_to_float2(k23);
            const float2 va = bf16x2_to_float2(v01), vc = bf16x2_to_float2(v23);
            uint16_t *kd = reinterpret_cast<uint16_t *>(p.pool8 + slot);
            uint16_t *vd = reinterpret_cast<uint16_t *>(p.pool8 + vslot);
            kd[lane] = quantize_pair_e4m3(ka.x, ka.y, sk);
            kd[32 + lane] = quantize_pair_e4m3(kc.x, kc.y, sk);
            vd[lane] = quantize_pair_e4m3(va.x, va.y, sv);
            vd[32 + lane] = quantize_pair_e4m3(vc.x, vc.y, sv);
        } else {
            uint32_t *kd = reinterpret_cast<uint32_t *>(p.pool + slot);
            uint32_t *vd = reinterpret_cast<uint32_t *>(p.pool + vslot);
            kd[lane] = k01;
            kd[32 + lane] = k23;
            vd[lane] = v01;
            vd[32 + lane] = v23;
        }
    }
}

// --------------------------------------------------------------- attention --
// One page tile (K and V of one page and KV head, 8 KiB): the pool's 5-D
// tensor map (64 dims, 16 tokens, 2 halves of D, K/V plane, page*2*Hkv +
// head) lands it as [plane][half][token][64 dims], 128-byte rows swizzled by
// (token % 8).
__device__ __forceinline__ void tma_load_page_tile(uint32_t dst, const CUtensorMap *map,
                                                   int plane_row, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %2, %2, %2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(plane_row), "r"(bar)
        : "memory");
}

// One FP8 page tile: [plane][token][128 bytes of D], 4 KiB, 128-byte
// swizzled rows (the pool's 4-D tensor map: bytes of D, token, plane,
// page*2*Hkv + head).
__device__ __forceinline__ void tma_load_page_tile_fp8(uint32_t dst, const CUtensorMap *map,
                                                       int plane_row, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %2, %2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(plane_row), "r"(bar)
        : "memory");
}

// Two E4M3 codes (low byte first) as a bf16 pair: exact (every E4M3 value
// is a bf16 value; NaN stays NaN).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two_codes) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(
        static_cast<__nv_fp8x2_storage_t>(two_codes & 0xFFFFu), __NV_E4M3);
    const float lo = __half2float(__half(__half_raw{h.x}));
    const float hi = __half2float(__half(__half_raw{h.y}));
    return (__float_as_uint(lo) >> 16) | (__float_as_uint(hi) & 0xffff0000u);
}

template <bool kFp8>
__global__ void __launch_bounds__(kThreads, 2)
    prefill_attention_kernel(const __grid_constant__ CUtensorMap kv_map,
                             const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int kSlot = kFp8 ? kFp8TileBytes : kTileBytes;  // ring slot
    // FP8: after the ring, the scale windows of every slot, then two bf16
    // tiles the codes are converted into
    uint8_t *extra = sm + pf_ring_bytes<kFp8>();
    uint8_t *conv = extra + kPfStages * kFp8SlotExtra;
    uint8_t *tail = extra + pf_extra_bytes<kFp8>();
    const uint32_t full0 = smem_u32(tail);
    const uint32_t empty0 = full0 + kPfStages * 8;
    volatile int *slot_ok = reinterpret_cast<volatile int *>(tail + 2 * kPfStages * 8);
    volatile int *misc = reinterpret_cast<volatile int *>(tail + 2 * kPfStages * 8 + kPfStages * 4);
    // misc: [0] abort, [1] sequence, [2] query block, [3] pages issued;
    // FP8: [4] conv_full[2], conv_empty[2] barriers (8-byte aligned), then
    // the scale index of every slot
    const uint32_t convb0 = smem_u32(tail + 2 * kPfStages * 8 + kPfStages * 4 + 32);
    volatile int *slot_si =
        reinterpret_cast<volatile int *>(tail + 2 * kPfStages * 8 + kPfStages * 4 + 64);
    const int g = blockIdx.x % p.Hkv;
    const int unit = blockIdx.x / p.Hkv;

    // ---- which (sequence, block) this CTA takes: units enumerate every
    // sequence's blocks from its last (most keys) to its first
    if (warp == 0) {
        const int per = (p.B + 31) / 32;
        int cnt = 0;
        for (int i = 0; i < per; ++i) {
            const int b = lane * per + i;
            int n, L;
            if (b < p.B && chunk_ok(p, b, n, L)) cnt += (n + kPfRows - 1) / kPfRows;
        }
        int incl = cnt;  // inclusive prefix over the lanes
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += v;
        }
        const int excl = incl - cnt;
        if (lane == 0) misc[1] = -1;
        __syncwarp();
        if (unit >= excl && unit < incl) {
            int k = unit - excl;
            for (int i = 0; i < per; ++i) {
                const int b = lane * per + i;
                int n, L;
                if (b >= p.B || !chunk_ok(p, b, n, L)) continue;
                const int nb = (n + kPfRows - 1) / kPfRows;
                if (k < nb) {
                    misc[1] = b;
                    misc[2] = nb - 1 - k;
                    break;
                }
                k -= nb;
            }
        }
        if (blockIdx.x == 0) {  // report malformed chunks once
            for (int b = lane; b < p.B; b += 32) {
                int n, L;
                if (!chunk_ok(p, b, n, L)) flag_error(p.err, QDEC_FLAG_BAD_SEQLEN);
            }
        }
        if (tid == 0) {
            for (int s = 0; s < kPfStages; ++s) {
                mbar_init(full0 + 8 * s, 1);
                mbar_init(empty0 + 8 * s, kConsumerWarps);  // every warp reads every tile
            }
            if (kFp8)
                for (int i = 0; i < 4; ++i) mbar_init(convb0 + 8 * i, kConsumerWarps);
            misc[0] = 0;
            misc[3] = 0;
            misc[5] = 0;
            fence_mbar_init();
        }
    }
    __syncthreads();
    const int b = misc[1];
    if (b < 0) return;  // no unit for this CTA (the grid is an upper bound)
    const int qb = misc[2];
    int n, L;
    chunk_ok(p, b, n, L);
    const int row0 = p.qo_indptr[b] + qb * kPfRows;             // first packed row
    const int nrows = min(kPfRows, n - qb * kPfRows);           // rows of this block
    const int t0 = L - n + qb * kPfRows;                        // token index of row 0
    const int npages = (t0 + nrows - 1) / kPageSize + 1;        // pages up to the last query

    if (warp == kConsumerWarps) {
        // ------------------------------------------------ TMA producer --
        uint32_t i = 0;
        bool stop = false;
        for (int base = 0; base < npages && !stop; base += 32) {
            int page = -1;
            if (base + lane < npages)
                page = p.block_table[static_cast<int64_t>(b) * p.max_blocks + base + lane];
            const int cnt = min(32, npages - base);
            for (int j = 0; j < cnt; ++j, ++i) {
                const int pj = __shfl_sync(kFull, page, j);
                if (lane == 0) {
                    const int slot = i % kPfStages;
                    const uint32_t full = full0 + 8 * slot;
                    if (misc[0]) {
                        stop = true;
                    } else if (i >= static_cast<uint32_t>(kPfStages) &&
                               !mbar_wait_bounded(empty0 + 8 * slot, ((i / kPfStages) - 1) & 1,
                                                  misc, p.wait_cycles)) {
                        misc[0] = 1;
                        flag_error(p.err, QDEC_FLAG_TIMEOUT);
                        stop = true;
                    } else if (p.withhold_first && i == 0) {
                        // test hook: this tile's barrier phase never completes
                    } else if (pj >= 0 && pj < p.num_pages) {
                        slot_ok[slot] = 1;
                        if constexpr (kFp8) {
                            // the tile and the two 16-byte windows of kv_scale
                            // holding its K and V scales (Hkv even: a window
                            // never straddles pages)
                            const int64_t si = static_cast<int64_t>(pj) * 2 * p.Hkv + g;
                            slot_si[slot] = static_cast<int>(((si & 3) | (((si + p.Hkv) & 3) << 2)));
                            const uint32_t win = smem_u32(extra + slot * kFp8SlotExtra);
                            mbar_arrive_expect_tx(full, kFp8TileBytes + kFp8SlotExtra);
                            tma_load_page_tile_fp8(smem_u32(sm + slot * kSlot), &kv_map,
                                                   pj * 2 * p.Hkv + g, full);
                            bulk_load(win, p.kv_scale + (si & ~3ll), kScaleWindowBytes, full);
                            bulk_load(win + kScaleWindowBytes, p.kv_scale + ((si + p.Hkv) & ~3ll),
                                      kScaleWindowBytes, full);
                        } else {
                            mbar_arrive_expect_tx(full, kTileBytes);
                            tma_load_page_tile(smem_u32(sm + slot * kSlot), &kv_map,
                                               pj * 2 * p.Hkv + g, full);
                        }
                    } else {
                        slot_ok[slot] = 0;
                        flag_error(p.err, QDEC_FLAG_BAD_PAGE);
                        mbar_arrive(full);
                    }
                }
                stop = __shfl_sync(kFull, stop, 0);
                if (stop) break;
            }
        }
        if (lane == 0) misc[3] = static_cast<int>(i);
    } else {
        // ------------------------------------------- consumer warps --
        const int h = g * kGroup + warp;
        const int gq = lane >> 2, tq = lane & 3;  // fragment row group, column pair
        // Q fragments (A of m16n8k16, 16 tokens x 128 dims in 8 k-steps),
        // scaled to log2 units, as bf16 hi + lo
        uint32_t qh[8][4], ql[8][4];
        {
            const float *q0 = p.q_rot_in + (static_cast<int64_t>(row0 + gq) * p.Hq + h) * kHeadDim;
            const float *q1 = q0 + 8 * static_cast<int64_t>(p.Hq) * kHeadDim;
            const bool v0 = gq < nrows, v1 = gq + 8 < nrows;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float *src = (e & 1) ? q1 : q0;
                    const bool valid = (e & 1) ? v1 : v0;
                    const int col = 16 * kk + 2 * tq + ((e >> 1) << 3);
                    float2 x = valid ? *reinterpret_cast<const float2 *>(src + col)
                                     : make_float2(0.f, 0.f);
                    x.x *= p.qscale;
                    x.y *= p.qscale;
                    const __nv_bfloat16 hx = __float2bfloat16_rn(x.x), hy = __float2bfloat16_rn(x.y);
                    qh[kk][e] = static_cast<uint32_t>(__bfloat16_as_ushort(hx)) |
                                (static_cast<uint32_t>(__bfloat16_as_ushort(hy)) << 16);
                    ql[kk][e] = pack_bf16x2(x.x - __bfloat162float(hx), x.y - __bfloat162float(hy));
                }
            }
        }
        // the last key each of this thread's two rows may see (causal, and
        // never past the sequence)
        const int lim0 = min(t0 + gq, L - 1), lim1 = min(t0 + gq + 8, L - 1);
        float o[16][4];
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        const int mi = lane >> 3, r8 = lane & 7;
        // this lane's matrix-load offsets within a tile: K (keys (mi >> 1) * 8
        // + r8, dim chunk 2 kk + (mi & 1)) and V (keys (mi & 1) * 8 + r8, dim
        // chunk 2 pr + (mi >> 1)), for chunk pairs j = kk, pr mod 4 (the
        // halves of D add 2 KiB)
        uint32_t koff[4], voff[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int kt = (mi >> 1) * 8 + r8, vt = (mi & 1) * 8 + r8;
            koff[j] = kt * 128 + (((2 * j + (mi & 1)) ^ (kt & 7)) << 4);
            voff[j] = kPlaneBytes + vt * 128 + (((2 * j + (mi >> 1)) ^ (vt & 7)) << 4);
        }
        bool aborted = false;
        for (int pg = 0; pg < npages; ++pg) {
            const int slot = pg % kPfStages;
            if (!mbar_wait_bounded(full0 + 8 * slot, (pg / kPfStages) & 1, misc, p.wait_cycles)) {
                if (lane == 0) {
                    misc[0] = 1;
                    flag_error(p.err, QDEC_FLAG_TIMEOUT);
                }
                aborted = true;
                break;
            }
            const bool ok = slot_ok[slot];
            uint32_t tile = smem_u32(sm + slot * kSlot);
            float sk = 1.f, sv = 1.f;  // FP8: the tile's K and V scales
            if constexpr (kFp8) {
                // convert this warp's quarter of the codes into buffer pg & 1
                // (once its previous tile has been read by every warp), hand
                // the ring slot back, wait for the other quarters
                const int cb = pg & 1;
                if (pg >= 2 && !mbar_wait_bounded(convb0 + 8 * (2 + cb), ((pg >> 1) - 1) & 1,
                                                  misc, p.wait_cycles)) {
                    if (lane == 0) {
                        misc[0] = 1;
                        flag_error(p.err, QDEC_FLAG_TIMEOUT);
                    }
                    aborted = true;
                    break;
                }
                uint8_t *cvt = conv + cb * kTileBytes;
                if (ok) {
                    const int si = slot_si[slot];
                    const float *win = reinterpret_cast<const float *>(extra + slot * kFp8SlotExtra);
                    sk = win[si & 3];
                    sv = win[4 + (si >> 2)];
#pragma unroll
                    for (int it = 0; it < 2; ++it) {
                        // item: plane, token, 16 codes of dims 16 c .. 16 c + 15
                        const int item = (warp * 32 + lane) + 128 * it;
                        const int plane = item >> 7, tok = (item >> 3) & 15, c = item & 7;
                        const uint4 codes = *reinterpret_cast<const uint4 *>(
                            sm + slot * kSlot + plane * kFp8PlaneBytes + tok * 128 +
                            ((c ^ (tok & 7)) << 4));
                        const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
                        uint32_t bf[8];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            bf[2 * q] = e4m3x2_to_bf16x2(w[q]);
                            bf[2 * q + 1] = e4m3x2_to_bf16x2(w[q] >> 16);
                        }
                        // bf16 chunks 2c, 2c + 1 of the token: half c / 4
                        uint8_t *dst = cvt + plane * kPlaneBytes + (c >> 2) * kTileHalfBytes + tok * 128;
                        *reinterpret_cast<uint4 *>(dst + ((((2 * c) & 7) ^ (tok & 7)) << 4)) =
                            make_uint4(bf[0], bf[1], bf[2], bf[3]);
                        *reinterpret_cast<uint4 *>(dst + ((((2 * c + 1) & 7) ^ (tok & 7)) << 4)) =
                            make_uint4(bf[4], bf[5], bf[6], bf[7]);
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(empty0 + 8 * slot);     // the codes are no longer needed
                    mbar_arrive(convb0 + 8 * cb);       // this warp's quarter is in place
                }
                if (!mbar_wait_bounded(convb0 + 8 * cb, (pg >> 1) & 1, misc, p.wait_cycles)) {
                    if (lane == 0) {
                        misc[0] = 1;
                        flag_error(p.err, QDEC_FLAG_TIMEOUT);
                    }
                    aborted = true;
                    break;
                }
                tile = smem_u32(cvt);
            }
            if (ok) {
                // ---- S = Q K^T: 16 tokens x 16 keys (two n-tiles of 8 keys)
                // (the hi and lo products in separate accumulators: four
                // independent chains of 8 MMAs instead of two of 16)
                float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                float sl[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    uint32_t kb[4];
                    // matrices: keys 0-7 / 8-15 (mi >> 1) x dims 16kk.. / 16kk+8.. (mi & 1)
                    ldmatrix_x4(kb, tile + (kk >> 2) * kTileHalfBytes + koff[kk & 3]);
                    mma_bf16(s[0], qh[kk], kb[0], kb[1]);
                    mma_bf16(s[1], qh[kk], kb[2], kb[3]);
                    mma_bf16(sl[0], ql[kk], kb[0], kb[1]);
                    mma_bf16(sl[1], ql[kk], kb[2], kb[3]);
                }
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) s[j][e] = (s[j][e] + sl[j][e]) * sk;
                // ---- causal mask: key 16 pg + 8 j + 2 tq + e against each
                // row's limit (only tiles that reach past a limit need it)
                const int kbase = pg * kPageSize + 2 * tq;
                if (pg * kPageSize + kPageSize - 1 > lim0) {
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int key = kbase + 8 * j + e;
                            if (key > lim0) s[j][e] = -INFINITY;
                            if (key > lim1) s[j][2 + e] = -INFINITY;
                        }
                    }
                }
                // ---- online softmax (log2 units), rows gq and gq + 8.  The
                // running maximum is kept until a tile's maximum exceeds it
                // by more than 2^8 (weights then stay below 256, exact enough
                // in bf16 and fp32), so most tiles rescale nothing.
                float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
                float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
#pragma unroll
                for (int off = 1; off < 4; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, off));
                }
                // a row that has seen no key yet keeps m = -inf, weights 0
                if (mx0 > m0 + 8.f || mx1 > m1 + 8.f) {
                    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
                    const float a0 = n0 == -INFINITY ? 1.f : exp2f(m0 - n0);
                    const float a1 = n1 == -INFINITY ? 1.f : exp2f(m1 - n1);
                    l0 *= a0;
                    l1 *= a1;
                    m0 = n0;
                    m1 = n1;
#pragma unroll
                    for (int nt = 0; nt < 16; ++nt) {
                        o[nt][0] *= a0;
                        o[nt][1] *= a0;
                        o[nt][2] *= a1;
                        o[nt][3] *= a1;
                    }
                }
                float pw[2][4];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        pw[j][e] = m0 == -INFINITY ? 0.f : exp2f(s[j][e] - m0);
                        pw[j][2 + e] = m1 == -INFINITY ? 0.f : exp2f(s[j][2 + e] - m1);
                    }
                }
                l0 += pw[0][0] + pw[0][1] + pw[1][0] + pw[1][1];
                l1 += pw[0][2] + pw[0][3] + pw[1][2] + pw[1][3];
                // ---- O += P V: P (16 tokens x 16 keys) from the score
                // accumulators as the A operand; V rows past the sequence
                // (possibly not finite) are zeroed in the B fragments
                // (FP8: the V scale folded into the weights)
                uint32_t pa[4];
                pa[0] = pack_bf16x2(pw[0][0] * sv, pw[0][1] * sv);
                pa[1] = pack_bf16x2(pw[0][2] * sv, pw[0][3] * sv);
                pa[2] = pack_bf16x2(pw[1][0] * sv, pw[1][1] * sv);
                pa[3] = pack_bf16x2(pw[1][2] * sv, pw[1][3] * sv);
                const int ntok = min(kPageSize, L - pg * kPageSize);  // keys of this page in the sequence
                // this thread's B elements hold keys 2 tq, 2 tq + 1 (b0) and +8 (b1)
                const uint32_t keep0 = (2 * tq < ntok ? 0x0000ffffu : 0u) |
                                       (2 * tq + 1 < ntok ? 0xffff0000u : 0u);
                const uint32_t keep1 = (2 * tq + 8 < ntok ? 0x0000ffffu : 0u) |
                                       (2 * tq + 9 < ntok ? 0xffff0000u : 0u);
#pragma unroll
                for (int pr = 0; pr < 8; ++pr) {
                    uint32_t vb[4];
                    // matrices: keys 0-7 / 8-15 (mi & 1) x dims 16pr.. / 16pr+8.. (mi >> 1)
                    ldmatrix_x4_trans(vb, tile + (pr >> 2) * kTileHalfBytes + voff[pr & 3]);
                    if (ntok < kPageSize) {  // the sequence's last page
                        vb[0] &= keep0;
                        vb[1] &= keep1;
                        vb[2] &= keep0;
                        vb[3] &= keep1;
                    }
                    mma_bf16(o[2 * pr], pa, vb[0], vb[1]);
                    mma_bf16(o[2 * pr + 1], pa, vb[2], vb[3]);
                }
            }
            __syncwarp();
            if (lane == 0) {
                if (kFp8)
                    mbar_arrive(convb0 + 8 * (2 + (pg & 1)));  // buffer pg & 1 read
                else
                    mbar_arrive(empty0 + 8 * slot);
            }
        }
        // ---- normalise and write the block's rows of head h
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
            l0 += __shfl_xor_sync(kFull, l0, off);
            l1 += __shfl_xor_sync(kFull, l1, off);
        }
        if (!aborted && !misc[0]) {
            const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
            __nv_bfloat16 *d0 = p.out + (static_cast<int64_t>(row0 + gq) * p.Hq + h) * kHeadDim;
            __nv_bfloat16 *d1 = d0 + 8 * static_cast<int64_t>(p.Hq) * kHeadDim;
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                const int col = 8 * nt + 2 * tq;
                if (gq < nrows)
                    *reinterpret_cast<uint32_t *>(d0 + col) = pack_bf16x2(o[nt][0] * i0, o[nt][1] * i0);
                if (gq + 8 < nrows)
                    *reinterpret_cast<uint32_t *>(d1 + col) = pack_bf16x2(o[nt][2] * i1, o[nt][3] * i1);
            }
        }
    }
    __syncthreads();
    // a wait that gave up may leave copies in flight: let them land (bounded)
    if (tid == 0 && misc[0]) {
        const uint32_t issued = static_cast<uint32_t>(misc[3]);
        const uint32_t first = issued > static_cast<uint32_t>(kPfStages) ? issued - kPfStages : 0;
        volatile int never = 0;
        for (uint32_t t = first; t < issued; ++t)
            mbar_wait_bounded(full0 + 8 * (t % kPfStages), (t / kPfStages) & 1, &never,
                              p.wait_cycles);
    }
}

// ------------------------------------- attention on the 5th-gen tensor core --
// prefill_attention_tc_kernel: the same causal paged attention (bf16 pool)
// with both products on the tensor core (tcgen05, accumulators in tensor
// memory).  One CTA per (sequence, KV head, block of 64 chunk tokens), the
// blocks with the most keys first.  The block is two tiles of M = 128 rows:
// tile u holds tokens 32 u .. 32 u + 31 of the block for the 4 query heads
// of the group (row 32 j + i: head 4 g + j, token 32 u + i), so each K/V
// stage in shared memory serves 256 query rows.  Per stage of 64 keys (4
// pages) one producer warp brings K and another V, each into its own ring,
// as two 8 KiB regions [dims 0-63][dims 64-127] of [64 keys][128 bytes],
// 128-byte swizzled (one 2 KiB TMA box per page and region): a K slot is
// refilled as soon as the stage's score products are done, while V is only
// needed by the value products, one softmax later.  For each tile, from its
// own issuing thread (warps 9 and 11),
//   S = Q K^T  (M 128, N 64, K 128: 8 MMAs of K 16; Q and K both K-major;
//               q enters as bf16),
//   O += P V   (M 128, N 128, K 64: 4 MMAs; P read from tensor memory, V
//               read in place from shared memory as an MN-major operand).
// S is double-buffered in tensor memory per tile, so the scores of stage
// j + 1 are formed while the softmax warps (warps 4 u .. 4 u + 3 for tile u,
// thread r of the group owning row r, its tensor-memory lane) work on stage
// j: load the 64 scores, mask keys past each row's token, keep a stale
// running maximum (O in tensor memory is rescaled only when a stage's
// maximum exceeds it by more than 2^8, so the weights stay below 256), and
// write P as bf16 into tensor memory over the scores just read.  V rows of
// keys past the sequence (or of pages not brought) are zeroed before a value
// product reads them.  The epilogue reads O out of tensor memory, divides by
// the row sum and stores the row.  Every wait is bounded; the decisions that
// lead to warp-collective tensor-memory loads and stores are warp-uniform.
constexpr int kTcTiles = 2;                                // query tiles per CTA
constexpr int kTcTileTok = 32;                             // chunk tokens per tile
constexpr int kTcTok = kTcTiles * kTcTileTok;              // chunk tokens per CTA
constexpr int kTcRows = kTcTileTok * kGroup;               // M = 128 rows per tile
constexpr int kTcKeys = 64;                                // keys per stage
constexpr int kTcPagesPerStage = kTcKeys / kPageSize;      // 4
constexpr int kTcStages = 4;
constexpr int kTcRegion = kTcKeys * 128;                   // [64 keys][64 dims] bf16, 8 KiB
constexpr int kTcSlotBytes = 2 * kTcRegion;                // K (or V): dims 0-63, dims 64-127
constexpr int kTcQHalf = kTcRows * 128;                    // [128 rows][64 dims] bf16, 16 KiB
constexpr int kTcQBytes = 2 * kTcQHalf;                    // one tile's Q
constexpr int kTcOffQ = 0;                                 // Q of tile u at u * kTcQBytes
constexpr int kTcOffKRing = kTcOffQ + kTcTiles * kTcQBytes;
constexpr int kTcOffVRing = kTcOffKRing + kTcStages * kTcSlotBytes;
constexpr int kTcOffTail = kTcOffVRing + kTcStages * kTcSlotBytes;
// tail: barriers k_full[S], k_empty[S], v_full[S], v_empty[S]; per tile
// s_full[2], (unused)[2], p_full[2], o_done[2]; q_ready, done; then ints:
// abort, sequence, block, K stages issued, tensor-memory address, V stages
// issued, and the mask of pages brought into every V slot
constexpr int kTcBars = 4 * kTcStages + kTcTiles * 8 + 2;
constexpr int kTcTailBytes = kTcBars * 8 + (6 + kTcStages) * 4;
constexpr int kTcSmemBytes = kTcOffTail + kTcTailBytes + 1024;
constexpr int kTcSoftmaxWarps = 4 * kTcTiles;
constexpr int kTcProducerWarp = kTcSoftmaxWarps;           // K stages
constexpr int kTcMmaWarp = kTcSoftmaxWarps + 1;
constexpr int kTcVProducerWarp = kTcSoftmaxWarps + 2;      // V stages
constexpr int kTcMmaWarp1 = kTcSoftmaxWarps + 3;           // tile 1's products (tile 0: kTcMmaWarp)
constexpr int kTcThreads = (kTcSoftmaxWarps + 4) * 32;
// tile u: S buffers at columns 256 u + {0, 64}, O at 256 u + 128
constexpr uint32_t kTcTmemCols = 256 * kTcTiles;
static_assert(kTcSmemBytes <= 227 * 1024, "one CTA per SM");
static_assert(kTcOffKRing % 1024 == 0 && kTcOffVRing % 1024 == 0,
              "swizzled operands start on 1024-byte boundaries");
static_assert(kTcTmemCols <= 512, "tensor memory");

// One (page, plane, half of D) region of a page: 16 tokens x 64 dims, 2 KiB,
// with the pool's region map (5-D: 64 dims, token, half, plane, page*2*Hkv +
// head; box 64 x 16 x 1 x 1 x 1).
__device__ __forceinline__ void tma_load_region(uint32_t dst, const CUtensorMap *map, int half,
                                                int plane, int row, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(half), "r"(plane), "r"(row), "r"(bar)
        : "memory");
}

// 2^x by the hardware's approximation (one instruction; relative error
// about 2^-22, far below the bf16 rounding of the weights it feeds;
// 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Offset of 16-byte chunk c of row r in a [rows][128 bytes] 128-byte
// swizzled block starting on a 1024-byte boundary.
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
    return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_attention_tc_kernel(const __grid_constant__ CUtensorMap region_map,
                                const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint8_t *tail = sm + kTcOffTail;
    const uint32_t k_full0 = smem_u32(tail);
    const uint32_t k_empty0 = k_full0 + 8 * kTcStages;
    const uint32_t v_full0 = k_empty0 + 8 * kTcStages;
    const uint32_t v_empty0 = v_full0 + 8 * kTcStages;
    // per tile u: s_full, p_full, o_done, two of each (buffer q)
    const uint32_t tile_bar0 = v_empty0 + 8 * kTcStages;
    auto s_full = [&](int u, int q) { return tile_bar0 + 64 * u + 8 * q; };
    auto p_full = [&](int u, int q) { return tile_bar0 + 64 * u + 32 + 8 * q; };
    auto o_done = [&](int u, int q) { return tile_bar0 + 64 * u + 48 + 8 * q; };
    const uint32_t q_ready = tile_bar0 + 64 * kTcTiles;
    const uint32_t done_bar = q_ready + 8;
    // misc: [0] abort, [1] sequence, [2] query block, [3] K stages issued,
    // [4] tensor-memory address, [5] V stages issued; pmask[s]: pages
    // brought into V slot s
    volatile int *misc = reinterpret_cast<volatile int *>(tail + kTcBars * 8);
    volatile int *pmask = misc + 6;
    const int g = blockIdx.x % p.Hkv;
    const int unit = blockIdx.x / p.Hkv;
    if (p.pdl && tid == 0) launch_dependents();

    // ---- which (sequence, block) this CTA takes: units enumerate every
    // sequence's blocks from its last (most keys) to its first
    if (warp == 0) {
        const int per = (p.B + 31) / 32;
        int cnt = 0;
        for (int i = 0; i < per; ++i) {
            const int b = lane * per + i;
            int n, L;
            if (b < p.B && chunk_ok(p, b, n, L)) cnt += (n + kTcTok - 1) / kTcTok;
        }
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += v;
        }
        const int excl = incl - cnt;
        if (lane == 0) misc[1] = -1;
        __syncwarp();
        if (unit >= excl && unit < incl) {
            int k = unit - excl;
            for (int i = 0; i < per; ++i) {
                const int b = lane * per + i;
                int n, L;
                if (b >= p.B || !chunk_ok(p, b, n, L)) continue;
                const int nb = (n + kTcTok - 1) / kTcTok;
                if (k < nb) {
                    misc[1] = b;
                    misc[2] = nb - 1 - k;
                    break;
                }
                k -= nb;
            }
        }
        if (blockIdx.x == 0) {  // report malformed chunks once
            for (int b = lane; b < p.B; b += 32) {
                int n, L;
                if (!chunk_ok(p, b, n, L)) flag_error(p.err, QDEC_FLAG_BAD_SEQLEN);
            }
        }
        if (lane == 0) {
            for (int s = 0; s < kTcStages; ++s) {
                mbar_init(k_full0 + 8 * s, 1);    // the K producer's arrival + the bytes
                mbar_init(k_empty0 + 8 * s, kTcTiles);  // each tile's commit of its score product
                mbar_init(v_full0 + 8 * s, 1);    // the V producer's arrival + the bytes
                mbar_init(v_empty0 + 8 * s, kTcTiles);  // each tile's commit of its value product
            }
            for (int u = 0; u < kTcTiles; ++u) {
                for (int q = 0; q < 2; ++q) {
                    mbar_init(s_full(u, q), 1);   // commit of the score product
                    mbar_init(p_full(u, q), 4);   // the tile's softmax warps have written P
                    mbar_init(o_done(u, q), 1);   // commit of the value product
                }
            }
            mbar_init(q_ready, kTcSoftmaxWarps);
            mbar_init(done_bar, kTcTiles);  // each MMA issuer, once its products are done
            misc[0] = 0;
            misc[3] = 0;
            fence_mbar_init();
        }
    }
    if (warp == kTcMmaWarp) tc::alloc(smem_u32(const_cast<int *>(misc + 4)), kTcTmemCols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = static_cast<uint32_t>(misc[4]);
    const int b = misc[1];
    if (b < 0) {  // no unit for this CTA (the grid is an upper bound)
        if (warp == kTcMmaWarp) tc::dealloc(tmem, kTcTmemCols);
        return;
    }
    const int qb = misc[2];
    int n, L;
    chunk_ok(p, b, n, L);
    const int row0 = p.qo_indptr[b] + qb * kTcTok;       // first packed row
    const int nrows = min(kTcTok, n - qb * kTcTok);      // rows of this block
    const int t0 = L - n + qb * kTcTok;                  // token index of row 0
    const int ntiles = (t0 + nrows - 1) / kTcKeys + 1;   // stages up to the last query
    const int npg = (L + kPageSize - 1) / kPageSize;     // pages of the sequence

    if (warp == kTcProducerWarp || warp == kTcVProducerWarp) {
        // ----------------------------------------------- TMA producers --
        // One warp brings the K halves of every stage, the other the V
        // halves, each into its own ring: a K slot frees as soon as the
        // stage's score products are done, a V slot once its value products
        // are.  Lanes 0-3 each bring one page of the stage (its two regions);
        // the block-table entries are looked up 32 pages (8 stages) at a time,
        // one group ahead.
        const bool isv = warp == kTcVProducerWarp;
        const uint32_t full0 = isv ? v_full0 : k_full0;
        const uint32_t empty0 = isv ? v_empty0 : k_empty0;
        uint8_t *ringp = sm + (isv ? kTcOffVRing : kTcOffKRing);
        int issued = 0;
        auto lookup = [&](int grp) {  // lane l: page index 32 grp + l of the sequence
            const int pg = 32 * grp + lane;
            return pg < npg ? p.block_table[static_cast<int64_t>(b) * p.max_blocks + pg] : -1;
        };
        int cur = lookup(0), nxt = lookup(1);
        // the chunk's keys and values were appended by the kernel before
        if (p.pdl) grid_dependency_wait();
        for (int j = 0; j < ntiles; ++j) {
            const int s = j % kTcStages;
            if (j > 0 && (j * kTcPagesPerStage) % 32 == 0) {
                cur = nxt;
                nxt = lookup(j * kTcPagesPerStage / 32 + 1);
            }
            bool stop = false;
            if (lane == 0) {
                if (misc[0]) {
                    stop = true;
                } else if (j >= kTcStages &&
                           !mbar_wait_bounded(empty0 + 8 * s, ((j / kTcStages) - 1) & 1, misc,
                                              p.wait_cycles)) {
                    misc[0] = 1;
                    flag_error(p.err, QDEC_FLAG_TIMEOUT);
                    stop = true;
                }
            }
            if (__shfl_sync(kFull, stop, 0)) break;
            const int pg = j * kTcPagesPerStage + lane;
            const int page = __shfl_sync(kFull, cur, (j * kTcPagesPerStage + (lane & 3)) & 31);
            const bool ok = lane < kTcPagesPerStage && pg < npg && page >= 0 && page < p.num_pages;
            if (!isv && lane < kTcPagesPerStage && pg < npg && !ok) flag_error(p.err, QDEC_FLAG_BAD_PAGE);
            const unsigned mask = __ballot_sync(kFull, ok) & 0xFu;
            const bool withheld = !isv && p.withhold_first && j == 0;  // test hook: never lands
            if (lane == 0) {
                if (isv) pmask[s] = static_cast<int>(mask);
                if (!withheld) {
                    if (mask == 0)
                        mbar_arrive(full0 + 8 * s);
                    else
                        mbar_arrive_expect_tx(full0 + 8 * s, __popc(mask) * 2 * (kPageSize * 128));
                }
            }
            __syncwarp();
            if (ok && !withheld) {
                const uint32_t dst = smem_u32(ringp + s * kTcSlotBytes) + lane * (kPageSize * 128);
                const int row = page * 2 * p.Hkv + g;
#pragma unroll
                for (int h = 0; h < 2; ++h)  // region h: dims 64 h .. 64 h + 63 of the plane
                    tma_load_region(dst + h * kTcRegion, &region_map, h, isv ? 1 : 0, row,
                                    full0 + 8 * s);
            }
            issued = j + 1;
        }
        if (lane == 0) misc[isv ? 5 : 3] = issued;
    } else if (warp == kTcMmaWarp || warp == kTcMmaWarp1) {
        // ------------------------------------------- the MMA issuers --
        // one thread per query tile issues its products, so neither tile
        // waits for the other's softmax; the two meet only in the K and V
        // rings, whose slots free once both tiles' commits have arrived
        if (lane == 0) {
            const int u = warp == kTcMmaWarp ? 0 : 1;
            const uint32_t qt = smem_u32(sm + kTcOffQ) + u * kTcQBytes;
            const uint32_t kring = smem_u32(sm + kTcOffKRing), vring = smem_u32(sm + kTcOffVRing);
            constexpr uint32_t kIdS = tc::idesc_bf16(kTcRows, kTcKeys, false);
            constexpr uint32_t kIdO = tc::idesc_bf16(kTcRows, kHeadDim, true);
            const uint32_t tile_tm = tmem + 256 * u;
            // O += P_t V_t once V_t has landed and the tile's softmax warps
            // have written P (over the scores of stage t, in tensor memory);
            // the commits free that buffer for the scores of stage t + 2
            // (o_done) and, with the other tile's, the V slot (v_empty)
            auto value_product = [&](int t) -> bool {
                if (!mbar_wait_bounded(v_full0 + 8 * (t % kTcStages), (t / kTcStages) & 1, misc,
                                       p.wait_cycles) ||
                    !mbar_wait_bounded(p_full(u, t & 1), (t >> 1) & 1, misc, p.wait_cycles))
                    return false;
                tc::fence_after();
                const uint32_t vst = vring + (t % kTcStages) * kTcSlotBytes;
                const uint32_t tp = tile_tm + (t & 1) * kTcKeys;  // P: 32 columns
#pragma unroll
                for (int kk = 0; kk < kTcKeys / 16; ++kk)
                    tc::mma_ts(tile_tm + 128, tp + 8 * kk,
                               tc::desc_sw128(vst + kk * 2048, kTcRegion, 1024), kIdO,
                               t > 0 || kk > 0);
                tc::commit(o_done(u, t & 1));
                tc::commit(v_empty0 + 8 * (t % kTcStages));
                return true;
            };
            bool ok = mbar_wait_bounded(q_ready, 0, misc, p.wait_cycles);
            for (int j = 0; ok && j < ntiles; ++j) {
                const int s = j % kTcStages;
                // the buffer holds P of stage j - 2 until its value product is done
                if (!mbar_wait_bounded(k_full0 + 8 * s, (j / kTcStages) & 1, misc, p.wait_cycles) ||
                    (j >= 2 && !mbar_wait_bounded(o_done(u, j & 1), ((j - 2) >> 1) & 1, misc,
                                                  p.wait_cycles))) {
                    ok = false;
                    break;
                }
                tc::fence_after();
                const uint32_t kst = kring + s * kTcSlotBytes;
                const uint32_t tS = tile_tm + (j & 1) * kTcKeys;
#pragma unroll
                for (int kk = 0; kk < kHeadDim / 16; ++kk) {
                    const uint32_t o = (kk >> 2) * kTcRegion + 32 * (kk & 3);
                    const uint32_t qo = (kk >> 2) * kTcQHalf + 32 * (kk & 3);
                    tc::mma(tS, tc::desc_sw128(qt + qo, 16, 1024),
                            tc::desc_sw128(kst + o, 16, 1024), kIdS, kk > 0);
                }
                tc::commit(s_full(u, j & 1));
                tc::commit(k_empty0 + 8 * s);  // with the other tile's: the K slot is free
                if (j >= 1 && !value_product(j - 1)) ok = false;
            }
            if (ok && !value_product(ntiles - 1)) ok = false;
            if (!ok) {
                misc[0] = 1;
                flag_error(p.err, QDEC_FLAG_TIMEOUT);
            }
            tc::commit(done_bar);  // every MMA this thread issued has completed
        }
        __syncwarp();
    } else {
        // --------------------------------------------- softmax warps --
        const int u = warp >> 2;                  // query tile
        const int r = tid & (kTcRows - 1);        // row of the tile, tensor-memory lane
        const int hj = r >> 5, ti = r & 31;       // head 4 g + hj, token t0 + 32 u + ti
        const int tok = kTcTileTok * u + ti;      // token of the block
        const bool live = tok < nrows;
        // a wait every lane of the warp passes, or none: the tensor-memory
        // loads and stores below are warp-collective
        auto wait_all = [&](uint32_t bar, uint32_t parity) {
            bool ok = mbar_wait_bounded(bar, parity, misc, p.wait_cycles);
            ok = __all_sync(kFull, ok);
            if (!ok && lane == 0) {
                misc[0] = 1;
                flag_error(p.err, QDEC_FLAG_TIMEOUT);
            }
            return ok;
        };
        if (p.pdl) grid_dependency_wait();  // q_rot, the pool and out of the kernel before
        {
            // Q of the tile, scaled to log2 units, as bf16: warp w converts
            // rows w % 4, w % 4 + 4, ..., lane l taking dims 4 l .. 4 l + 3 of
            // each (one coalesced 512-byte row per warp load, all in flight)
            uint8_t *qt = sm + kTcOffQ + u * kTcQBytes;
            const int half = lane >> 4, cc = (lane & 15) >> 1, sub = (lane & 1) * 8;
            float4 x[kTcRows / 4];
#pragma unroll
            for (int k = 0; k < kTcRows / 4; ++k) {
                const int rr = (warp & 3) + 4 * k, tt = kTcTileTok * u + (rr & 31);
                x[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (tt < nrows)
                    x[k] = reinterpret_cast<const float4 *>(
                        p.q_rot_in + (static_cast<int64_t>(row0 + tt) * p.Hq + g * kGroup + (rr >> 5)) *
                                         kHeadDim)[lane];
            }
#pragma unroll
            for (int k = 0; k < kTcRows / 4; ++k) {
                const int rr = (warp & 3) + 4 * k;
                const uint2 w = make_uint2(pack_bf16x2(x[k].x * p.qscale, x[k].y * p.qscale),
                                           pack_bf16x2(x[k].z * p.qscale, x[k].w * p.qscale));
                *reinterpret_cast<uint2 *>(qt + half * kTcQHalf + sw128_off(rr, cc) + sub) = w;
            }
            fence_proxy_async_smem();  // read next by the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(q_ready);
        }
        const int lim = min(t0 + tok, L - 1);     // the last key this row sees
        const uint32_t trow = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + 256 * u;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            const int s = j % kTcStages;
            if (!wait_all(s_full(u, j & 1), (j >> 1) & 1)) {
                ok = false;
                break;
            }
            tc::fence_after();
            float sc[kTcKeys];
            {
                uint32_t v0[32], v1[32];
                tc::ld32(v0, trow + (j & 1) * kTcKeys);
                tc::ld32(v1, trow + (j & 1) * kTcKeys + 32);
                tc::wait_ld();
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    sc[c] = __uint_as_float(v0[c]);
                    sc[32 + c] = __uint_as_float(v1[c]);
                }
            }
            const int kb = j * kTcKeys;
            if (kb + kTcKeys - 1 > lim) {
#pragma unroll
                for (int c = 0; c < kTcKeys; ++c)
                    if (kb + c > lim) sc[c] = -INFINITY;
            }
            // the row maximum as a tree (short dependency chains)
            float mq[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) mq[q] = fmaxf(sc[q], sc[8 + q]);
#pragma unroll
            for (int c = 16; c < kTcKeys; c += 8)
#pragma unroll
                for (int q = 0; q < 8; ++q) mq[q] = fmaxf(mq[q], sc[c + q]);
            const float mx = fmaxf(fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])),
                                   fmaxf(fmaxf(mq[4], mq[5]), fmaxf(mq[6], mq[7])));
            const bool grow = mx > m + 8.f;
            if (__any_sync(kFull, grow)) {
                const float mn = grow ? fmaxf(m, mx) : m;
                const float alpha = !grow ? 1.f : (m == -INFINITY ? 0.f : exp2f(m - mn));
                l *= alpha;
                m = mn;
                if (j > 0) {
                    // O holds stages 0 .. j-1 once their last product is done
                    if (!wait_all(o_done(u, (j - 1) & 1), ((j - 1) >> 1) & 1)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
#pragma unroll 1
                    for (int c0 = 0; c0 < kHeadDim; c0 += 32) {
                        uint32_t o[32];
                        tc::ld32(o, trow + 128 + c0);
                        tc::wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tc::st32(trow + 128 + c0, o);
                    }
                    tc::wait_st();
                    tc::fence_before();
                }
            }
            // P as bf16 over the first 32 columns of the scores just read (a
            // column holds two consecutive keys), the A operand of the value
            // product
            float ps[4] = {0.f, 0.f, 0.f, 0.f};   // the row sum in four chains
            uint32_t pw[kTcKeys / 2];
#pragma unroll
            for (int c = 0; c < kTcKeys / 2; ++c) {
                const float p0 = fast_exp2(sc[2 * c] - m);
                const float p1 = fast_exp2(sc[2 * c + 1] - m);
                ps[c & 3] += p0 + p1;
                pw[c] = pack_bf16x2(p0, p1);
            }
            tc::st32(trow + (j & 1) * kTcKeys, pw);
            l += (ps[0] + ps[1]) + (ps[2] + ps[3]);
            // V rows of keys past the sequence (and of pages not brought there)
            // are zeroed once the slot has landed, by each tile's warps: both
            // value products read them
            if (kb + kTcKeys > L) {
                if (!wait_all(v_full0 + 8 * s, (j / kTcStages) & 1)) {
                    ok = false;
                    break;
                }
                const int pm = pmask[s];
                uint8_t *vr = sm + kTcOffVRing + s * kTcSlotBytes;
                for (int e = r; e < kTcKeys * 16; e += kTcRows) {
                    const int kr = e >> 4, c = e & 15;
                    if (kb + kr >= L || !((pm >> (kr / kPageSize)) & 1))
                        *reinterpret_cast<uint4 *>(vr + (c >> 3) * kTcRegion + kr * 128 +
                                                   ((c & 7) << 4)) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            tc::wait_st();
            fence_proxy_async_smem();  // the zeroed rows are read by the tensor core
            tc::fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full(u, j & 1));
        }
        // ---- epilogue: O / l for this row, after every product has completed
        volatile int never = 0;
        bool fin = mbar_wait_bounded(done_bar, 0, &never, p.wait_cycles);
        fin = __all_sync(kFull, fin);
        ok = __all_sync(kFull, ok && !misc[0]);
        tc::fence_after();
        if (fin && ok) {
            const float inv = l > 0.f ? 1.f / l : 0.f;
            __nv_bfloat16 *dst =
                p.out + (static_cast<int64_t>(row0 + tok) * p.Hq + g * kGroup + hj) * kHeadDim;
#pragma unroll 1
            for (int c0 = 0; c0 < kHeadDim; c0 += 32) {
                uint32_t o[32];
                tc::ld32(o, trow + 128 + c0);
                tc::wait_ld();
                if (live) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(o[8 * q]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
                        *reinterpret_cast<uint4 *>(dst + c0 + 8 * q) = w;
                    }
                }
            }
        } else if (!fin && lane == 0) {
            misc[0] = 1;
            flag_error(p.err, QDEC_FLAG_TIMEOUT);
        }
        tc::fence_before();
    }
    __syncthreads();
    if (warp == kTcMmaWarp) {
        tc::fence_after();
        tc::dealloc(tmem, kTcTmemCols);
    }
    // a wait that gave up may leave copies in flight: let them land (bounded)
    if ((tid == kTcProducerWarp * 32 || tid == kTcVProducerWarp * 32) && misc[0]) {
        const bool isv = warp == kTcVProducerWarp;
        const uint32_t full0 = isv ? v_full0 : k_full0;
        const int issued = misc[isv ? 5 : 3];
        volatile int never = 0;
        for (int t = max(0, issued - kTcStages); t < issued; ++t)
            mbar_wait_bounded(full0 + 8 * (t % kTcStages), (t / kTcStages) & 1, &never,
                              p.wait_cycles);
    }
}

std::mutex g_pf_mu;
bool g_pf_smem_set[2][64];
bool g_pf_tc_smem_set[64];

}  // namespace

cudaError_t launch_prefill_append(const Params &p, bool fp8, cudaStream_t s) {
    if (p.T <= 0) return cudaSuccess;
    if (fp8)
        prefill_append_kernel<true><<<p.T, kPfAppendThreads, 0, s>>>(p);
    else
        prefill_append_kernel<false><<<p.T, kPfAppendThreads, 0, s>>>(p);
    return cudaGetLastError();
}

template <bool kFp8>
cudaError_t launch_attn(const Params &p, const CUtensorMap &kv_map, int dev, cudaStream_t s) {
    {
        std::lock_guard<std::mutex> lock(g_pf_mu);
        if (!g_pf_smem_set[kFp8 ? 1 : 0][dev]) {
            const cudaError_t e =
                cudaFuncSetAttribute(prefill_attention_kernel<kFp8>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, pf_smem_bytes<kFp8>());
            if (e != cudaSuccess) return e;
            g_pf_smem_set[kFp8 ? 1 : 0][dev] = true;
        }
    }
    // units: at most T / 16 + B blocks of 16 chunk rows, times the KV heads
    const int64_t units = (static_cast<int64_t>(p.T) + kPfRows - 1) / kPfRows + p.B;
    prefill_attention_kernel<kFp8>
        <<<static_cast<unsigned>(units * p.Hkv), kThreads, pf_smem_bytes<kFp8>(), s>>>(kv_map, p);
    return cudaGetLastError();
}

cudaError_t launch_prefill_attention_tc(const Params &p, const CUtensorMap &region_map,
                                        cudaStream_t s) {
    if (p.T <= 0) return cudaSuccess;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 63;
    {
        std::lock_guard<std::mutex> lock(g_pf_mu);
        if (!g_pf_tc_smem_set[dev]) {
            const cudaError_t e = cudaFuncSetAttribute(
                prefill_attention_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemBytes);
            if (e != cudaSuccess) return e;
            g_pf_tc_smem_set[dev] = true;
        }
    }
    // units: at most T / 64 + B blocks of 64 chunk rows, times the KV heads
    const int64_t units = (static_cast<int64_t>(p.T) + kTcTok - 1) / kTcTok + p.B;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(units * p.Hkv));
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = kTcSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = p.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, prefill_attention_tc_kernel, region_map, p);
}

cudaError_t launch_prefill_attention(const Params &p, const CUtensorMap &kv_map, bool fp8,
                                     cudaStream_t s) {
    if (p.T <= 0) return cudaSuccess;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 63;
    return fp8 ? launch_attn<true>(p, kv_map, dev, s) : launch_attn<false>(p, kv_map, dev, s);
}

}  // namespace qdec
