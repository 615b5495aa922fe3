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
// prefill_attention_tc_kernel -- causal paged attention of the chunk (article
//   "扔掉 vLLM！从零构建 Qwen3-8B 推理引擎" (news.rkmt.cn), section 4.4.1:
//   FlashAttention-2 prefill, the queries in blocks that each see only the
//   keys at or before them, never forming the whole score matrix) on the
//   5th-generation tensor core; see the kernel's own comment below.
//
// Over an FP8 (E4M3) pool the append stores codes, each row element divided
// by its (page, plane, head) scale in fp32 and rounded to nearest-even with
// saturation (the decode step's rule), and the attention converts each
// stage's codes to f16 in shared memory (exact: every E4M3 value is an f16
// value) for f16 tensor-core products, multiplies the scores by the K scale
// of their page and folds the V scale into the weights of the value product.
#include "qdec_internal.h"
#include "qdec_ptx.cuh"
#include "qdec_ff.cuh"
#include "qdec_tc.cuh"
#include "qdec.h"

#include <cuda_fp16.h>
#include <math.h>

#include <mutex>

namespace qdec {
namespace {

constexpr unsigned kFull = 0xffffffffu;
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

// Pages sequence b occupies in a widened scratch: all its pages if its chunk
// is well formed, none otherwise (both the widening and the attention use
// this to number the scratch pages).
__device__ __forceinline__ int widened_pages(const Params &p, int b) {
    int n, L;
    return chunk_ok(p, b, n, L) ? (L + kPageSize - 1) / kPageSize : 0;
}
__device__ __forceinline__ int warp_sum_int(int v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// ------------------------------------------------------------------ append --
// One CTA per chunk row, 256 threads: the 64 angles of the row's position are
// taken once (ff_sincos: float pairs) into shared memory; warp w then handles KV head
// w (and w + 8, ...): its four query rows in fp32 (q_rot's tolerance is
// absolute), its key row in float-float arithmetic rounded once to bf16 (the
// decode append's rule: the nearest-even bf16 of the exact value), and the
// copy of its value row.
constexpr int kPfAppendThreads = 256;

// E4M3 codes of a / s and b / s (fp32 division, one rounding each, then
// nearest-even with saturation to +-448), a in the low byte.
__device__ __forceinline__ uint16_t quantize_pair_e4m3(float a, float b, float s) {
    return f32x2_to_e4m3x2(__fdiv_rn(a, s), __fdiv_rn(b, s));
}

template <bool kFp8>
__global__ void __launch_bounds__(kPfAppendThreads) prefill_append_kernel(
    const __grid_constant__ Params p) {
    __shared__ RopeEntry rs[kRotPairs];
    const int r = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = seq_of_row(p.qo_indptr, p.B, r);
    int n, L;
    if (!chunk_ok(p, b, n, L) || r < p.qo_indptr[b] || r >= p.qo_indptr[b + 1]) {
        if (threadIdx.x == 0) flag_error(p.err, QDEC_FLAG_BAD_SEQLEN);
        return;  // uniform over the CTA
    }
    const int t = L - n + (r - p.qo_indptr[b]);  // token index in the sequence
    // A warp's inputs, loaded before the angles are ready so that their
    // latency overlaps the angle computation: the four query rows, the key
    // row and the value row of KV head g (lane l: dims 2l, 2l+1, 64+2l,
    // 65+2l; the value as two 4-byte words), and the page of the row's slot.
    struct RowIn {
        __nv_bfloat162 q[kGroup][2], k[2];
        uint32_t v[2];
        int page;
    };
    auto load_in = [&](int g) {
        RowIn in;
#pragma unroll
        for (int j = 0; j < kGroup; ++j) {
            const __nv_bfloat162 *qr = reinterpret_cast<const __nv_bfloat162 *>(
                p.q + static_cast<int64_t>(r) * p.q_stride + (g * kGroup + j) * kHeadDim);
            in.q[j][0] = qr[lane];
            in.q[j][1] = qr[32 + lane];
        }
        const __nv_bfloat162 *kr = reinterpret_cast<const __nv_bfloat162 *>(
            p.k + static_cast<int64_t>(r) * p.k_stride + g * kHeadDim);
        in.k[0] = kr[lane];
        in.k[1] = kr[32 + lane];
        const uint32_t *vr = reinterpret_cast<const uint32_t *>(
            p.v + static_cast<int64_t>(r) * p.v_stride + g * kHeadDim);
        in.v[0] = vr[lane];
        in.v[1] = vr[32 + lane];
        in.page = p.block_table[static_cast<int64_t>(b) * p.max_blocks + t / kPageSize];
        return in;
    };
    const __nv_bfloat162 wqa = reinterpret_cast<const __nv_bfloat162 *>(p.w_q)[lane];
    const __nv_bfloat162 wqc = reinterpret_cast<const __nv_bfloat162 *>(p.w_q + 64)[lane];
    const __nv_bfloat162 wka = reinterpret_cast<const __nv_bfloat162 *>(p.w_k)[lane];
    const __nv_bfloat162 wkc = reinterpret_cast<const __nv_bfloat162 *>(p.w_k + 64)[lane];
    RowIn in{};
    if (warp < p.Hkv) in = load_in(warp);
    // this lane's rotate-half pairs i = 2 lane, 2 lane + 1: dims i and i + 64;
    // angle i is positions[r] * theta^(-2i/D), from the step's table (row r)
    // or computed here once per row
    const RopeEntry *rope = p.rope + static_cast<int64_t>(r) * kRotPairs;
    if (!p.rope) {  // uniform over the CTA
        if (threadIdx.x < kRotPairs)
            rs[threadIdx.x] = ff_sincos(static_cast<double>(p.positions[r]) * p.inv_freq[threadIdx.x]);
        __syncthreads();
        rope = rs;
    }
    const RopeEntry e0 = rope[2 * lane], e1 = rope[2 * lane + 1];
    const float fc0 = e0.c_hi, fc1 = e1.c_hi, fs0 = e0.s_hi, fs1 = e1.s_hi;
    const float2 wa = __bfloat1622float2(wqa), wc = __bfloat1622float2(wqc);
    for (int g = warp; g < p.Hkv; g += kPfAppendThreads / 32) {
        if (g != warp) in = load_in(g);
#pragma unroll
        for (int j = 0; j < kGroup; ++j) {
            // RMSNorm (eps inside the root; x w exact in fp32, a product of
            // two bf16), then the rotation
            const float2 a = __bfloat1622float2(in.q[j][0]);
            const float2 c = __bfloat1622float2(in.q[j][1]);
            const float ss = warp_sum(a.x * a.x + a.y * a.y + c.x * c.x + c.y * c.y);
            const float rn = rsqrtf(ss * (1.0f / kHeadDim) + p.eps);
            const float n1a = a.x * wa.x * rn, n1b = a.y * wa.y * rn;
            const float n2a = c.x * wc.x * rn, n2b = c.y * wc.y * rn;
            float *dst = p.q_rot_out + (static_cast<int64_t>(r) * p.Hq + g * kGroup + j) * kHeadDim;
            reinterpret_cast<float2 *>(dst)[lane] =
                make_float2(n1a * fc0 - n2a * fs0, n1b * fc1 - n2b * fs1);
            reinterpret_cast<float2 *>(dst + 64)[lane] =
                make_float2(n2a * fc0 + n1a * fs0, n2b * fc1 + n1b * fs1);
        }
        const int page = in.page;
        if (page < 0 || page >= p.num_pages) {
            if (lane == 0) flag_error(p.err, QDEC_FLAG_BAD_PAGE);
            continue;
        }
        const int64_t slot =
            ((static_cast<int64_t>(page) * 2 * p.Hkv + g) * kPageSize + t % kPageSize) * kHeadDim;
        // the key: norm and rotation rounded once to bf16 (exactly)
        __nv_bfloat16 kb[4];
        key_row(p.eps, in.k[0], in.k[1], wka, wkc, e0, e1, kb);
        const uint32_t k01 = static_cast<uint32_t>(__bfloat16_as_ushort(kb[0])) |
                             (static_cast<uint32_t>(__bfloat16_as_ushort(kb[1])) << 16);
        const uint32_t k23 = static_cast<uint32_t>(__bfloat16_as_ushort(kb[2])) |
                             (static_cast<uint32_t>(__bfloat16_as_ushort(kb[3])) << 16);
        const uint32_t v01 = in.v[0], v23 = in.v[1];
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

// ------------------------------------------------------- FP8 widening --
// The E4M3 pages of every well-formed chunk's sequence dequantised once into
// a bf16 scratch laid out as a bf16 pool ([page][plane][head][16][128]):
// sequence b's page pg at scratch page base(b) + pg, base(b) = the widened
// pages of the sequences before b.  Each value is code x scale of its
// (page, plane, head), the exact product rounded to fp32 and then to the
// nearest bf16 (an error of at most 2^-8 of the value, well below the 2^-4
// of the E4M3 code itself; bf16 keeps fp32's range, so no scale overflows
// it).  Rows of tokens past the sequence, and pages whose block-table entry
// is not a valid page (flagged), are zero.  The tensor-core attention then
// reads the scratch exactly as it reads a bf16 pool (kPoolWide: only the
// page numbering differs), so each page is dequantised once instead of once
// per query block, and no scale enters the softmax.  One CTA of 256 threads
// per (sequence, page slot); a thread takes 16 codes at a time, issuing
// kWidenBatch loads before it converts and stores any.
constexpr int kWidenThreads = 256, kWidenBatch = 8;

__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2_scaled(uint32_t two_codes, float scale) {
    const uint32_t h = e4m3x2_to_f16x2(two_codes);
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
    const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
    return *reinterpret_cast<const uint32_t *>(&b);
}

__global__ void __launch_bounds__(kWidenThreads) prefill_widen_kernel(const __grid_constant__ Params p) {
    // the attention after this launch may start its prologue at once; it
    // waits for this grid's completion before it reads the scratch
    if (p.pdl) launch_dependents();
    const int b = blockIdx.x / p.max_blocks, pg = blockIdx.x % p.max_blocks;
    __shared__ int base_s;
    if (threadIdx.x < 32) {  // base(b): a warp sum over the sequences before b
        const int lane = threadIdx.x;
        int before = 0;
        for (int b2 = lane; b2 < b; b2 += 32) before += widened_pages(p, b2);
        before = warp_sum_int(before);
        if (lane == 0) base_s = before;
    }
    __syncthreads();
    int n, L;
    if (b >= p.B || !chunk_ok(p, b, n, L)) return;  // uniform over the CTA
    const int npg = (L + kPageSize - 1) / kPageSize;
    if (pg >= npg) return;
    const int page = p.block_table[static_cast<int64_t>(b) * p.max_blocks + pg];
    const bool valid = page >= 0 && page < p.num_pages;
    if (!valid && threadIdx.x == 0) flag_error(p.err, QDEC_FLAG_BAD_PAGE);
    // the append before wrote the chunk's slots, and the attention before
    // may still read the scratch: codes are read and the scratch written
    // only past this point
    if (p.pdl) grid_dependency_wait();
    const int64_t dst_page = static_cast<int64_t>(base_s) + pg;
    // 2 Hkv (plane, head) blocks of 16 rows x 128 codes; 16 codes per item
    constexpr int kItemsPerBlk = kPageSize * kHeadDim / 16;
    const int items = 2 * p.Hkv * kItemsPerBlk;
    for (int e0 = 0; e0 < items; e0 += kWidenThreads * kWidenBatch) {
        uint4 w[kWidenBatch];
        float sc[kWidenBatch];
#pragma unroll
        for (int k = 0; k < kWidenBatch; ++k) {
            const int e = e0 + k * kWidenThreads + threadIdx.x;
            const int blk = e / kItemsPerBlk;                      // plane * Hkv + head
            const int r = (e / (kHeadDim / 16)) % kPageSize, c = e % (kHeadDim / 16);
            w[k] = make_uint4(0u, 0u, 0u, 0u);
            sc[k] = 0.f;
            if (valid && e < items && pg * kPageSize + r < L) {
                const int64_t pb = static_cast<int64_t>(page) * 2 * p.Hkv + blk;
                w[k] = *reinterpret_cast<const uint4 *>(p.pool8 + (pb * kPageSize + r) * kHeadDim + 16 * c);
                sc[k] = p.kv_scale[pb];
            }
        }
#pragma unroll
        for (int k = 0; k < kWidenBatch; ++k) {
            const int e = e0 + k * kWidenThreads + threadIdx.x;
            if (e >= items) break;
            const int blk = e / kItemsPerBlk;
            const int r = (e / (kHeadDim / 16)) % kPageSize, c = e % (kHeadDim / 16);
            const uint4 lo = make_uint4(e4m3x2_to_bf16x2_scaled(w[k].x, sc[k]),
                                        e4m3x2_to_bf16x2_scaled(w[k].x >> 16, sc[k]),
                                        e4m3x2_to_bf16x2_scaled(w[k].y, sc[k]),
                                        e4m3x2_to_bf16x2_scaled(w[k].y >> 16, sc[k]));
            const uint4 hi = make_uint4(e4m3x2_to_bf16x2_scaled(w[k].z, sc[k]),
                                        e4m3x2_to_bf16x2_scaled(w[k].z >> 16, sc[k]),
                                        e4m3x2_to_bf16x2_scaled(w[k].w, sc[k]),
                                        e4m3x2_to_bf16x2_scaled(w[k].w >> 16, sc[k]));
            uint4 *dst = reinterpret_cast<uint4 *>(
                p.wide + ((dst_page * 2 * p.Hkv + blk) * kPageSize + r) * kHeadDim + 16 * c);
            dst[0] = lo;
            dst[1] = hi;
        }
    }
}

// ------------------------------------- attention on the 5th-gen tensor core --
// prefill_attention_tc_kernel: causal paged attention of the chunk with both
// products on the tensor core (tcgen05, accumulators in tensor memory).  One CTA per (sequence, KV head, block of 64 chunk tokens), the
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
// Per tile, tensor memory holds S (64 columns), P (32 columns: two 16-bit
// weights per column) and O (128 columns).  The softmax warps (warps
// 4 u .. 4 u + 3 for tile u, thread r of the group owning row r, its
// tensor-memory lane) load the 64 scores of stage j and at once hand S back,
// so the scores of stage j + 1 are formed while they mask keys past each
// row's token, keep a stale running maximum (O in tensor memory is rescaled
// only when a stage's maximum exceeds it by more than 2^8, so the weights
// stay below 256), and write P into its own columns once the value product
// of stage j - 1 has read the previous P.  Over a bf16 pool a weight is
// rounded to the nearest bf16 (ties away from zero) by an integer add on
// its bits (the conversion instruction costs more issue slots).  V rows of
// keys past the sequence (or of pages not brought) are zeroed before a value
// product reads them.  The epilogue reads O out of tensor memory, divides by
// the row sum and stores the row.  Every wait is bounded; the decisions that
// lead to warp-collective tensor-memory loads and stores are warp-uniform.
// Over an FP8 pool each producer brings its plane's codes into a staging
// ring (one 2 KiB box per page) and converts them, exactly, to f16 into its
// ring slot, zeroing the rows of keys past the sequence; Q and P are then f16
// and the products of kind f16; the K scale of a key's page multiplies its
// score and the V scale its weight in P (the row sum keeps the unscaled
// weights).
constexpr int kTcTiles = 2;                                // query tiles per CTA
constexpr int kTcTileTok = 32;                             // chunk tokens per tile
constexpr int kTcTok = kTcTiles * kTcTileTok;              // chunk tokens per CTA
constexpr int kTcRows = kTcTileTok * kGroup;               // M = 128 rows per tile
constexpr int kTcKeys = 64;                                // keys per stage
constexpr int kTcPagesPerStage = kTcKeys / kPageSize;      // 4
constexpr int kTcRegion = kTcKeys * 128;                   // [64 keys][64 dims] 16-bit, 8 KiB
constexpr int kTcSlotBytes = 2 * kTcRegion;                // K (or V): dims 0-63, dims 64-127
constexpr int kTcQHalf = kTcRows * 128;                    // [128 rows][64 dims] 16-bit, 16 KiB
constexpr int kTcQBytes = 2 * kTcQHalf;                    // one tile's Q
constexpr int kTcSoftmaxWarps = 4 * kTcTiles;
constexpr int kTcProducerWarp = kTcSoftmaxWarps;           // K stages
constexpr int kTcMmaWarp = kTcSoftmaxWarps + 1;
constexpr int kTcVProducerWarp = kTcSoftmaxWarps + 2;      // V stages
constexpr int kTcMmaWarp1 = kTcSoftmaxWarps + 3;           // tile 1's products (tile 0: kTcMmaWarp)
constexpr int kTcThreads = (kTcSoftmaxWarps + 4) * 32;
// tile u: S at columns 256 u .. +63, P at 256 u + 64 .. +95, O at 256 u + 128 .. +255
constexpr uint32_t kTcTmemCols = 256 * kTcTiles;
static_assert(kTcTmemCols <= 512, "tensor memory");
// FP8 pool: the K and V scales of a stage's four pages, written by the V
// producer when it issues the stage's copies and read by the softmax warps
// once the stage's V slot is full; kept per stage in rings deep enough that
// an entry is rewritten only after its softmax has read it (the V producer
// issues stage j + 8 only after converting stage j + 5, i.e. after the value
// products of stage j + 2, i.e. after every softmax of stage j + 2)
constexpr int kTcKScaleRing = 8, kTcVScaleRing = 8;

// Shared-memory layout of the tensor-core prefill, per pool type: Q of both
// tiles, the K and V rings of 16-bit slots, and for an FP8 pool the staging
// rings of codes (per plane, a stage is four 2 KiB page boxes) and the scale
// rings; then the barriers and a few ints.
// Pool kinds of the tensor-core prefill: a bf16 pool; an FP8 pool whose
// codes each CTA converts to f16 as they arrive; an FP8 pool dequantised to
// bf16 once beforehand (prefill_widen_kernel) into a scratch laid out as a
// bf16 pool, its pages renumbered in sequence order.
constexpr int kPoolBf16 = 0, kPoolFp8 = 1, kPoolWide = 2;

template <int kPool>
struct TcLayout {
    static constexpr bool kStage = kPool == kPoolFp8;      // codes staged and converted
    static constexpr bool kF16 = kStage;                   // f16 operands, per-page scales
    static constexpr int kStages = kStage ? 3 : 4;         // K and V ring depth
    static constexpr int kStg = kStage ? 3 : 0;            // FP8 staging slots per plane
    static constexpr int kStgSlot = kTcPagesPerStage * kFp8PlaneBytes;  // 8 KiB
    static constexpr int kOffQ = 0;                        // Q of tile u at u * kTcQBytes
    static constexpr int kOffKRing = kOffQ + kTcTiles * kTcQBytes;
    static constexpr int kOffVRing = kOffKRing + kStages * kTcSlotBytes;
    static constexpr int kOffStg = kOffVRing + kStages * kTcSlotBytes;  // [plane][kStg] slots
    static constexpr int kOffScale = kOffStg + 2 * kStg * kStgSlot;     // K [16][4], V [8][4] floats
    static constexpr int kScaleBytes = kF16 ? (kTcKScaleRing + kTcVScaleRing) * 4 * 4 : 0;
    static constexpr int kOffTail = kOffScale + kScaleBytes;
    // tail: barriers k_full[S], k_empty[S], v_full[S], v_empty[S], staging
    // full[2][kStg]; per tile s_full, s_free, p_full, o_done (and four unused);
    // q_ready, done; then ints: abort, sequence, block, K stages issued,
    // tensor-memory address, V stages issued, the sequence's first page in
    // a widened scratch, the pages brought into every V slot (bf16 pool) or
    // every staging slot (FP8 pool)
    static constexpr int kBars = 4 * kStages + 2 * kStg + kTcTiles * 8 + 2;
    static constexpr int kTailBytes = kBars * 8 + (7 + kStages + 2 * kStg) * 4;
    static constexpr int kSmemBytes = kOffTail + kTailBytes + 1024;
    static_assert(kSmemBytes <= 227 * 1024, "one CTA per SM");
    static_assert(kOffKRing % 1024 == 0 && kOffVRing % 1024 == 0 && kOffStg % 1024 == 0,
                  "swizzled operands and TMA boxes start on 1024-byte boundaries");
};

// One (page, plane, half of D) region of a bf16 page: 16 tokens x 64 dims,
// 2 KiB, with the pool's region map (5-D: 64 dims, token, half, plane,
// page*2*Hkv + head; box 64 x 16 x 1 x 1 x 1).
__device__ __forceinline__ void tma_load_region(uint32_t dst, const CUtensorMap *map, int half,
                                                int plane, int row, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(half), "r"(plane), "r"(row), "r"(bar)
        : "memory");
}
// One (page, plane) of an FP8 page: 16 tokens x 128 codes, 2 KiB, with the
// FP8 pool's plane map (4-D: 128 bytes of D, token, plane, page*2*Hkv +
// head; box 128 x 16 x 1 x 1).
__device__ __forceinline__ void tma_load_plane8(uint32_t dst, const CUtensorMap *map, int plane,
                                                int row, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(plane), "r"(row), "r"(bar)
        : "memory");
}

// Packed fp32 pairs: one instruction does the work of two (the softmax
// warps are issue-bound, not bound by the exponential unit).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    return static_cast<uint64_t>(__float_as_uint(lo)) | (static_cast<uint64_t>(__float_as_uint(hi)) << 32);
}
__device__ __forceinline__ float f2_lo(uint64_t a) { return __uint_as_float(static_cast<uint32_t>(a)); }
__device__ __forceinline__ float f2_hi(uint64_t a) { return __uint_as_float(static_cast<uint32_t>(a >> 32)); }
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Offset of 16-byte chunk c of row r in a [rows][128 bytes] 128-byte
// swizzled block starting on a 1024-byte boundary.
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
    return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// Two floats as the 16-bit operand type of the pool's products: bf16 over a
// bf16 pool, f16 over an FP8 pool (whose E4M3 codes are exact in f16).
template <bool kFp8>
__device__ __forceinline__ uint32_t pack16x2(float lo, float hi) {
    if constexpr (kFp8) {
        const __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t *>(&h);
    } else {
        return pack_bf16x2(lo, hi);
    }
}

template <int kPool>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_attention_tc_kernel(const __grid_constant__ CUtensorMap kv_map,
                                const __grid_constant__ Params p) {
    using Ly = TcLayout<kPool>;
    constexpr bool kF16 = Ly::kF16, kStage = Ly::kStage;
    constexpr int S = Ly::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint8_t *tail = sm + Ly::kOffTail;
    const uint32_t k_full0 = smem_u32(tail);
    const uint32_t k_empty0 = k_full0 + 8 * S;
    const uint32_t v_full0 = k_empty0 + 8 * S;
    const uint32_t v_empty0 = v_full0 + 8 * S;
    const uint32_t stg_full0 = v_empty0 + 8 * S;             // FP8: [plane][kStg]
    // per tile u: s_full (the scores are in tensor memory), s_free (the
    // softmax warps have loaded them), p_full (P is written), o_done (the
    // value product has completed); one phase per stage each
    const uint32_t tile_bar0 = stg_full0 + 16 * Ly::kStg;
    auto s_full = [&](int u) { return tile_bar0 + 64 * u; };
    auto s_free = [&](int u) { return tile_bar0 + 64 * u + 8; };
    auto p_full = [&](int u) { return tile_bar0 + 64 * u + 16; };
    auto o_done = [&](int u) { return tile_bar0 + 64 * u + 24; };
    const uint32_t q_ready = tile_bar0 + 64 * kTcTiles;
    const uint32_t done_bar = q_ready + 8;
    // misc: [0] abort, [1] sequence, [2] query block, [3] K stages issued,
    // [4] tensor-memory address, [5] V stages issued, [6] the sequence's
    // first page in a widened scratch; pmask[s]: pages brought into V slot s
    // (bf16 or widened pool); smask[plane][q]: pages brought into staging
    // slot q (FP8 pool)
    volatile int *misc = reinterpret_cast<volatile int *>(tail + Ly::kBars * 8);
    volatile int *pmask = misc + 7;
    volatile int *smask = misc + 7 + S;
    float *kscale = reinterpret_cast<float *>(sm + Ly::kOffScale);          // [16][4]
    float *vscale = kscale + kTcKScaleRing * kTcPagesPerStage;              // [8][4]
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
        if constexpr (kPool == kPoolWide) {
            __syncwarp();
            const int bb = misc[1];
            int before = 0;  // widened pages of the sequences before bb
            for (int i = 0; i < per; ++i) {
                const int b2 = lane * per + i;
                if (bb >= 0 && b2 < bb) before += widened_pages(p, b2);
            }
            before = warp_sum_int(before);
            if (lane == 0) misc[6] = before;
        }
        if (lane == 0) {
            for (int s = 0; s < S; ++s) {
                // bf16 pool: the producer's arrival + the bytes; FP8 pool: the
                // producer's arrival once the slot holds the converted codes
                mbar_init(k_full0 + 8 * s, 1);
                mbar_init(k_empty0 + 8 * s, kTcTiles);  // each tile's commit of its score product
                mbar_init(v_full0 + 8 * s, 1);
                mbar_init(v_empty0 + 8 * s, kTcTiles);  // each tile's commit of its value product
            }
            for (int q = 0; q < 2 * Ly::kStg; ++q) mbar_init(stg_full0 + 8 * q, 1);
            for (int u = 0; u < kTcTiles; ++u) {
                mbar_init(s_full(u), 1);   // commit of the score product
                mbar_init(s_free(u), 4);   // the tile's softmax warps have loaded S
                mbar_init(p_full(u), 4);   // the tile's softmax warps have written P
                mbar_init(o_done(u), 1);   // commit of the value product
            }
            mbar_init(q_ready, kTcSoftmaxWarps);
            mbar_init(done_bar, kTcTiles);  // each MMA issuer, once its products are done
            misc[0] = 0;
            misc[3] = 0;
            misc[5] = 0;
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
        // One warp brings the K half of every stage, the other the V half,
        // each into its own ring: a K slot frees as soon as the stage's score
        // products are done, a V slot once its value products are.
        const bool isv = warp == kTcVProducerWarp;
        const int plane = isv ? 1 : 0;
        const uint32_t full0 = isv ? v_full0 : k_full0;
        const uint32_t empty0 = isv ? v_empty0 : k_empty0;
        uint8_t *ringp = sm + (isv ? Ly::kOffVRing : Ly::kOffKRing);
        int issued = 0;
        // waits only lane 0 makes (its outcome is shared with the warp)
        auto lane0_wait = [&](uint32_t bar, uint32_t parity) {
            bool ok = true;
            if (lane == 0) {
                if (misc[0]) {
                    ok = false;
                } else if (!mbar_wait_bounded(bar, parity, misc, p.wait_cycles)) {
                    misc[0] = 1;
                    flag_error(p.err, QDEC_FLAG_TIMEOUT);
                    ok = false;
                }
            }
            return __shfl_sync(kFull, ok, 0) != 0;
        };
        if constexpr (!kStage) {
            // lanes 0-3 each bring one page of the stage (its two regions);
            // the block-table entries are looked up 32 pages (8 stages) at a
            // time, one group ahead.  A widened pool is read at the sequence's
            // scratch pages, which need no lookup (every page below npg is
            // there, zero where the block table has no valid entry)
            constexpr bool kWide = kPool == kPoolWide;
            auto lookup = [&](int grp) {  // lane l: page index 32 grp + l of the sequence
                const int pg = 32 * grp + lane;
                return !kWide && pg < npg ? p.block_table[static_cast<int64_t>(b) * p.max_blocks + pg]
                                          : -1;
            };
            int cur = lookup(0), nxt = lookup(1);
            const int wbase = kWide ? misc[6] : 0;
            // the chunk's keys and values were appended by the kernel before
            if (p.pdl) grid_dependency_wait();
            for (int j = 0; j < ntiles; ++j) {
                const int s = j % S;
                if (!kWide && j > 0 && (j * kTcPagesPerStage) % 32 == 0) {
                    cur = nxt;
                    nxt = lookup(j * kTcPagesPerStage / 32 + 1);
                }
                if (j >= S && !lane0_wait(empty0 + 8 * s, ((j / S) - 1) & 1)) break;
                const int pg = j * kTcPagesPerStage + lane;
                const int page = __shfl_sync(kFull, cur, (j * kTcPagesPerStage + (lane & 3)) & 31);
                const bool valid = kWide || (page >= 0 && page < p.num_pages);
                const bool ok = lane < kTcPagesPerStage && pg < npg && valid;
                if (!isv && lane < kTcPagesPerStage && pg < npg && !valid)
                    flag_error(p.err, QDEC_FLAG_BAD_PAGE);
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
                    const int row = (kWide ? wbase + pg : page) * 2 * p.Hkv + g;
#pragma unroll
                    for (int h = 0; h < 2; ++h)  // region h: dims 64 h .. 64 h + 63 of the plane
                        tma_load_region(dst + h * kTcRegion, &kv_map, h, plane, row, full0 + 8 * s);
                }
                issued = j + 1;
            }
        } else {
            // FP8 pool: each stage's codes land in a staging slot (lanes 0-3
            // each bring one page's plane, 2 KiB, and the V producer the
            // stage's scales); the warp then converts them to f16 (exact) into
            // the ring slot, zeroing the rows of keys past the sequence or on
            // pages not brought.  Page ids are looked up 32 at a time (lane l:
            // page 32 G + l of the sequence) two groups ahead and their scales
            // one group ahead, so no global load stalls the conversions.
            constexpr int Q = Ly::kStg;
            uint8_t *stg = sm + Ly::kOffStg + plane * Q * Ly::kStgSlot;
            const uint32_t sfull0 = stg_full0 + 8 * Q * plane;
            volatile int *sm_mask = smask + Q * plane;
            auto lookup = [&](int grp) {
                const int pg = 32 * grp + lane;
                return pg < npg ? p.block_table[static_cast<int64_t>(b) * p.max_blocks + pg] : -1;
            };
            // the K and V scale of page `page` (0 for an invalid id)
            auto scales = [&](int page, float &ks, float &vs) {
                ks = vs = 0.f;
                if (page >= 0 && page < p.num_pages) {
                    const int64_t si = static_cast<int64_t>(page) * 2 * p.Hkv + g;
                    ks = p.kv_scale[si];
                    vs = p.kv_scale[si + p.Hkv];
                }
            };
            int pc = lookup(0), pn = lookup(1), pn2 = lookup(2), grp = 0;
            // the chunk's keys and values were appended by the kernel before
            if (p.pdl) grid_dependency_wait();
            float ksc = 0.f, vsc = 0.f, ksn = 0.f, vsn = 0.f;
            if (isv) {
                scales(pc, ksc, vsc);
                scales(pn, ksn, vsn);
            }
            auto issue = [&](int jj) {
                const int G = jj * kTcPagesPerStage / 32;
                if (G != grp) {  // stages are issued in order: the next group
                    pc = pn;
                    pn = pn2;
                    pn2 = lookup(G + 2);
                    if (isv) {
                        ksc = ksn;
                        vsc = vsn;
                        scales(pn, ksn, vsn);
                    }
                    grp = G;
                }
                const int q = jj % Q;
                const int pg = jj * kTcPagesPerStage + lane;
                const int src = (jj * kTcPagesPerStage + (lane & 3)) & 31;
                const int page = __shfl_sync(kFull, pc, src);
                const bool ok = lane < kTcPagesPerStage && pg < npg && page >= 0 && page < p.num_pages;
                if (!isv && lane < kTcPagesPerStage && pg < npg && !ok)
                    flag_error(p.err, QDEC_FLAG_BAD_PAGE);
                const unsigned mask = __ballot_sync(kFull, ok) & 0xFu;
                const float ks = __shfl_sync(kFull, ksc, src), vs = __shfl_sync(kFull, vsc, src);
                if (isv && lane < kTcPagesPerStage) {  // both scales of each page of the stage
                    kscale[(jj % kTcKScaleRing) * kTcPagesPerStage + lane] = ok ? ks : 0.f;
                    vscale[(jj % kTcVScaleRing) * kTcPagesPerStage + lane] = ok ? vs : 0.f;
                }
                const bool withheld = !isv && p.withhold_first && jj == 0;  // test hook
                if (lane == 0) {
                    sm_mask[q] = static_cast<int>(mask);
                    if (!withheld) {
                        if (mask == 0)
                            mbar_arrive(sfull0 + 8 * q);
                        else
                            mbar_arrive_expect_tx(sfull0 + 8 * q, __popc(mask) * kFp8PlaneBytes);
                    }
                }
                __syncwarp();
                if (ok && !withheld)
                    tma_load_plane8(smem_u32(stg + q * Ly::kStgSlot) + lane * kFp8PlaneBytes, &kv_map,
                                    plane, page * 2 * p.Hkv + g, sfull0 + 8 * q);
            };
            int staged = 0;
            for (; staged < Q && staged < ntiles; ++staged) issue(staged);
            for (int j = 0; j < ntiles; ++j) {
                const int s = j % S, q = j % Q;
                if (!lane0_wait(sfull0 + 8 * q, (j / Q) & 1)) break;
                if (j >= S && !lane0_wait(empty0 + 8 * s, ((j / S) - 1) & 1)) break;
                const int mask = sm_mask[q];
                const uint8_t *src = stg + q * Ly::kStgSlot;
                uint8_t *dst = ringp + s * kTcSlotBytes;
                // lane l, item i = 8 h + i': key row kr (page kr / 16), codes
                // 16 c .. 16 c + 15, to the f16 chunks 2 c' and 2 c' + 1
                // (c' = c % 4) of region c / 4.  Eight items' codes are
                // loaded before any is stored (the stores could alias the
                // loads as far as the compiler knows, which would serialise
                // them item by item).
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint4 cv[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int e = lane + 32 * (8 * h + i), kr = e >> 3, c = e & 7, tr = kr & 15;
                        const bool zero = j * kTcKeys + kr >= L || !((mask >> (kr >> 4)) & 1);
                        cv[i] = zero ? make_uint4(0u, 0u, 0u, 0u)
                                     : *reinterpret_cast<const uint4 *>(
                                           src + (kr >> 4) * kFp8PlaneBytes + tr * 128 +
                                           ((c ^ (tr & 7)) << 4));
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int e = lane + 32 * (8 * h + i), kr = e >> 3, c = e & 7;
                        const uint4 w = cv[i];   // zero codes convert to +0
                        const uint4 lo = make_uint4(e4m3x2_to_f16x2(w.x), e4m3x2_to_f16x2(w.x >> 16),
                                                    e4m3x2_to_f16x2(w.y), e4m3x2_to_f16x2(w.y >> 16));
                        const uint4 hi = make_uint4(e4m3x2_to_f16x2(w.z), e4m3x2_to_f16x2(w.z >> 16),
                                                    e4m3x2_to_f16x2(w.w), e4m3x2_to_f16x2(w.w >> 16));
                        uint8_t *reg = dst + (c >> 2) * kTcRegion;
                        *reinterpret_cast<uint4 *>(reg + sw128_off(kr, 2 * (c & 3))) = lo;
                        *reinterpret_cast<uint4 *>(reg + sw128_off(kr, 2 * (c & 3) + 1)) = hi;
                    }
                }
                fence_proxy_async_smem();  // read next by the tensor core
                __syncwarp();
                if (lane == 0) mbar_arrive(full0 + 8 * s);
                issued = j + 1;
                if (staged < ntiles) issue(staged++);  // into the staging slot just read
            }
            if (lane == 0) misc[isv ? 5 : 3] = staged;  // staging copies issued
        }
        if constexpr (!kStage)
            if (lane == 0) misc[isv ? 5 : 3] = issued;
    } else if (warp == kTcMmaWarp || warp == kTcMmaWarp1) {
        // ------------------------------------------- the MMA issuers --
        // one thread per query tile issues its products, so neither tile
        // waits for the other's softmax; the two meet only in the K and V
        // rings, whose slots free once both tiles' commits have arrived
        if (lane == 0) {
            const int u = warp == kTcMmaWarp ? 0 : 1;
            const uint32_t qt = smem_u32(sm + Ly::kOffQ) + u * kTcQBytes;
            const uint32_t kring = smem_u32(sm + Ly::kOffKRing), vring = smem_u32(sm + Ly::kOffVRing);
            constexpr uint32_t kIdS = kF16 ? tc::idesc_f16(kTcRows, kTcKeys, false)
                                           : tc::idesc_bf16(kTcRows, kTcKeys, false);
            constexpr uint32_t kIdO = kF16 ? tc::idesc_f16(kTcRows, kHeadDim, true)
                                           : tc::idesc_bf16(kTcRows, kHeadDim, true);
            const uint32_t tile_tm = tmem + 256 * u;
            // O += P_t V_t once V_t has landed and the tile's softmax warps
            // have written P; the commits free P for the weights of stage
            // t + 1 (o_done) and, with the other tile's, the V slot (v_empty)
            auto value_product = [&](int t) -> bool {
                if (!mbar_wait_bounded(v_full0 + 8 * (t % S), (t / S) & 1, misc, p.wait_cycles) ||
                    !mbar_wait_bounded(p_full(u), t & 1, misc, p.wait_cycles))
                    return false;
                tc::fence_after();
                const uint32_t vst = vring + (t % S) * kTcSlotBytes;
#pragma unroll
                for (int kk = 0; kk < kTcKeys / 16; ++kk)
                    tc::mma_ts(tile_tm + 128, tile_tm + 64 + 8 * kk,
                               tc::desc_sw128(vst + kk * 2048, kTcRegion, 1024), kIdO,
                               t > 0 || kk > 0);
                tc::commit(o_done(u));
                tc::commit(v_empty0 + 8 * (t % S));
                return true;
            };
            bool ok = mbar_wait_bounded(q_ready, 0, misc, p.wait_cycles);
            for (int j = 0; ok && j < ntiles; ++j) {
                const int s = j % S;
                // S is free once the softmax warps have loaded the scores of
                // stage j - 1
                if (!mbar_wait_bounded(k_full0 + 8 * s, (j / S) & 1, misc, p.wait_cycles) ||
                    (j >= 1 && !mbar_wait_bounded(s_free(u), (j - 1) & 1, misc, p.wait_cycles))) {
                    ok = false;
                    break;
                }
                tc::fence_after();
                const uint32_t kst = kring + s * kTcSlotBytes;
                const uint32_t tS = tile_tm;
#pragma unroll
                for (int kk = 0; kk < kHeadDim / 16; ++kk) {
                    const uint32_t o = (kk >> 2) * kTcRegion + 32 * (kk & 3);
                    const uint32_t qo = (kk >> 2) * kTcQHalf + 32 * (kk & 3);
                    tc::mma(tS, tc::desc_sw128(qt + qo, 16, 1024),
                            tc::desc_sw128(kst + o, 16, 1024), kIdS, kk > 0);
                }
                tc::commit(s_full(u));
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
            // Q of the tile, scaled to log2 units, in the 16-bit operand type:
            // warp w converts rows w % 4, w % 4 + 4, ..., lane l taking dims
            // 4 l .. 4 l + 3 of each (one coalesced 512-byte row per warp
            // load, all in flight)
            uint8_t *qt = sm + Ly::kOffQ + u * kTcQBytes;
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
                const uint2 w = make_uint2(pack16x2<kF16>(x[k].x * p.qscale, x[k].y * p.qscale),
                                           pack16x2<kF16>(x[k].z * p.qscale, x[k].w * p.qscale));
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
            const int s = j % S;
            if (!wait_all(s_full(u), j & 1)) {
                ok = false;
                break;
            }
            tc::fence_after();
            float sc[kTcKeys];
            {
                uint32_t v0[32], v1[32];
                tc::ld32(v0, trow);
                tc::ld32(v1, trow + 32);
                tc::wait_ld();
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    sc[c] = __uint_as_float(v0[c]);
                    sc[32 + c] = __uint_as_float(v1[c]);
                }
            }
            // the scores are in registers: S may take the next stage's
            tc::fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free(u));
            // FP8 pool: the stage's scales, once its V slot is full (the V
            // producer wrote them before); the scores of page q of the stage
            // times its K scale
            float vs[kTcPagesPerStage] = {1.f, 1.f, 1.f, 1.f};
            if constexpr (kF16) {
                if (!wait_all(v_full0 + 8 * s, (j / S) & 1)) {
                    ok = false;
                    break;
                }
                const float *ks = kscale + (j % kTcKScaleRing) * kTcPagesPerStage;
                const float *vsr = vscale + (j % kTcVScaleRing) * kTcPagesPerStage;
#pragma unroll
                for (int q = 0; q < kTcPagesPerStage; ++q) vs[q] = vsr[q];
#pragma unroll
                for (int c = 0; c < kTcKeys; c += 2) {  // a pair shares its page
                    const float k = ks[c / kPageSize];
                    const uint64_t q = f2_mul(f2_pack(sc[c], sc[c + 1]), f2_pack(k, k));
                    sc[c] = f2_lo(q);
                    sc[c + 1] = f2_hi(q);
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
                    if (!wait_all(o_done(u), (j - 1) & 1)) {
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
            // P (a column holds two consecutive keys), the A operand of the
            // value product, and the row sum of the fp32 weights.  bf16 pool:
            // each weight rounded to the nearest bf16 (ties away from zero:
            // 0x8000 added to its bits, the upper half kept); FP8 pool: f16
            // weights times their page's V scale
            // (pairs of keys in packed fp32: the subtraction of the maximum
            // and the row sum, two chains per packed accumulator)
            uint64_t ps2[2] = {0ull, 0ull};
            const uint64_t mm = f2_pack(m, m);
            uint32_t pw[kTcKeys / 2];
#pragma unroll
            for (int c = 0; c < kTcKeys / 2; ++c) {
                const uint64_t d = f2_sub(f2_pack(sc[2 * c], sc[2 * c + 1]), mm);
                const float p0 = fast_exp2(f2_lo(d));
                const float p1 = fast_exp2(f2_hi(d));
                const uint64_t pp = f2_pack(p0, p1);
                ps2[c & 1] = f2_add(ps2[c & 1], pp);
                if constexpr (kF16) {
                    const float sv = vs[(2 * c) / kPageSize];
                    const uint64_t q = f2_mul(pp, f2_pack(sv, sv));
                    pw[c] = pack16x2<kF16>(f2_lo(q), f2_hi(q));
                } else {
                    pw[c] = __byte_perm(__float_as_uint(p0) + 0x8000u, __float_as_uint(p1) + 0x8000u,
                                        0x7632);
                }
            }
            const float ps[4] = {f2_lo(ps2[0]), f2_hi(ps2[0]), f2_lo(ps2[1]), f2_hi(ps2[1])};
            // P of stage j - 1 stays until its value product is done
            if (j > 0) {
                if (!wait_all(o_done(u), (j - 1) & 1)) {
                    ok = false;
                    break;
                }
                tc::fence_after();
            }
            tc::st32(trow + 64, pw);
            l += (ps[0] + ps[1]) + (ps[2] + ps[3]);
            if constexpr (!kStage) {
                // V rows of keys past the sequence (and of pages not brought
                // there) are zeroed once the slot has landed, by each tile's
                // warps: both value products read them
                if (kb + kTcKeys > L) {
                    if (!wait_all(v_full0 + 8 * s, (j / S) & 1)) {
                        ok = false;
                        break;
                    }
                    const int pm = pmask[s];
                    uint8_t *vr = sm + Ly::kOffVRing + s * kTcSlotBytes;
                    for (int e = r; e < kTcKeys * 16; e += kTcRows) {
                        const int kr = e >> 4, c = e & 15;
                        if (kb + kr >= L || !((pm >> (kr / kPageSize)) & 1))
                            *reinterpret_cast<uint4 *>(vr + (c >> 3) * kTcRegion + kr * 128 +
                                                       ((c & 7) << 4)) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
            tc::wait_st();
            fence_proxy_async_smem();  // the zeroed rows are read by the tensor core
            tc::fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full(u));
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
        const int issued = misc[isv ? 5 : 3];
        volatile int never = 0;
        if constexpr (kStage) {
            const uint32_t sfull0 = stg_full0 + 8 * Ly::kStg * (isv ? 1 : 0);
            for (int t = max(0, issued - Ly::kStg); t < issued; ++t)
                mbar_wait_bounded(sfull0 + 8 * (t % Ly::kStg), (t / Ly::kStg) & 1, &never,
                                  p.wait_cycles);
        } else {
            const uint32_t full0 = isv ? v_full0 : k_full0;
            for (int t = max(0, issued - S); t < issued; ++t)
                mbar_wait_bounded(full0 + 8 * (t % S), (t / S) & 1, &never, p.wait_cycles);
        }
    }
}

std::mutex g_pf_mu;
bool g_pf_tc_smem_set[3][64];

template <int kPool>
cudaError_t launch_tc(const Params &p, const CUtensorMap &kv_map, int dev, cudaStream_t s) {
    using Ly = TcLayout<kPool>;
    {
        std::lock_guard<std::mutex> lock(g_pf_mu);
        if (!g_pf_tc_smem_set[kPool][dev]) {
            const cudaError_t e = cudaFuncSetAttribute(prefill_attention_tc_kernel<kPool>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       Ly::kSmemBytes);
            if (e != cudaSuccess) return e;
            g_pf_tc_smem_set[kPool][dev] = true;
        }
    }
    // units: at most T / 64 + B blocks of 64 chunk rows, times the KV heads
    const int64_t units = (static_cast<int64_t>(p.T) + kTcTok - 1) / kTcTok + p.B;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(units * p.Hkv));
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = Ly::kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = p.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, prefill_attention_tc_kernel<kPool>, kv_map, p);
}

}  // namespace

cudaError_t launch_prefill_append(const Params &p, bool fp8, cudaStream_t s) {
    if (p.T <= 0) return cudaSuccess;
    if (fp8)
        prefill_append_kernel<true><<<p.T, kPfAppendThreads, 0, s>>>(p);
    else
        prefill_append_kernel<false><<<p.T, kPfAppendThreads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_prefill_attention(const Params &p, const CUtensorMap &kv_map, int pool,
                                     cudaStream_t s) {
    if (p.T <= 0) return cudaSuccess;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 63;
    switch (pool) {
    case kPrefillPoolFp8: return launch_tc<kPoolFp8>(p, kv_map, dev, s);
    case kPrefillPoolWide: return launch_tc<kPoolWide>(p, kv_map, dev, s);
    default: return launch_tc<kPoolBf16>(p, kv_map, dev, s);
    }
}

cudaError_t launch_prefill_widen(const Params &p, cudaStream_t s) {
    if (p.T <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.B) * static_cast<unsigned>(p.max_blocks));
    cfg.blockDim = dim3(kWidenThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = p.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, prefill_widen_kernel, p);
}

}  // namespace qdec
