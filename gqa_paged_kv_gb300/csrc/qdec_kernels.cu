// qdec_kernels.cu -- sm_103a kernels of libqdec.
//
// Work layout.  The KV work of one launch is the list of page tiles
// (sequence b, KV head g, page) in that order; a "segment" is the run of
// tiles of one (b, g).  The part of a segment one CTA holds is a "piece": it
// gets a local softmax state, and the pieces of a segment are reduced with
// the exact log-sum-exp rule (blog "GPU 算子与执行优化：从 26 到 100 token/s 的推理引擎破茧之路" (yuzheng310.github.io), part 8,
// split-KV: local softmax per CTA, then a reduction).  Two layouts, chosen
// by the host from the shape:
//   flat    -- CTA j of G takes tiles [j*W/G, (j+1)*W/G) of the W tiles, so
//              every CTA streams the same number of pages whatever the mix of
//              context lengths; pieces of a split segment meet in the
//              workspace and the last CTA to finish merges them.  For large
//              per-CTA work (long ragged batches), where the merge is cheap
//              next to the stream.
//   cluster -- every segment is cut into K equal chunks (K fixed by the
//              shape), one chunk per cluster of C CTAs, one piece per CTA;
//              each CTA pushes its piece into rank 0's shared memory
//              (distributed shared memory) and one cluster barrier later
//              rank 0 merges them; with K > 1 the chunks then meet in the
//              workspace.  A CTA needs only its own sequence's length and
//              block-table row.  For short per-CTA work (small or moderate
//              batches), where global round trips would dominate.
// In both, the grid depends on the shape only (the lengths are read on the
// device), so a launch can be captured in a CUDA graph.
//
// Inside a CTA one producer warp streams page tiles (K and V of one page and
// one KV head, 4 KiB each) from HBM into a shared-memory ring with TMA,
// 128-byte swizzled; four consumer warps take tiles round-robin.  Per tile a
// warp forms S^T = K q^T for the 4 query heads of the group and
// O^T += V^T P^T with bf16 mma.sync (fp32 accumulate).  q and P are fed as
// bf16 hi + lo pairs, so the products carry ~16 mantissa bits while K and V
// enter exactly; the softmax statistics stay in fp32.
//
// With an FP8 (E4M3) pool the tiles are 4 KiB; each also brings its two
// scales (16-byte windows of kv_scale) on the same barrier.  The scores come
// from E4M3 mma.sync (m16n8k32) on the K codes as they are, the query rows
// entering as four E4M3 terms (q 2^e = T0 + T1/16 + T2/256 + T3/4096); the V
// codes are turned into f16 pairs (exact) for an f16 mma.sync with P as f16
// hi + lo.  The K scale and 2^-e multiply the scores; the V scale multiplies
// the weights in the P operand of each tile's product.  The new token's k and v are quantized with
// the scales of their page: fp32 division, then E4M3 nearest-even,
// saturating.
//
// The kernel's mode (template argument): split -- q_rot read from memory,
// the pieces of split segments left in the workspace for merge_kernel (flat
// layout only); fused -- steps 1-4, the new-token rows normed, rotated and
// appended in the kernel, the last piece of a split segment merging it;
// decode -- q_rot read from memory (the slot already appended) with the
// fused mode's layouts and in-kernel merge.
//
// The producer reads only data that no kernel of the step writes (seq_lens,
// the block table, cached pool pages), so when the launch is a programmatic
// dependent of the previous layer it streams pages while that layer is still
// finishing; the consumers wait for the previous kernel before they touch q,
// k, v, the pool slot they append to, the workspace or `out`.  In decode
// mode the previous kernel wrote the appended slots, so there the producer
// waits too before its first copy.
#include "qdec_internal.h"
#include "qdec_ptx.cuh"
#include "qdec_ff.cuh"
#include "qdec.h"

#include <cuda_fp16.h>
#include <math.h>

#include <mutex>

namespace qdec {
namespace {

constexpr float kNegInf = -INFINITY;
constexpr float kRescaleThreshold = 8.0f;          // log2 units: p <= 2^8 between rescales
constexpr unsigned kFull = 0xffffffffu;

// Cody-Waite split of 2*pi for the double-precision angle reduction.
constexpr double kTwoPiHi = 6.283185307179586232;
constexpr double kTwoPiLo = 2.4492935982947064e-16;
constexpr double kInvTwoPi = 0.15915494309189533577;

// ------------------------------------------------------ shared memory map --
constexpr int kQbStride = kHeadDim + 8;  // bf16 per q-operand row (272 B: no bank conflicts)
// prologue buffers (also the whole shared memory of the append kernel)
constexpr int kOffQb = 0;                                        // bf16 [8][kQbStride]
constexpr int kOffKvNew = kOffQb + 8 * kQbStride * 2;            // bf16 [2][D]
constexpr int kOffRope = kOffKvNew + 2 * kHeadDim * 2;           // RopeEntry [D/2]
constexpr int kPrologueBytes = kOffRope + kRotPairs * 16;
// attention-only buffers
constexpr int kOffBar = kPrologueBytes;                          // full[S], empty[S]
constexpr int kOffSlotOk = kOffBar + 2 * kMaxStages * 8;
constexpr int kOffMisc = kOffSlotOk + kMaxStages * 4;            // abort, last, issued
constexpr int kOffKvReady = kOffMisc + 16;                       // mbarrier: new key/value ready
constexpr int kOffPbuf = kOffMisc + 8 * 4;                       // bf16 [warps][8][16]
constexpr int kOffMs = kOffPbuf + kConsumerWarps * 8 * 16 * 2;   // float [warps][G]
constexpr int kOffLs = kOffMs + kConsumerWarps * kGroup * 4;     // float [warps][G]
constexpr int kOffOs = kOffLs + kConsumerWarps * kGroup * 4;     // see below
constexpr int kOsBytes = kConsumerWarps * kGroup * kHeadDim * 4;  // float [warps][G][D]
constexpr int kPartStride = kHeadDim + 4;                        // num[D], M, den, pad
constexpr int kRecvSlotBytes = kGroup * kPartStride * 4;         // one peer's piece
static_assert(kOffKvNew % 16 == 0 && kOffRope % 16 == 0 && kOffBar % 8 == 0 &&
              kOffOs % 16 == 0 && kOffPbuf % 4 == 0 && kRecvSlotBytes % 16 == 0,
              "smem alignment");
static_assert(kOsBytes <= kTileBytes, "the warp-combine scratch fits in one ring slot");
static_assert(kOsBytes + (kMaxCluster - 1) * kRecvSlotBytes <= 4 * kTileBytes,
              "scratch and receive buffer fit in a 4-slot bf16 ring");
// bytes of one ring slot (the FP8 tiles' scales live after the ring)
template <bool kFp8>
__host__ __device__ constexpr int slot_bytes() {
    return kFp8 ? kFp8TileBytes : kTileBytes;
}

// From kOffOs on, the layouts differ:
//   flat (C = 0):   os[warps][G][D] (the warp combine of each piece), then
//                   int pre[B+1], sl[B], then the ring;
//   cluster, C <= kMaxDirectRecv:  the receive buffer float [C-1][G][D+4]
//                   for the peers' pieces, then the ring;
//   cluster, larger C: the ring right away; rank 0 receives in its drained
//                   ring from slot 1 on (peers push only after rank 0 has
//                   arrived on the cluster barrier with its tiles consumed).
// In both cluster layouts one piece per CTA, so once the ring has drained
// its first kOsBytes are the warp-combine scratch (and a receiving ring
// takes the peers' pieces right after).  kMaxDirectRecv is the largest C
// whose receive buffer still leaves room for a 12-slot bf16 ring at 2 CTAs
// per SM.
__host__ __device__ constexpr bool ring_receives(int C) { return C > kMaxDirectRecv; }
__host__ __device__ constexpr int pre_offset(int C) {
    return kOffOs + (C == 0 ? kOsBytes : ring_receives(C) ? 0 : (C - 1) * kRecvSlotBytes);
}
// the ring starts at a 1024-byte boundary (128-byte swizzle atoms); the
// dynamic base itself is aligned with 1024 bytes of slack
__host__ __device__ constexpr int ring_offset(int B, int C) {
    return (pre_offset(C) + (C == 0 ? 4 * (2 * B + 1) : 0) + 1023) / 1024 * 1024;
}

// ------------------------------------------------------------ PTX helpers --
// One whole page tile: the K and V planes of one (page, KV head), 8 KiB,
// landing as [plane][half of D][token][64 dims] in 128-byte swizzled rows.
// The pool's tensor map is 5-D (dims, token, half, plane, page*2*Hkv + head);
// only the last coordinate varies.
__device__ __forceinline__ void tma_load_tile(uint32_t dst, const CUtensorMap *map, int plane_row,
                                              uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %2, %2, %2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(plane_row), "r"(bar)
        : "memory");
}
// One FP8 page tile: [plane][token][128 bytes of D], 4 KiB, 128-byte
// swizzled rows.  The tensor map is 4-D (bytes of D, token, plane,
// page*2*Hkv + head).
__device__ __forceinline__ void tma_load_tile_fp8(uint32_t dst, const CUtensorMap *map,
                                                  int plane_row, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %2, %2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(plane_row), "r"(bar)
        : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}
// D += A (16x32 E4M3, row) * B (32x8 E4M3, col), fp32 accumulate.
__device__ __forceinline__ void mma_e4m3(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// D += A (16x16 f16, row) * B (16x8 f16, col), fp32 accumulate.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// E4M3 codes of a / s and b / s (fp32 division, one rounding each, then
// nearest-even with saturation to +-448), a in the low byte.
__device__ __forceinline__ uint32_t quantize2_e4m3(float a, float b, float s) {
    return f32x2_to_e4m3x2(__fdiv_rn(a, s), __fdiv_rn(b, s));
}
__device__ __forceinline__ void consumer_sync() {  // the 128 consumer threads only
    asm volatile("bar.sync 1, 128;" ::: "memory");
}

// Release/acquire fence at GPU scope (lighter than the sequentially
// consistent one __threadfence issues).
// Atomic add with acquire-release semantics at GPU scope; returns the old value.
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int32_t *addr, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void flag_error(int32_t *err, int bits) {
    if (err) atomicOr(err, bits);
}
// Defensive bounds check on an index derived inside the kernel: a failure
// means an internal inconsistency; the access is skipped and flagged.
__device__ __forceinline__ bool in_bounds(const Params &p, bool ok) {
    if (!ok) flag_error(p.err, QDEC_FLAG_BAD_INDEX);
    return ok;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}
__device__ __forceinline__ uint32_t pack_bf16(__nv_bfloat16 lo, __nv_bfloat16 hi) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(lo)) |
           (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
}

// ------------------------------------------------------------ RoPE angles --
// Angle i of position pos is pos * theta^(-2i/D), formed in double (the
// frequency comes in as a double).  precise: cos/sin as float pairs from
// ff_sincos (double reduction, float-float series); otherwise the angle is
// reduced modulo 2 pi in double and sin/cos are taken in fp32 (the lo parts
// are then zero).
__device__ RopeEntry rope_entry(int pos, double inv_freq, bool precise) {
    const double th = static_cast<double>(pos) * inv_freq;
    RopeEntry e;
    if (precise) {
        e = ff_sincos(th);
    } else {
        const double kq = rint(th * kInvTwoPi);
        double red = fma(-kq, kTwoPiHi, th);
        red = fma(-kq, kTwoPiLo, red);
        sincosf(static_cast<float>(red), &e.s_hi, &e.c_hi);
        e.c_lo = e.s_lo = 0.f;
    }
    return e;
}

// ------------------------------------------------------ sequence metadata --
// Warp-wide: sl[b] = validated length (0 if outside [1, max_blocks * P]),
// pre[b] = pages of sequences before b, pre[B] = total pages.
__device__ void build_prefix(const Params &p, int *pre, int *sl, bool report) {
    const int lane = threadIdx.x & 31;
    const int per = (p.B + 31) / 32;
    const int b0 = lane * per;
    const int cap = p.max_blocks * kPageSize;
    int local = 0, bad = 0;
    for (int i = 0; i < per; ++i) {
        const int b = b0 + i;
        if (b < p.B) {
            int L = p.seq_lens[b];
            if (L < 1 || L > cap) {
                bad = 1;
                L = 0;
            }
            sl[b] = L;
            local += (L + kPageSize - 1) / kPageSize;
        }
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += t;
    }
    int run = incl - local;
    for (int i = 0; i < per; ++i) {
        const int b = b0 + i;
        if (b < p.B) {
            pre[b] = run;
            run += (sl[b] + kPageSize - 1) / kPageSize;
        }
    }
    if (lane == 31) pre[p.B] = incl;
    if (report && __any_sync(kFull, bad) && lane == 0) flag_error(p.err, QDEC_FLAG_BAD_SEQLEN);
}

// CTA that owns flat tile f when W tiles are cut into G equal ranges.
__device__ __forceinline__ int cta_of(long long f, long long W, int G) {
    return static_cast<int>(((f + 1) * G - 1) / W);
}

__device__ int seq_of(const int *pre, int B, int Hkv, long long f) {
    int lo = 0, hi = B - 1;  // largest b with Hkv * pre[b] <= f
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (static_cast<long long>(Hkv) * pre[mid] <= f)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}
// (b, g, page index) of flat tile f
__device__ __forceinline__ void tile_coords(const int *pre, int B, int Hkv, long long f, int &b,
                                            int &g, int &pg) {
    b = seq_of(pre, B, Hkv, f);
    const int n = pre[b + 1] - pre[b];
    if (n <= 0) {  // cannot happen for f inside the tile range; defensive
        g = 0;
        pg = -1;
        return;
    }
    const long long rem = f - static_cast<long long>(Hkv) * pre[b];
    g = static_cast<int>(rem / n);
    pg = static_cast<int>(rem % n);
}

// Walks the pieces of one CTA's tile range in order.
struct Walk {
    int b, g, pg;
    long long f, hi;
};
__device__ void walk_start(Walk &w, const int *pre, int B, int Hkv, long long lo, long long hi) {
    w.f = lo;
    w.hi = hi;
    w.b = w.g = w.pg = 0;
    if (lo < hi) tile_coords(pre, B, Hkv, lo, w.b, w.g, w.pg);
}
__device__ __forceinline__ int piece_len(const Walk &w, const int *pre) {
    const int n = pre[w.b + 1] - pre[w.b];
    const long long left = w.hi - w.f;
    return static_cast<int>(min(static_cast<long long>(n - w.pg), left));
}
__device__ void walk_next(Walk &w, const int *pre, int Hkv, int cnt) {
    w.f += cnt;
    if (w.f >= w.hi) return;
    w.pg = 0;
    if (++w.g == Hkv) {
        w.g = 0;
        do {
            ++w.b;
        } while (pre[w.b + 1] == pre[w.b]);
    }
}

// The new key/value row of (sequence b, KV head g), on one warp: lane l holds
// dims 2l, 2l+1, 64+2l, 65+2l.  bf16(k_rot) (float-float norm and rotation,
// one rounding) and v go to kv_new in shared memory and to the pool slot of
// token L-1.  With an FP8 pool both rows are first quantized with the K and
// V scales of that slot's (page, head): kv_new then holds 128 K codes and
// 128 V codes.
struct KvIn {
    __nv_bfloat162 ka, kc, wka, wkc;
    uint32_t va, vc;
    int page;
    RopeEntry e0, e1;
};

// Loads of key_value_row, issued early so that their latency overlaps other work.
__device__ __forceinline__ KvIn load_kv_inputs(const Params &p, int b, int g, int L) {
    const int lane = threadIdx.x & 31;
    const __nv_bfloat16 *krow = p.k + b * p.k_stride + static_cast<int64_t>(g) * kHeadDim;
    const __nv_bfloat16 *vrow = p.v + b * p.v_stride + static_cast<int64_t>(g) * kHeadDim;
    KvIn in;
    in.ka = reinterpret_cast<const __nv_bfloat162 *>(krow)[lane];
    in.kc = reinterpret_cast<const __nv_bfloat162 *>(krow + 64)[lane];
    in.wka = reinterpret_cast<const __nv_bfloat162 *>(p.w_k)[lane];
    in.wkc = reinterpret_cast<const __nv_bfloat162 *>(p.w_k + 64)[lane];
    in.va = reinterpret_cast<const uint32_t *>(vrow)[lane];
    in.vc = reinterpret_cast<const uint32_t *>(vrow + 64)[lane];
    in.page = p.block_table[static_cast<int64_t>(b) * p.max_blocks + (L - 1) / kPageSize];
    if (p.rope) {
        const RopeEntry *rope = p.rope + static_cast<int64_t>(b) * kRotPairs;
        in.e0 = rope[2 * lane];
        in.e1 = rope[2 * lane + 1];
    } else {
        const int pos = p.positions[b];
        in.e0 = rope_entry(pos, p.inv_freq[2 * lane], true);
        in.e1 = rope_entry(pos, p.inv_freq[2 * lane + 1], true);
    }
    return in;
}

template <bool kFp8>
__device__ void key_value_row(const Params &p, int b, int g, int L, uint8_t *sm, const KvIn &in) {
    const int lane = threadIdx.x & 31;
    // FP8: the slot's scales are loaded before the key arithmetic, which
    // hides their latency
    const bool page_ok = in.page >= 0 && in.page < p.num_pages;
    float sk = 1.f, sv = 1.f;
    if (kFp8 && page_ok) {
        const int64_t si = static_cast<int64_t>(in.page) * 2 * p.Hkv + g;
        sk = __ldg(p.kv_scale + si);
        sv = __ldg(p.kv_scale + si + p.Hkv);
    }
    __nv_bfloat16 kb[4];
    key_row(p.eps, in.ka, in.kc, in.wka, in.wkc, in.e0, in.e1, kb);
    if constexpr (kFp8) {
        const int slot = L - 1;
        const __nv_bfloat162 va = *reinterpret_cast<const __nv_bfloat162 *>(&in.va);
        const __nv_bfloat162 vc = *reinterpret_cast<const __nv_bfloat162 *>(&in.vc);
        const uint32_t k0 = quantize2_e4m3(__bfloat162float(kb[0]), __bfloat162float(kb[1]), sk);
        const uint32_t k1 = quantize2_e4m3(__bfloat162float(kb[2]), __bfloat162float(kb[3]), sk);
        const uint32_t v0 = quantize2_e4m3(__low2float(va), __high2float(va), sv);
        const uint32_t v1 = quantize2_e4m3(__low2float(vc), __high2float(vc), sv);
        uint16_t *kv_new = reinterpret_cast<uint16_t *>(sm + kOffKvNew);  // [K 128 B][V 128 B]
        kv_new[lane] = static_cast<uint16_t>(k0);
        kv_new[32 + lane] = static_cast<uint16_t>(k1);
        kv_new[64 + lane] = static_cast<uint16_t>(v0);
        kv_new[96 + lane] = static_cast<uint16_t>(v1);
        if (page_ok) {
            const int64_t row =
                ((static_cast<int64_t>(in.page) * 2 * p.Hkv + g) * kPageSize + slot % kPageSize) *
                kHeadDim;
            uint16_t *kdst = reinterpret_cast<uint16_t *>(p.pool8 + row);
            uint16_t *vdst = reinterpret_cast<uint16_t *>(
                p.pool8 + row + static_cast<int64_t>(p.Hkv) * kPageSize * kHeadDim);
            kdst[lane] = static_cast<uint16_t>(k0);
            kdst[32 + lane] = static_cast<uint16_t>(k1);
            vdst[lane] = static_cast<uint16_t>(v0);
            vdst[32 + lane] = static_cast<uint16_t>(v1);
        } else if (lane == 0) {
            flag_error(p.err, QDEC_FLAG_BAD_PAGE);
        }
        return;
    }
    const uint32_t k0 = pack_bf16(kb[0], kb[1]), k1 = pack_bf16(kb[2], kb[3]);
    uint32_t *kv_new = reinterpret_cast<uint32_t *>(sm + kOffKvNew);
    kv_new[lane] = k0;
    kv_new[32 + lane] = k1;
    kv_new[64 + lane] = in.va;
    kv_new[96 + lane] = in.vc;
    const int slot = L - 1;
    if (in.page >= 0 && in.page < p.num_pages) {
        const int64_t row =
            ((static_cast<int64_t>(in.page) * 2 * p.Hkv + g) * kPageSize + slot % kPageSize) *
            kHeadDim;
        uint32_t *kdst = reinterpret_cast<uint32_t *>(p.pool + row);
        uint32_t *vdst =
            reinterpret_cast<uint32_t *>(p.pool + row + static_cast<int64_t>(p.Hkv) * kPageSize * kHeadDim);
        kdst[lane] = k0;
        kdst[32 + lane] = k1;
        vdst[lane] = in.va;
        vdst[32 + lane] = in.vc;
    } else if (lane == 0) {
        flag_error(p.err, QDEC_FLAG_BAD_PAGE);
    }
}

// FP8 pools multiply K codes as they are (E4M3 mma.sync, m16n8k32), so the
// query row goes in as E4M3 too, split into four terms: with 2^e putting the
// row's largest magnitude in [128, 256),
//   q * 2^e = T0 + T1 / 16 + T2 / 256 + T3 / 4096 + (error below 2^-16 of it),
// each T_i the E4M3 value nearest to what the previous terms left (times 16).
// Row w of the group (lane l: dims 2l, 2l+1, 64+2l, 65+2l, scaled) writes
// term i to operand column 4i + w of q8 ([16][kQ8Stride] bytes: columns 0-7
// feed n-tile 0, 8-15 n-tile 1) and 2^-e to the head's unscale slot.
constexpr int kQ8Stride = 136;                                  // bytes per operand column
constexpr int kOffQScale = kOffKvNew + 2 * kHeadDim;             // float [G], after the FP8 kv_new
static_assert(16 * kQ8Stride <= kOffKvNew - kOffQb, "FP8 q operand fits the q buffer");
static_assert(kOffQScale + kGroup * 4 <= kOffRope, "unscale slots fit the kv_new buffer");

__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_codes) {
    const uint32_t h = e4m3x2_to_f16x2(two_codes);
    return make_float2(__half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu))),
                       __half2float(__ushort_as_half(static_cast<unsigned short>(h >> 16))));
}

__device__ void store_q_e4m3(uint8_t *sm, int w, int lane, const float (&ys)[4]) {
    float amax = fmaxf(fmaxf(fabsf(ys[0]), fabsf(ys[1])), fmaxf(fabsf(ys[2]), fabsf(ys[3])));
#pragma unroll
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
    int e = 0;
    if (amax > 0.f && amax <= 3.0e38f) e = 134 - static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF);
    float x[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) x[k] = ldexpf(ys[k], e);
    uint8_t *q8 = sm + kOffQb;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t c01 = f32x2_to_e4m3x2(x[0], x[1]);
        const uint32_t c23 = f32x2_to_e4m3x2(x[2], x[3]);
        uint16_t *col = reinterpret_cast<uint16_t *>(q8 + (4 * i + w) * kQ8Stride);
        col[lane] = static_cast<uint16_t>(c01);
        col[32 + lane] = static_cast<uint16_t>(c23);
        const float2 d01 = e4m3x2_to_float2(c01), d23 = e4m3x2_to_float2(c23);
        x[0] = (x[0] - d01.x) * 16.f;
        x[1] = (x[1] - d01.y) * 16.f;
        x[2] = (x[2] - d23.x) * 16.f;
        x[3] = (x[3] - d23.y) * 16.f;
    }
    if (lane == 0) reinterpret_cast<float *>(sm + kOffQScale)[w] = ldexpf(1.f, -e);
}

// Bounds of the new-token work of (sequence b, KV head g) with L tokens.
__device__ __forceinline__ bool new_token_in_bounds(const Params &p, int b, int g, int L) {
    return in_bounds(p, b >= 0 && b < p.B && g >= 0 && g < p.Hkv && L >= 1 &&
                            (L - 1) / kPageSize < p.max_blocks);
}

// Query row w of the group (head 4g + w) of sequence b, on one warp: normed
// and rotated in fp32 with the angles `rope` (the sequence's 64 entries).
// Lane l holds dims 2l, 2l+1, 64+2l, 65+2l: both members of two rotate-half
// pairs.
// Q_OUT = 0: scaled operand rows into shared memory (bf16 hi/lo rows over a
// bf16 pool, four E4M3 terms over an FP8 pool);
// Q_OUT = 1: fp32 rows to p.q_rot_out (unscaled).
template <int Q_OUT, bool kFp8>
__device__ void new_token_row(const Params &p, int b, int g, int w, const RopeEntry *rope,
                              uint8_t *sm) {
    const int lane = threadIdx.x & 31;
    const RopeEntry e0 = rope[2 * lane], e1 = rope[2 * lane + 1];

    const int hq = g * kGroup + w;
    const __nv_bfloat16 *qrow = p.q + b * p.q_stride + static_cast<int64_t>(hq) * kHeadDim;
    const __nv_bfloat162 qa = reinterpret_cast<const __nv_bfloat162 *>(qrow)[lane];
    const __nv_bfloat162 qc = reinterpret_cast<const __nv_bfloat162 *>(qrow + 64)[lane];
    const __nv_bfloat162 wa = reinterpret_cast<const __nv_bfloat162 *>(p.w_q)[lane];
    const __nv_bfloat162 wc = reinterpret_cast<const __nv_bfloat162 *>(p.w_q + 64)[lane];
    float x[4] = {__low2float(qa), __high2float(qa), __low2float(qc), __high2float(qc)};
    const float ss = warp_sum(x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3]);
    const float r = rsqrtf(ss * (1.0f / kHeadDim) + p.eps);
    x[0] = x[0] * r * __low2float(wa);
    x[1] = x[1] * r * __high2float(wa);
    x[2] = x[2] * r * __low2float(wc);
    x[3] = x[3] * r * __high2float(wc);
    const float y0 = x[0] * e0.c_hi - x[2] * e0.s_hi;
    const float y2 = x[2] * e0.c_hi + x[0] * e0.s_hi;
    const float y1 = x[1] * e1.c_hi - x[3] * e1.s_hi;
    const float y3 = x[3] * e1.c_hi + x[1] * e1.s_hi;
    if (Q_OUT == 0 && kFp8) {
        const float ys[4] = {y0 * p.qscale, y1 * p.qscale, y2 * p.qscale, y3 * p.qscale};
        store_q_e4m3(sm, w, lane, ys);
    } else if (Q_OUT == 0) {
        __nv_bfloat16 *qb = reinterpret_cast<__nv_bfloat16 *>(sm + kOffQb);
        const float ys[4] = {y0 * p.qscale, y1 * p.qscale, y2 * p.qscale, y3 * p.qscale};
        __nv_bfloat16 hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            hi[e] = __float2bfloat16_rn(ys[e]);
            lo[e] = __float2bfloat16_rn(ys[e] - __bfloat162float(hi[e]));
        }
        uint32_t *hrow = reinterpret_cast<uint32_t *>(qb + w * kQbStride);
        uint32_t *lrow = reinterpret_cast<uint32_t *>(qb + (kGroup + w) * kQbStride);
        hrow[lane] = pack_bf16(hi[0], hi[1]);
        hrow[32 + lane] = pack_bf16(hi[2], hi[3]);
        lrow[lane] = pack_bf16(lo[0], lo[1]);
        lrow[32 + lane] = pack_bf16(lo[2], lo[3]);
    } else {
        float *dst = p.q_rot_out + (static_cast<int64_t>(b) * p.Hq + hq) * kHeadDim;
        reinterpret_cast<float2 *>(dst)[lane] = make_float2(y0, y1);
        reinterpret_cast<float2 *>(dst + 64)[lane] = make_float2(y2, y3);
    }
}

// The sequence's angles: from the step's table, or computed into shared
// memory by the first kRotPairs of `nthreads` threads that then meet on
// named barrier `bar`.
__device__ __forceinline__ const RopeEntry *rope_of(const Params &p, int b, uint8_t *sm, int bar,
                                                    int nthreads) {
    if (p.rope) return p.rope + static_cast<int64_t>(b) * kRotPairs;
    RopeEntry *rs = reinterpret_cast<RopeEntry *>(sm + kOffRope);
    if (threadIdx.x < kRotPairs) rs[threadIdx.x] = rope_entry(p.positions[b], p.inv_freq[threadIdx.x], false);
    asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(nthreads) : "memory");
    return rs;
}

// The new-token query rows of (sequence b, KV head g), on the 128 consumer
// threads: warp w takes query row 4g + w.  With need_k, warp 0 then also
// produces and appends the key/value row.
template <int Q_OUT, bool kFp8>
__device__ void new_token_rows(const Params &p, int b, int g, int L, bool need_k, uint8_t *sm) {
    const int w = threadIdx.x >> 5;
    if (!new_token_in_bounds(p, b, g, L)) return;  // uniform over the CTA
    const RopeEntry *rope = rope_of(p, b, sm, 1, kConsumerWarps * 32);  // the consumer barrier
    new_token_row<Q_OUT, kFp8>(p, b, g, w, rope, sm);
    if (need_k && w == 0) key_value_row<kFp8>(p, b, g, L, sm, load_kv_inputs(p, b, g, L));
}

// ----------------------------------------------------------- tile math --
// One warp, one 16-token page tile of one KV head, the 4 query heads of its
// group.  Lane (tg = lane/4, c = lane%4) keeps the softmax state of heads
// hA = 2(c&1) and hB = hA + 1 and the O^T accumulator columns 2c, 2c+1
// (c < 2: hi halves of hA, hB; c >= 2: lo halves), for dims 16mt + tg and
// 16mt + tg + 8.
struct WarpState {
    float mA, mB, lA, lB;
    float o[8][4];
};

__device__ __forceinline__ void tile_math(uint32_t ks, uint32_t vs, const uint32_t (&qf)[8][2],
                                          int ntok, int lane, WarpState &st,
                                          __nv_bfloat16 *pbuf) {
    const int tg = lane >> 2, c = lane & 3;
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
    const int ktok = (lane & 7) + ((lane >> 3) & 1) * 8;
    const int kch = lane >> 4;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int chunk = 2 * j + kch;
        const uint32_t addr = ks + (chunk >> 3) * kTileHalfBytes + ktok * 128 +
                              (((chunk & 7) ^ (ktok & 7)) << 4);
        uint32_t a[4];
        ldmatrix_x4(a, addr);
        if (j & 1)
            mma_bf16(s1, a, qf[j][0], qf[j][1]);
        else
            mma_bf16(s0, a, qf[j][0], qf[j][1]);
    }
    float s[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        s[e] = s0[e] + s1[e];
        s[e] += __shfl_xor_sync(kFull, s[e], 2);  // hi column + lo column
    }
    const bool v0 = tg < ntok, v1 = tg + 8 < ntok;
    const float sA0 = v0 ? s[0] : kNegInf, sB0 = v0 ? s[1] : kNegInf;
    const float sA1 = v1 ? s[2] : kNegInf, sB1 = v1 ? s[3] : kNegInf;
    const bool grow = fmaxf(sA0, sA1) > st.mA + kRescaleThreshold ||
                      fmaxf(sB0, sB1) > st.mB + kRescaleThreshold;
    if (__any_sync(kFull, grow)) {
        float tA = fmaxf(sA0, sA1), tB = fmaxf(sB0, sB1);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            tA = fmaxf(tA, __shfl_xor_sync(kFull, tA, o));
            tB = fmaxf(tB, __shfl_xor_sync(kFull, tB, o));
        }
        const float nA = fmaxf(st.mA, tA), nB = fmaxf(st.mB, tB);
        const float aA = st.mA == kNegInf ? 0.f : fast_exp2(st.mA - nA);
        const float aB = st.mB == kNegInf ? 0.f : fast_exp2(st.mB - nB);
        st.mA = nA;
        st.mB = nB;
        st.lA *= aA;
        st.lB *= aB;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            st.o[mt][0] *= aA;
            st.o[mt][2] *= aA;
            st.o[mt][1] *= aB;
            st.o[mt][3] *= aB;
        }
    }
    const float bA = st.mA == kNegInf ? 0.f : st.mA;
    const float bB = st.mB == kNegInf ? 0.f : st.mB;
    const float pA0 = fast_exp2(sA0 - bA), pA1 = fast_exp2(sA1 - bA);
    const float pB0 = fast_exp2(sB0 - bB), pB1 = fast_exp2(sB1 - bB);
    st.lA += pA0 + pA1;
    st.lB += pB0 + pB1;

    // P^T operand: column n < 4 holds bf16(p) of head n, column 4 + n the
    // bf16 remainder p - bf16(p); row = token.
    const bool hi = c < 2;
    const int colA = (hi ? 0 : kGroup) + 2 * (c & 1);
    auto part = [hi](float v) {
        const __nv_bfloat16 h = __float2bfloat16_rn(v);
        return hi ? h : __float2bfloat16_rn(v - __bfloat162float(h));
    };
    pbuf[colA * 16 + tg] = part(pA0);
    pbuf[colA * 16 + tg + 8] = part(pA1);
    pbuf[(colA + 1) * 16 + tg] = part(pB0);
    pbuf[(colA + 1) * 16 + tg + 8] = part(pB1);
    __syncwarp();
    const uint32_t b0 = *reinterpret_cast<const uint32_t *>(pbuf + tg * 16 + 2 * c);
    const uint32_t b1 = *reinterpret_cast<const uint32_t *>(pbuf + tg * 16 + 2 * c + 8);
    const int vtok = (lane & 7) + (lane >> 4) * 8;
    const int vch = (lane >> 3) & 1;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        const int chunk = 2 * mt + vch;
        const uint32_t addr = vs + (chunk >> 3) * kTileHalfBytes + vtok * 128 +
                              (((chunk & 7) ^ (vtok & 7)) << 4);
        uint32_t a[4];
        ldmatrix_x4_trans(a, addr);
        mma_bf16(st.o[mt], a, b0, b1);
    }
    __syncwarp();
}

// Rows of the tile that are not part of the context: V rows >= ntok become
// zero (a NaN there would survive the zero weight inside the MMA); with
// patch, row ntok-1 takes the new key/value just computed.
__device__ void fix_tile(uint8_t *tile, int ntok, bool patch, const __nv_bfloat16 *kv_new,
                         int lane) {
    if (patch) {
        const int plane = lane >> 4, half = (lane >> 3) & 1, cc = lane & 7;
        const int r = ntok - 1;
        const uint4 val =
            reinterpret_cast<const uint4 *>(kv_new + plane * kHeadDim + half * 64)[cc];
        *reinterpret_cast<uint4 *>(tile + plane * kPlaneBytes + half * kTileHalfBytes + r * 128 +
                                   ((cc ^ (r & 7)) << 4)) = val;
    }
    const int rows = kPageSize - ntok;
    for (int e = lane; e < rows * 16; e += 32) {
        const int r = ntok + (e >> 4), half = (e >> 3) & 1, cc = e & 7;
        *reinterpret_cast<uint4 *>(tile + kPlaneBytes + half * kTileHalfBytes + r * 128 +
                                   cc * 16) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();  // ordered before the ring slot is refilled by TMA
    __syncwarp();
}

// The same tile on an FP8 pool.  The order of the reduction dimension is
// free in both products, so each lane reads whole 16-byte runs of a row:
//   S^T = K q^T on E4M3 codes as they are (m16n8k32): lane (tg, c) reads
//     dims 32c .. 32c+31 of tokens tg and tg + 8; in k-step j the bytes
//     32c+8j .. 32c+8j+7 stand for MMA columns 4c .. 4c+3 and 16+4c ..
//     16+4c+3, and q's four E4M3 terms are read the same way (n-tile 0:
//     terms 0, 1; n-tile 1: terms 2, 3; column 4i + h within the pair);
//   O^T += V^T P^T in f16 (m16n8k16): the MMA rows of m-tile mt are dims
//     16r + mt (r < 8) and 16(r-8) + 8 + mt, so lane (tg, c) reads dims
//     16tg .. 16tg+15 of tokens 2c, 2c+1, 2c+8, 2c+9, pairs the tokens'
//     bytes with byte permutes and turns them into f16 (exact).
// Accumulator element o[mt][e] then holds dim 16tg + 8(e >> 1) + mt.  The K
// scale and the query terms' 2^-e multiply the scores; the V scale multiplies
// the weights in the P operand (the row sums keep the unscaled weights).
__device__ __forceinline__ void tile_math_fp8(uint32_t ks, uint32_t vs, const uint32_t (&qf)[8][2],
                                              int ntok, int lane, WarpState &st, __half *pbuf,
                                              float uA, float uB, float sv) {
    const int tg = lane >> 2, c = lane & 3;
    const uint4 k0 = lds128(ks + tg * 128 + (((2 * c) ^ tg) << 4));
    const uint4 k1 = lds128(ks + tg * 128 + (((2 * c + 1) ^ tg) << 4));
    const uint4 k2 = lds128(ks + (tg + 8) * 128 + (((2 * c) ^ tg) << 4));
    const uint4 k3 = lds128(ks + (tg + 8) * 128 + (((2 * c + 1) ^ tg) << 4));
    const uint32_t kr[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
    const uint32_t kr8[8] = {k2.x, k2.y, k2.z, k2.w, k3.x, k3.y, k3.z, k3.w};
    // two accumulators per n-tile (even and odd k-steps): shorter chains
    float t0e[4] = {0.f, 0.f, 0.f, 0.f}, t0o[4] = {0.f, 0.f, 0.f, 0.f};
    float t1e[4] = {0.f, 0.f, 0.f, 0.f}, t1o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t a[4] = {kr[2 * j], kr8[2 * j], kr[2 * j + 1], kr8[2 * j + 1]};
        mma_e4m3(j & 1 ? t0o : t0e, a, qf[j][0], qf[j][1]);
        mma_e4m3(j & 1 ? t1o : t1e, a, qf[4 + j][0], qf[4 + j][1]);
    }
    // columns 2c, 2c+1: terms 0 (c < 2) or 1 (c >= 2) in n-tile 0, terms 2
    // or 3 in n-tile 1; the partner lane c ^ 2 holds the other term of each
    float s[4];
    const bool lead = c < 2;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float x = (t0e[e] + t0o[e]) + (t1e[e] + t1o[e]) * (1.f / 256.f);
        const float y = __shfl_xor_sync(kFull, x, 2);
        s[e] = lead ? x + y * (1.f / 16.f) : y + x * (1.f / 16.f);
        s[e] *= (e & 1) ? uB : uA;
    }
    const bool v0 = tg < ntok, v1 = tg + 8 < ntok;
    const float sA0 = v0 ? s[0] : kNegInf, sB0 = v0 ? s[1] : kNegInf;
    const float sA1 = v1 ? s[2] : kNegInf, sB1 = v1 ? s[3] : kNegInf;
    const bool grow = fmaxf(sA0, sA1) > st.mA + kRescaleThreshold ||
                      fmaxf(sB0, sB1) > st.mB + kRescaleThreshold;
    if (__any_sync(kFull, grow)) {
        float tA = fmaxf(sA0, sA1), tB = fmaxf(sB0, sB1);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            tA = fmaxf(tA, __shfl_xor_sync(kFull, tA, o));
            tB = fmaxf(tB, __shfl_xor_sync(kFull, tB, o));
        }
        const float nA = fmaxf(st.mA, tA), nB = fmaxf(st.mB, tB);
        const float aA = st.mA == kNegInf ? 0.f : fast_exp2(st.mA - nA);
        const float aB = st.mB == kNegInf ? 0.f : fast_exp2(st.mB - nB);
        st.mA = nA;
        st.mB = nB;
        st.lA *= aA;
        st.lB *= aB;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            st.o[mt][0] *= aA;
            st.o[mt][2] *= aA;
            st.o[mt][1] *= aB;
            st.o[mt][3] *= aB;
        }
    }
    const float bA = st.mA == kNegInf ? 0.f : st.mA;
    const float bB = st.mB == kNegInf ? 0.f : st.mB;
    const float pA0 = fast_exp2(sA0 - bA), pA1 = fast_exp2(sA1 - bA);
    const float pB0 = fast_exp2(sB0 - bB), pB1 = fast_exp2(sB1 - bB);
    st.lA += pA0 + pA1;
    st.lB += pB0 + pB1;

    // P^T operand in f16, each weight times the tile's V scale (p <= 2^8
    // between rescales; the row sums above keep the unscaled weights): column
    // n < 4 holds f16(p sv) of head n, column 4 + n the f16 remainder; row =
    // token.
    const bool hi = c < 2;
    const int colA = (hi ? 0 : kGroup) + 2 * (c & 1);
    auto part = [hi, sv](float v) {
        const float x = v * sv;
        const __half h = __float2half_rn(x);
        return hi ? h : __float2half_rn(x - __half2float(h));
    };
    pbuf[colA * 16 + tg] = part(pA0);
    pbuf[colA * 16 + tg + 8] = part(pA1);
    pbuf[(colA + 1) * 16 + tg] = part(pB0);
    pbuf[(colA + 1) * 16 + tg + 8] = part(pB1);
    __syncwarp();
    const uint32_t b0 = *reinterpret_cast<const uint32_t *>(pbuf + tg * 16 + 2 * c);
    const uint32_t b1 = *reinterpret_cast<const uint32_t *>(pbuf + tg * 16 + 2 * c + 8);
    // rows 2c, 2c+1, 2c+8, 2c+9 (swizzle row index & 7: 2c, 2c+1, 2c, 2c+1)
    const uint4 va = lds128(vs + (2 * c) * 128 + ((tg ^ (2 * c)) << 4));
    const uint4 vb = lds128(vs + (2 * c + 1) * 128 + ((tg ^ (2 * c + 1)) << 4));
    const uint4 vc = lds128(vs + (2 * c + 8) * 128 + ((tg ^ (2 * c)) << 4));
    const uint4 vd = lds128(vs + (2 * c + 9) * 128 + ((tg ^ (2 * c + 1)) << 4));
    const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w};
    const uint32_t wc[4] = {vc.x, vc.y, vc.z, vc.w}, wd[4] = {vd.x, vd.y, vd.z, vd.w};
    // token pairs of byte 4w + i: i = 0, 1 in the halves of perm 0x5140, i = 2, 3 of 0x7362
    uint32_t lo01[4], lo23[4], hi01[4], hi23[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        lo01[w] = __byte_perm(wa[w], wb[w], 0x5140);
        lo23[w] = __byte_perm(wa[w], wb[w], 0x7362);
        hi01[w] = __byte_perm(wc[w], wd[w], 0x5140);
        hi23[w] = __byte_perm(wc[w], wd[w], 0x7362);
    }
    // m-tiles 4w + 2ip and 4w + 2ip + 1 from the halves of one permuted word
    // each: dims 16tg + mt (t: tokens 2c, 2c+1; t8: tokens 2c+8, 2c+9) and
    // 16tg + 8 + mt (u, u8)
#pragma unroll
    for (int w = 0; w < 2; ++w) {
#pragma unroll
        for (int ip = 0; ip < 2; ++ip) {
            uint32_t t[2], t8[2], u[2], u8[2];
            e4m3x4_to_f16x2x2(ip ? lo23[w] : lo01[w], t[0], t[1]);
            e4m3x4_to_f16x2x2(ip ? hi23[w] : hi01[w], t8[0], t8[1]);
            e4m3x4_to_f16x2x2(ip ? lo23[w + 2] : lo01[w + 2], u[0], u[1]);
            e4m3x4_to_f16x2x2(ip ? hi23[w + 2] : hi01[w + 2], u8[0], u8[1]);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t a[4] = {t[h], u[h], t8[h], u8[h]};
                mma_f16(st.o[4 * w + 2 * ip + h], a, b0, b1);
            }
        }
    }
    __syncwarp();
}

// fix_tile for an FP8 tile ([plane][token][128 B]): V rows >= ntok become
// zero; with patch, row ntok-1 of both planes takes the new codes.
__device__ void fix_tile_fp8(uint8_t *tile, int ntok, bool patch, const uint8_t *kv_new8, int lane) {
    if (patch && lane < 16) {
        const int plane = lane >> 3, cc = lane & 7;
        const int r = ntok - 1;
        const uint4 val = reinterpret_cast<const uint4 *>(kv_new8 + plane * kHeadDim)[cc];
        *reinterpret_cast<uint4 *>(tile + plane * kFp8PlaneBytes + r * 128 + ((cc ^ (r & 7)) << 4)) =
            val;
    }
    const int rows = kPageSize - ntok;
    for (int e = lane; e < rows * 8; e += 32) {
        const int r = ntok + (e >> 3), cc = e & 7;
        *reinterpret_cast<uint4 *>(tile + kFp8PlaneBytes + r * 128 + cc * 16) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();  // ordered before the ring slot is refilled by TMA
    __syncwarp();
}

// Log-sum-exp merge of the np partials with workspace ids pid0 .. pid0+np-1
// into out[b][4g..4g+3].  128 threads: warp h merges head h, lane l owns
// dims 4l..4l+3.  The lse values are fetched one per lane and the partial
// rows eight at a time, so the L2 round trips overlap.
__device__ void merge_pieces(const Params &p, int64_t pid0, int b, int g, int np) {
    const int t = threadIdx.x, h = t >> 5, lane = t & 31, d0 = lane * 4;
    if (!in_bounds(p, pid0 >= 0 && np >= 1 && pid0 + np <= p.ws_pieces && b >= 0 && b < p.B &&
                          g >= 0 && g < p.Hkv))
        return;
    if (np <= 8) {
        float4 o[8];
        float lse[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            o[u] = u < np ? __ldcg(reinterpret_cast<const float4 *>(
                                p.ws_o + ((pid0 + u) * kGroup + h) * kHeadDim + d0))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
            lse[u] = u < np ? __ldcg(p.ws_lse + (pid0 + u) * kGroup + h) : kNegInf;
        }
        float Ms = kNegInf;
#pragma unroll
        for (int u = 0; u < 8; ++u) Ms = fmaxf(Ms, lse[u]);
        float dn = 0.f;
        float4 nm = make_float4(0.f, 0.f, 0.f, 0.f);
        if (Ms != kNegInf) {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const float e = lse[u] == kNegInf ? 0.f : exp2f(lse[u] - Ms);
                dn += e;
                nm.x += e * o[u].x;
                nm.y += e * o[u].y;
                nm.z += e * o[u].z;
                nm.w += e * o[u].w;
            }
        }
        const float iv = dn > 0.f ? 1.f / dn : 0.f;
        __nv_bfloat16 *dst8 =
            p.out + (static_cast<int64_t>(b) * p.Hq + g * kGroup + h) * kHeadDim + d0;
        reinterpret_cast<uint2 *>(dst8)[0] =
            make_uint2(pack_bf16(__float2bfloat16_rn(nm.x * iv), __float2bfloat16_rn(nm.y * iv)),
                       pack_bf16(__float2bfloat16_rn(nm.z * iv), __float2bfloat16_rn(nm.w * iv)));
        return;
    }
    float M = kNegInf;
    for (int j = lane; j < np; j += 32) M = fmaxf(M, __ldcg(p.ws_lse + (pid0 + j) * kGroup + h));
#pragma unroll
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
    float den = 0.f;
    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != kNegInf) {
        for (int base = 0; base < np; base += 32) {
            const int j = base + lane;
            const float e = j < np ? exp2f(__ldcg(p.ws_lse + (pid0 + j) * kGroup + h) - M) : 0.f;
            den += e;
            const int cnt = min(32, np - base);
            for (int k0 = 0; k0 < cnt; k0 += 8) {
                float4 o[8];
                float ek[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    ek[u] = __shfl_sync(kFull, e, (k0 + u) & 31);
                    o[u] = k0 + u < cnt
                               ? __ldcg(reinterpret_cast<const float4 *>(
                                     p.ws_o + ((pid0 + base + k0 + u) * kGroup + h) * kHeadDim + d0))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float w = k0 + u < cnt ? ek[u] : 0.f;
                    num.x += w * o[u].x;
                    num.y += w * o[u].y;
                    num.z += w * o[u].z;
                    num.w += w * o[u].w;
                }
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) den += __shfl_xor_sync(kFull, den, o);
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    __nv_bfloat16 *dst =
        p.out + (static_cast<int64_t>(b) * p.Hq + g * kGroup + h) * kHeadDim + d0;
    reinterpret_cast<uint2 *>(dst)[0] =
        make_uint2(pack_bf16(__float2bfloat16_rn(num.x * inv), __float2bfloat16_rn(num.y * inv)),
                   pack_bf16(__float2bfloat16_rn(num.z * inv), __float2bfloat16_rn(num.w * inv)));
}

// -------------------------------------------------------- piece processing --
// The 128 consumer threads process pages [pg0, pg0+cnt) of segment (b, g):
// prologue (the group's query rows as MMA operands; with has_last also the
// new key/value), then the tiles, round-robin over the 4 warps by the CTA's
// running tile counter i (shared with the producer).
//
// The new key/value (piece holding the segment's last page) is computed after
// the query rows by warp (i + cnt) % 4, which has the fewest tiles of the
// piece and never the last one; it arrives on the kv-ready barrier (phase =
// kv_uses, the number of such pieces before in this CTA) and the warp that
// patches the last page waits for it.
template <bool kFused, bool kFp8>
__device__ void process_piece(const Params &p, uint8_t *sm, uint8_t *ring, uint32_t full0,
                              uint32_t empty0, volatile int *slot_ok, volatile int *misc, int b,
                              int g, int pg0, int cnt, int L, int n, uint32_t &i,
                              WarpState &st, int &kv_uses, bool early_kv) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tg = lane >> 2, c = lane & 3;
    const int NS = p.stages;
    __nv_bfloat16 *qb = reinterpret_cast<__nv_bfloat16 *>(sm + kOffQb);
    const __nv_bfloat16 *kv_new = reinterpret_cast<const __nv_bfloat16 *>(sm + kOffKvNew);
    __nv_bfloat16 *pbuf = reinterpret_cast<__nv_bfloat16 *>(sm + kOffPbuf) + warp * 8 * 16;
    const bool has_last = pg0 + cnt == n;
    // the warp that will produce the new key: with early_kv (one piece per
    // CTA, latency-bound) it issues its loads first, so their latency overlaps
    // the query rows
    const bool key_warp = kFused && has_last && warp == static_cast<int>((i + cnt) & 3) &&
                          new_token_in_bounds(p, b, g, L);
    KvIn kv_in;
    if (key_warp && early_kv) kv_in = load_kv_inputs(p, b, g, L);

    if (kFused) {
        new_token_rows<0, kFp8>(p, b, g, L, false, sm);
    } else {
        const float *src =
            p.q_rot_in + (static_cast<int64_t>(b) * p.Hq + g * kGroup + warp) * kHeadDim;
        const float2 ya = reinterpret_cast<const float2 *>(src)[lane];
        const float2 yb = reinterpret_cast<const float2 *>(src + 64)[lane];
        const float ys[4] = {ya.x * p.qscale, ya.y * p.qscale, yb.x * p.qscale, yb.y * p.qscale};
        if constexpr (kFp8) {
            store_q_e4m3(sm, warp, lane, ys);
        } else {
            __nv_bfloat16 h4[4], l4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                h4[e] = __float2bfloat16_rn(ys[e]);
                l4[e] = __float2bfloat16_rn(ys[e] - __bfloat162float(h4[e]));
            }
            uint32_t *hrow = reinterpret_cast<uint32_t *>(qb + warp * kQbStride);
            uint32_t *lrow = reinterpret_cast<uint32_t *>(qb + (kGroup + warp) * kQbStride);
            hrow[lane] = pack_bf16(h4[0], h4[1]);
            hrow[32 + lane] = pack_bf16(h4[2], h4[3]);
            lrow[lane] = pack_bf16(l4[0], l4[1]);
            lrow[32 + lane] = pack_bf16(l4[2], l4[3]);
        }
    }
    consumer_sync();
    uint32_t qf[8][2];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if constexpr (kFp8) {  // n-tile j / 4, k-step j % 4 (see tile_math_fp8)
            const uint2 q2 = *reinterpret_cast<const uint2 *>(
                sm + kOffQb + ((j >> 2) * 8 + tg) * kQ8Stride + 32 * c + 8 * (j & 3));
            qf[j][0] = q2.x;
            qf[j][1] = q2.y;
        } else {
            const __nv_bfloat16 *row = qb + tg * kQbStride + 16 * j + 2 * c;
            qf[j][0] = *reinterpret_cast<const uint32_t *>(row);
            qf[j][1] = *reinterpret_cast<const uint32_t *>(row + 8);
        }
    }
    // FP8: 2^-e of the query terms of this lane's heads 2(c&1), 2(c&1)+1
    float qunA = 1.f, qunB = 1.f;
    if constexpr (kFp8) {
        const float *qs = reinterpret_cast<const float *>(sm + kOffQScale);
        qunA = qs[2 * (c & 1)];
        qunB = qs[2 * (c & 1) + 1];
    }
    const uint32_t kv_bar = smem_u32(sm + kOffKvReady);
    const uint32_t kv_parity = static_cast<uint32_t>(kv_uses) & 1;
    if (kFused && has_last) {
        if (warp == static_cast<int>((i + cnt) & 3)) {
            if (key_warp)
                key_value_row<kFp8>(p, b, g, L, sm, early_kv ? kv_in : load_kv_inputs(p, b, g, L));
            __syncwarp();
            if (lane == 0) mbar_arrive(kv_bar);
        }
        ++kv_uses;
    }
    // this warp's tiles of the piece: ring positions i0 + k with (i0 + k) % 4
    // == warp; as NS is a multiple of 4, each step of 4 advances the slot by
    // 4 and flips the phase when it wraps
    const uint32_t i0 = i;
    const int kfirst = (warp - static_cast<int>(i0 & 3)) & 3;
    int slot = static_cast<int>((i0 + kfirst) % NS);
    uint32_t phase = ((i0 + kfirst) / NS) & 1;
    i = i0 + cnt;
    for (int k = kfirst; k < cnt; k += 4) {
        const int cur = slot;
        const uint32_t par = phase;
        slot += 4;
        if (slot >= NS) {
            slot -= NS;
            phase ^= 1;
        }
        const bool ok = mbar_wait_bounded(full0 + 8 * cur, par, misc, p.wait_cycles);
        if (!ok && lane == 0) {
            misc[0] = 1;
            flag_error(p.err, QDEC_FLAG_TIMEOUT);
        }
        const int pg = pg0 + k;
        const int ntok = min(kPageSize, L - pg * kPageSize);
        if (ok && slot_ok[cur]) {
            uint8_t *tile = ring + cur * slot_bytes<kFp8>();
            bool patch = kFused && pg == n - 1;
            if (patch && !mbar_wait_bounded(kv_bar, kv_parity, misc, p.wait_cycles)) {
                if (lane == 0) {
                    misc[0] = 1;
                    flag_error(p.err, QDEC_FLAG_TIMEOUT);
                }
                patch = false;
            }
            const uint32_t ks = smem_u32(tile);
            if constexpr (kFp8) {
                if (patch || ntok < kPageSize)
                    fix_tile_fp8(tile, ntok, patch, reinterpret_cast<const uint8_t *>(kv_new), lane);
                // this slot's K and V scale, stored by the producer
                const float *win = reinterpret_cast<const float *>(
                    ring + NS * kFp8TileBytes + cur * kFp8SlotExtra);
                const float sk = win[0];
                tile_math_fp8(ks, ks + kFp8PlaneBytes, qf, ntok, lane, st,
                              reinterpret_cast<__half *>(pbuf), qunA * sk, qunB * sk,
                              win[1]);
            } else {
                if (patch || ntok < kPageSize) fix_tile(tile, ntok, patch, kv_new, lane);
                tile_math(ks, ks + kPlaneBytes, qf, ntok, lane, st, pbuf);
            }
        }
        __syncwarp();
        // a slot whose copy may still be landing is never handed back
        if (ok && lane == 0) mbar_arrive(empty0 + 8 * cur);
    }
}

__device__ __forceinline__ void reset_state(WarpState &st) {
    st.mA = st.mB = kNegInf;
    st.lA = st.lB = 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) st.o[mt][0] = st.o[mt][1] = st.o[mt][2] = st.o[mt][3] = 0.f;
}

// The four warps' states of one piece, merged: thread t ends with head
// t/32's max M (log2 units), sum den and numerator num for dims 4(t%32)..
struct PieceResult {
    float M, den;
    float4 num;
};
// `os` is the scratch for the warps' accumulators (kOsBytes).  The
// accumulator element o[mt][e] of lane (tg, c) holds dim 16mt + tg + 8(e>>1)
// (bf16 tiles) or 16tg + mt + 8(e>>1) (FP8 tiles).
template <bool kFp8>
__device__ PieceResult combine_warps(WarpState &st, uint8_t *sm, float *os) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tg = lane >> 2, c = lane & 3;
    float *ms = reinterpret_cast<float *>(sm + kOffMs);
    float *ls = reinterpret_cast<float *>(sm + kOffLs);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        st.lA += __shfl_xor_sync(kFull, st.lA, o);
        st.lB += __shfl_xor_sync(kFull, st.lB, o);
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) st.o[mt][e] += __shfl_xor_sync(kFull, st.o[mt][e], 2);
    if (c < 2) {
        const int hA = 2 * c, hB = hA + 1;
        float *oA = os + (warp * kGroup + hA) * kHeadDim;
        float *oB = os + (warp * kGroup + hB) * kHeadDim;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const int d = kFp8 ? 16 * tg + mt : 16 * mt + tg;
            oA[d] = st.o[mt][0];
            oB[d] = st.o[mt][1];
            oA[d + 8] = st.o[mt][2];
            oB[d + 8] = st.o[mt][3];
        }
        if (tg == 0) {
            ms[warp * kGroup + hA] = st.mA;
            ms[warp * kGroup + hB] = st.mB;
            ls[warp * kGroup + hA] = st.lA;
            ls[warp * kGroup + hB] = st.lB;
        }
    }
    consumer_sync();
    const int h = tid >> 5, d0 = (tid & 31) * 4;
    PieceResult r;
    r.M = kNegInf;
#pragma unroll
    for (int q = 0; q < kConsumerWarps; ++q) r.M = fmaxf(r.M, ms[q * kGroup + h]);
    r.den = 0.f;
    r.num = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r.M != kNegInf) {
#pragma unroll
        for (int q = 0; q < kConsumerWarps; ++q) {
            const float mq = ms[q * kGroup + h];
            const float e = mq == kNegInf ? 0.f : exp2f(mq - r.M);
            const float4 o4 =
                *reinterpret_cast<const float4 *>(os + (q * kGroup + h) * kHeadDim + d0);
            r.den += e * ls[q * kGroup + h];
            r.num.x += e * o4.x;
            r.num.y += e * o4.y;
            r.num.z += e * o4.z;
            r.num.w += e * o4.w;
        }
    }
    return r;
}

__device__ __forceinline__ void store_out(const Params &p, int b, int g, const PieceResult &r) {
    const int tid = threadIdx.x, h = tid >> 5, d0 = (tid & 31) * 4;
    const float inv = r.den > 0.f ? 1.f / r.den : 0.f;
    if (!in_bounds(p, b >= 0 && b < p.B && g >= 0 && g < p.Hkv)) return;
    __nv_bfloat16 *dst = p.out + (static_cast<int64_t>(b) * p.Hq + g * kGroup + h) * kHeadDim + d0;
    reinterpret_cast<uint2 *>(dst)[0] = make_uint2(
        pack_bf16(__float2bfloat16_rn(r.num.x * inv), __float2bfloat16_rn(r.num.y * inv)),
        pack_bf16(__float2bfloat16_rn(r.num.z * inv), __float2bfloat16_rn(r.num.w * inv)));
}

// Write this piece's (o, lse) as workspace partial `pid`; with kMerge count
// it against segment sigma's np partials, and if it is the last to arrive
// merge all of them (ids pid0 .. pid0+np-1) into out.
template <bool kMerge>
__device__ void store_partial(const Params &p, volatile int *misc, int64_t pid, int sigma,
                              int64_t pid0, int np, int b, int g, const PieceResult &r) {
    const int tid = threadIdx.x, h = tid >> 5, d0 = (tid & 31) * 4;
    const float inv = r.den > 0.f ? 1.f / r.den : 0.f;
    if (!in_bounds(p, pid >= 0 && pid < p.ws_pieces && sigma >= 0 && sigma < p.B * p.Hkv))
        return;  // uniform over the CTA
    *reinterpret_cast<float4 *>(p.ws_o + (pid * kGroup + h) * kHeadDim + d0) =
        make_float4(r.num.x * inv, r.num.y * inv, r.num.z * inv, r.num.w * inv);
    if ((tid & 31) == 0) p.ws_lse[pid * kGroup + h] = r.den > 0.f ? r.M + log2f(r.den) : kNegInf;
    if (!kMerge) return;
    // release the partial (all 128 threads' stores, ordered by the barrier),
    // count it; the last piece in acquires all of them
    consumer_sync();
    if (tid == 0) {
        const int prev = atomic_add_acq_rel_gpu(p.ws_cnt + sigma, 1);
        misc[1] = prev == np - 1;
    }
    consumer_sync();
    if (misc[1]) {
        merge_pieces(p, pid0, b, g, np);
        if (tid == 0) p.ws_cnt[sigma] = 0;  // ready for the next launch
    }
}


// ------------------------------------------------------ attention kernel --
template <int kMode, bool kCluster, bool kFp8>
__global__ void __launch_bounds__(kThreads, ctas_per_sm(kCluster, kFp8))
    attention_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ Params p) {
    constexpr bool kFused = kMode == kAttnFused;      // steps 1-3 in the kernel
    constexpr bool kMerge = kMode != kAttnSplit;      // the last piece merges
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (p.pdl && tid == 0) launch_dependents();

    uint8_t *ring = sm + ring_offset(p.B, kCluster ? p.cluster : 0);
    const uint32_t full0 = smem_u32(sm + kOffBar);
    const uint32_t empty0 = full0 + kMaxStages * 8;
    volatile int *slot_ok = reinterpret_cast<volatile int *>(sm + kOffSlotOk);
    volatile int *misc = reinterpret_cast<volatile int *>(sm + kOffMisc);  // 0 abort, 1 last, 2 issued
    int *pre = reinterpret_cast<int *>(sm + pre_offset(kCluster ? p.cluster : 0));
    int *sl = pre + p.B + 1;
    const int NS = p.stages;
    // Ring slot s is always consumed by warp s % 4 only when NS is a multiple
    // of the consumer warp count; then each warp waits on its slots' phases in
    // order.  Otherwise two warps could wait on consecutive phases of one slot
    // and the parity wait of the later one would pass on the earlier phase.
    // A receiving ring must hold the combine scratch and C - 1 pieces; the
    // FP8 scale windows need an even number of KV heads.
    const bool ring_short = kCluster && ring_receives(p.cluster) &&
                            NS * slot_bytes<kFp8>() < kOsBytes + (p.cluster - 1) * kRecvSlotBytes;
    if (NS < kConsumerWarps || NS % kConsumerWarps != 0 || NS > kMaxStages || ring_short ||
        (kFp8 && (p.Hkv & 1))) {
        if (tid == 0) flag_error(p.err, QDEC_FLAG_BAD_INDEX);
        return;  // uniform: no barrier has been touched yet
    }

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        mbar_init(smem_u32(sm + kOffKvReady), 1);
        misc[0] = 0;
        misc[1] = 0;
        misc[2] = 0;
        fence_mbar_init();
    }

    // ---- this CTA's tiles: pages [pg_lo, pg_hi) of segment (cb, cg) in the
    // cluster layout; the flat range [lo, hi) of the (b, g, page) order in
    // the flat layout
    long long W = 0, lo = 0, hi = 0;
    int G = 1;
    int cb = 0, cg = 0, cn = 0, cL = 0, crank = 0, pg_lo = 0, pg_hi = 0;
    long long cid = 0;
    if (kCluster) {
        const int C = p.cluster, K = p.chunks;
        cid = blockIdx.x / C;
        crank = static_cast<int>(blockIdx.x % C);
        const int sigma = static_cast<int>(cid / K), ck = static_cast<int>(cid % K);
        cb = sigma / p.Hkv;
        cg = sigma % p.Hkv;
        cL = p.seq_lens[cb];
        if (cL < 1 || cL > p.max_blocks * kPageSize) {
            if (tid == 0 && crank == 0 && ck == 0 && cg == 0) flag_error(p.err, QDEC_FLAG_BAD_SEQLEN);
            cL = 0;
        }
        cn = (cL + kPageSize - 1) / kPageSize;
        const int c0 = static_cast<int>(static_cast<long long>(ck) * cn / K);
        const int c1 = static_cast<int>(static_cast<long long>(ck + 1) * cn / K);
        pg_lo = c0 + crank * (c1 - c0) / C;
        pg_hi = c0 + (crank + 1) * (c1 - c0) / C;
        __syncthreads();  // barrier initialisation
        // first cluster phase: every CTA has started (its shared memory may be
        // written by peers once this phase completes).  When rank 0 receives
        // in its ring, the phase also means rank 0 has drained the ring, so
        // rank 0's threads arrive only once they are done with it.
        if (crank != 0 || !ring_receives(C)) cluster_arrive_relaxed();
    } else {
        if (warp == kConsumerWarps) build_prefix(p, pre, sl, blockIdx.x == 0);
        __syncthreads();
        W = static_cast<long long>(p.Hkv) * pre[p.B];
        if (W == 0) return;
        G = static_cast<int>(min(static_cast<long long>(p.grid), W));
        if (static_cast<int>(blockIdx.x) >= G) return;  // the whole CTA leaves together
        lo = static_cast<long long>(blockIdx.x) * W / G;
        hi = static_cast<long long>(blockIdx.x + 1) * W / G;
    }

    if (warp == kConsumerWarps) {
        // ------------------------------------------------ TMA producer --
        // 32 tiles at a time: every lane looks up one tile's page, lane 0
        // issues the copies in order as ring slots come free.  Over an FP8
        // pool the page ids are looked up two groups ahead and their scales
        // one group ahead, so no global load of the lookup stalls the
        // copies.  In decode mode the previous kernel may have written the
        // pages' new slots.
        if (kMode == kAttnDecode && p.pdl) grid_dependency_wait();
        const long long ntiles = kCluster ? pg_hi - pg_lo : hi - lo;
        uint32_t i = 0;
        int next_slot = 0;   // i % NS
        uint32_t wraps = 0;  // i / NS
        bool stop = false;
        // lane's tile `base + lane`: its page (-1 if none or out of range) and head
        auto page_of = [&](long long base, int &g) {
            g = cg;
            if (base + lane >= ntiles) return -1;
            int b, pg;
            if (kCluster) {
                b = cb;
                pg = pg_lo + static_cast<int>(base) + lane;
            } else {
                tile_coords(pre, p.B, p.Hkv, lo + base + lane, b, g, pg);
            }
            if (!in_bounds(p, b >= 0 && b < p.B && pg >= 0 && pg < p.max_blocks && g >= 0 &&
                                  g < p.Hkv))
                return -1;
            return p.block_table[static_cast<int64_t>(b) * p.max_blocks + pg];
        };
        auto scales_of = [&](int page, int g, float &sk, float &sv) {
            sk = sv = 0.f;
            if (kFp8 && page >= 0 && page < p.num_pages) {
                const int64_t si = static_cast<int64_t>(page) * 2 * p.Hkv + g;
                sk = p.kv_scale[si];
                sv = p.kv_scale[si + p.Hkv];
            }
        };
        int g_c = cg, g_n = cg, page_c = -1, page_n = -1;
        float sck = 0.f, scv = 0.f;  // FP8: the current group's K and V scale
        if constexpr (kFp8) {
            page_c = page_of(0, g_c);
            page_n = page_of(32, g_n);
            scales_of(page_c, g_c, sck, scv);
        }
        for (long long base = 0; base < ntiles && !stop; base += 32) {
            // bf16 pool: the group's pages looked up in place (the lookahead
            // measured slower there)
            int g = g_c, g_n2 = cg, page_n2 = -1;
            float sck_n = 0.f, scv_n = 0.f;
            int page = page_c;
            if constexpr (kFp8) {
                page_n2 = page_of(base + 64, g_n2);
                scales_of(page_n, g_n, sck_n, scv_n);
            } else {
                page = page_of(base, g);
            }
            const int cnt = static_cast<int>(min(32ll, ntiles - base));
            for (int j = 0; j < cnt; ++j, ++i) {
                const int pj = __shfl_sync(kFull, page, j);
                const int gj = __shfl_sync(kFull, g, j);
                const float skj = __shfl_sync(kFull, sck, j), svj = __shfl_sync(kFull, scv, j);
                const int slot = next_slot;
                const uint32_t wr = wraps;
                if (++next_slot == NS) {
                    next_slot = 0;
                    ++wraps;
                }
                if (lane == 0) {
                    const uint32_t full = full0 + 8 * slot;
                    if (misc[0]) {
                        stop = true;  // another thread gave up: issue nothing more
                    } else if (wr > 0 &&
                        !mbar_wait_bounded(empty0 + 8 * slot, (wr - 1) & 1, misc,
                                           p.wait_cycles)) {
                        misc[0] = 1;
                        flag_error(p.err, QDEC_FLAG_TIMEOUT);
                        stop = true;
                    } else if (p.withhold_first && i == 0) {
                        // test hook: this tile's barrier phase never completes
                    } else if (pj >= 0 && pj < p.num_pages && gj >= 0 && gj < p.Hkv) {
                        slot_ok[slot] = 1;
                        if constexpr (kFp8) {
                            // the tile's scales by plain stores (ordered before
                            // the consumers' acquire by the arrive's release),
                            // then the tile: one copy per slot
                            float *win = reinterpret_cast<float *>(ring + NS * kFp8TileBytes +
                                                                   slot * kFp8SlotExtra);
                            win[0] = skj;
                            win[1] = svj;
                            mbar_arrive_expect_tx(full, kFp8TileBytes);
                            tma_load_tile_fp8(smem_u32(ring + slot * kFp8TileBytes), &kv_map,
                                              pj * 2 * p.Hkv + gj, full);
                        } else {
                            mbar_arrive_expect_tx(full, kTileBytes);
                            tma_load_tile(smem_u32(ring + slot * kTileBytes), &kv_map,
                                          pj * 2 * p.Hkv + gj, full);
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
            if constexpr (kFp8) {
                page_c = page_n;
                g_c = g_n;
                sck = sck_n;
                scv = scv_n;
                page_n = page_n2;
                g_n = g_n2;
            }
        }
        if (lane == 0) misc[2] = static_cast<int>(i);
        if (kCluster) {  // the producer warp takes part in both cluster phases
            if (crank == 0 && ring_receives(p.cluster)) cluster_arrive_release();
            cluster_wait();
            cluster_sync_all();
        }
    } else if (!kCluster) {
        // -------------------------------------- consumer warps, flat layout --
        if (p.pdl) grid_dependency_wait();  // q/k/v, pool slot, workspace, out
        Walk w;
        walk_start(w, pre, p.B, p.Hkv, lo, hi);
        uint32_t i = 0;
        int kv_uses = 0;
        while (w.f < w.hi) {
            const int cnt = piece_len(w, pre);
            const int b = w.b, g = w.g;
            const int n = pre[b + 1] - pre[b];
            WarpState st;
            reset_state(st);
            process_piece<kFused, kFp8>(p, sm, ring, full0, empty0, slot_ok, misc, b, g, w.pg, cnt,
                                        sl[b], n, i, st, kv_uses, false);
            const PieceResult r =
                combine_warps<kFp8>(st, sm, reinterpret_cast<float *>(sm + kOffOs));
            const long long seg0 = static_cast<long long>(p.Hkv) * pre[b] + static_cast<long long>(g) * n;
            const int j0 = cta_of(seg0, W, G);
            const int np = cta_of(seg0 + n - 1, W, G) - j0 + 1;
            const int sigma = b * p.Hkv + g;
            if (np == 1)
                store_out(p, b, g, r);
            else
                store_partial<kMerge>(p, misc, sigma + static_cast<int64_t>(blockIdx.x), sigma,
                                      sigma + static_cast<int64_t>(j0), np, b, g, r);
            consumer_sync();  // the shared scratch is reused by the next piece
            walk_next(w, pre, p.Hkv, cnt);
        }
    } else {
        // ----------------------------------- consumer warps, cluster layout --
        if (p.pdl) grid_dependency_wait();
        const int C = p.cluster, K = p.chunks;
        const int cnt = pg_hi - pg_lo;
        WarpState st;
        reset_state(st);
        uint32_t i = 0;
        int kv_uses = 0;
        if (cnt > 0)
            process_piece<kFused, kFp8>(p, sm, ring, full0, empty0, slot_ok, misc, cb, cg, pg_lo,
                                        cnt, cL, cn, i, st, kv_uses, true);
        // every tile has been consumed (so no copy is landing in the ring)
        // before the ring's first kOsBytes become the combine scratch
        consumer_sync();
        PieceResult r = combine_warps<kFp8>(st, sm, reinterpret_cast<float *>(ring));
        // a peer pushes its piece into slot crank - 1 of rank 0's receive
        // buffer; rank 0 keeps its own in registers
        const bool in_ring = ring_receives(C);
        if (crank == 0 && in_ring) cluster_arrive_release();
        cluster_wait();
        const int h = tid >> 5, d0 = (tid & 31) * 4;
        float *recv = reinterpret_cast<float *>(in_ring ? ring + kOsBytes : sm + kOffOs);
        if (crank > 0) {
            float *dst = cluster_peer(recv, 0) + ((crank - 1) * kGroup + h) * kPartStride;
            *reinterpret_cast<float4 *>(dst + d0) = r.num;
            if ((tid & 31) == 0) {
                dst[kHeadDim] = r.M;
                dst[kHeadDim + 1] = r.den;
            }
        }
        cluster_sync_all();
        if (crank == 0) {
            PieceResult m;
            m.M = r.M;
            for (int q = 0; q + 1 < C; ++q)
                m.M = fmaxf(m.M, recv[(q * kGroup + h) * kPartStride + kHeadDim]);
            m.den = 0.f;
            m.num = make_float4(0.f, 0.f, 0.f, 0.f);
            if (m.M != kNegInf) {
                if (r.M != kNegInf) {
                    const float e = exp2f(r.M - m.M);
                    m.den = e * r.den;
                    m.num = make_float4(e * r.num.x, e * r.num.y, e * r.num.z, e * r.num.w);
                }
                for (int q = 0; q + 1 < C; ++q) {
                    const float *pp = recv + (q * kGroup + h) * kPartStride;
                    const float mq = pp[kHeadDim];
                    const float e = mq == kNegInf ? 0.f : exp2f(mq - m.M);
                    const float4 o4 = *reinterpret_cast<const float4 *>(pp + d0);
                    m.den += e * pp[kHeadDim + 1];
                    m.num.x += e * o4.x;
                    m.num.y += e * o4.y;
                    m.num.z += e * o4.z;
                    m.num.w += e * o4.w;
                }
            }
            if (K == 1) {
                store_out(p, cb, cg, m);
            } else {
                const int sigma = cb * p.Hkv + cg;
                store_partial<kMerge>(p, misc, cid, sigma, static_cast<int64_t>(sigma) * K, K, cb,
                                      cg, m);
            }
        }
    }
    __syncthreads();
    // A wait that gave up may leave bulk copies in flight: let them land
    // (bounded) before the CTA's shared memory is released.
    if (tid == 0 && misc[0]) {
        const uint32_t issued = static_cast<uint32_t>(misc[2]);
        const uint32_t first = issued > static_cast<uint32_t>(NS) ? issued - NS : 0;
        volatile int never = 0;
        for (uint32_t t = first; t < issued; ++t)
            mbar_wait_bounded(full0 + 8 * (t % NS), (t / NS) & 1, &never, p.wait_cycles);
    }
}

// ------------------------------------------------------------ rope table --
constexpr int kRopeThreads = 32;
// cos/sin of every (sequence, frequency) of the step, computed once and
// shared by all layers (the angles depend on the positions only), one angle
// per thread over many small CTAs.  A following attention launch may start early: it reads the
// table only after its dependency wait.
__global__ void __launch_bounds__(kRopeThreads) rope_table_kernel(const __grid_constant__ Params p) {
    launch_dependents();
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= p.B * kRotPairs) return;
    const int b = idx / kRotPairs, i = idx % kRotPairs;
    p.rope_out[idx] = rope_entry(p.positions[b], p.inv_freq[i], true);
}

// ---------------------------------------------------------- append kernel --
// Steps 1-3 for (KV head blockIdx.x, sequence blockIdx.y): q rows to
// q_rot_out, k and v into the pool.  Warps 0-3 produce the four query rows,
// warp 4 the key/value row, so the key's loads do not wait behind a query
// row's (the attention launched after this kernel waits for all of it).
constexpr int kAppendThreads = 5 * 32;
template <bool kFp8>
__global__ void __launch_bounds__(kAppendThreads) append_rope_kernel(const __grid_constant__ Params p) {
    __shared__ __align__(16) uint8_t sm[kPrologueBytes];
    // as a programmatic dependent (the flag's contract: the previous kernel
    // writes neither seq_lens nor the block table): the attention after it
    // may be scheduled at once, and q/k/v, the pool slot and q_rot are only
    // touched once the previous kernel has completed
    if (p.pdl) launch_dependents();
    const int g = blockIdx.x, b = blockIdx.y;
    const int L = p.seq_lens[b];
    if (L < 1 || L > p.max_blocks * kPageSize) {
        if (threadIdx.x == 0 && g == 0) flag_error(p.err, QDEC_FLAG_BAD_SEQLEN);
        return;
    }
    if (p.pdl) grid_dependency_wait();
    const int warp = threadIdx.x >> 5;
    if (warp >= kGroup) {
        if (new_token_in_bounds(p, b, g, L))
            key_value_row<kFp8>(p, b, g, L, sm, load_kv_inputs(p, b, g, L));
        return;
    }
    if (!new_token_in_bounds(p, b, g, L)) return;  // uniform over the CTA
    const RopeEntry *rope = rope_of(p, b, sm, 2, kGroup * 32);
    new_token_row<1, kFp8>(p, b, g, warp, rope, sm);
}

// ----------------------------------------------------------- merge kernel --
// One CTA per (sequence, KV head): merges the pieces the split kernel left.
__global__ void __launch_bounds__(128) merge_kernel(const __grid_constant__ Params p) {
    __shared__ int pre[kMaxBatch + 1];
    __shared__ int sl[kMaxBatch];
    if (threadIdx.x < 32) build_prefix(p, pre, sl, false);
    __syncthreads();
    const int sigma = blockIdx.x, b = sigma / p.Hkv, g = sigma % p.Hkv;
    const int n = pre[b + 1] - pre[b];
    if (n == 0) return;
    const long long W = static_cast<long long>(p.Hkv) * pre[p.B];
    const int G = static_cast<int>(min(static_cast<long long>(p.grid), W));
    const long long seg0 = static_cast<long long>(p.Hkv) * pre[b] + static_cast<long long>(g) * n;
    const int j0 = cta_of(seg0, W, G);
    const int np = cta_of(seg0 + n - 1, W, G) - j0 + 1;
    if (np == 1) return;  // the split kernel wrote this output itself
    merge_pieces(p, static_cast<int64_t>(sigma) + j0, b, g, np);
}

// Largest dynamic shared memory each attention kernel variant has been
// allowed on each device.  The attribute only ever grows: a launch (or an
// occupancy query) that needs less leaves it as it is, so a later launch
// that needs more than a smaller request in between still finds it set.
std::mutex g_smem_mu;
size_t g_smem_attr[12][64];

template <int kMode, bool kCluster, bool kFp8>
cudaError_t allow_smem(int dev, size_t smem) {
    std::lock_guard<std::mutex> lock(g_smem_mu);
    size_t &attr = g_smem_attr[(kFp8 ? 6 : 0) + 2 * kMode + (kCluster ? 1 : 0)][dev];
    if (attr >= smem) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(attention_kernel<kMode, kCluster, kFp8>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
    if (e == cudaSuccess) attr = smem;
    return e;
}

template <int kMode, bool kCluster, bool kFp8>
cudaError_t launch_one(const Params &p, const CUtensorMap &kv_map, size_t smem, int dev,
                       cudaStream_t s) {
    auto kern = attention_kernel<kMode, kCluster, kFp8>;
    const cudaError_t e = allow_smem<kMode, kCluster, kFp8>(dev, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (kCluster) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = p.cluster;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    if (p.pdl) {
        attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, kv_map, p);
}

}  // namespace

size_t attention_smem_bytes(int B, int stages, int cluster, bool fp8) {
    const size_t slot = fp8 ? kFp8TileBytes + kFp8SlotExtra : kTileBytes;
    return static_cast<size_t>(ring_offset(B, cluster)) + static_cast<size_t>(stages) * slot + 1024;
}

int min_stages(int cluster, bool fp8) {
    int need = kConsumerWarps;
    if (cluster > 0 && ring_receives(cluster)) {
        const int bytes = kOsBytes + (cluster - 1) * kRecvSlotBytes;
        const int slot = fp8 ? kFp8TileBytes : kTileBytes;
        need = (bytes + slot - 1) / slot;
        need = (need + kConsumerWarps - 1) / kConsumerWarps * kConsumerWarps;
    }
    return need;
}

static int current_device() {
    int d = 0;
    cudaGetDevice(&d);
    return d < 64 ? d : 63;
}

template <bool kFp8>
static int max_active_clusters_of(int cluster, size_t smem) {
    auto kern = attention_kernel<kAttnFused, true, kFp8>;
    if (allow_smem<kAttnFused, true, kFp8>(current_device(), smem) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cluster * 64);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = cluster;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return 0;
    return n;
}

int max_active_clusters(int cluster, size_t smem, bool fp8) {
    return fp8 ? max_active_clusters_of<true>(cluster, smem)
               : max_active_clusters_of<false>(cluster, smem);
}

// The split kernel of the three-call path always runs the flat layout (its
// merge kernel reads that layout), so it has no cluster variant.
template <bool kFp8>
cudaError_t launch_mode(const Params &p, const CUtensorMap &kv_map, AttnMode mode, size_t smem,
                        int dev, cudaStream_t s) {
    switch (mode) {
    case kAttnSplit:
        if (p.cluster) return cudaErrorInvalidValue;
        return launch_one<kAttnSplit, false, kFp8>(p, kv_map, smem, dev, s);
    case kAttnFused:
        return p.cluster ? launch_one<kAttnFused, true, kFp8>(p, kv_map, smem, dev, s)
                         : launch_one<kAttnFused, false, kFp8>(p, kv_map, smem, dev, s);
    case kAttnDecode:
        return p.cluster ? launch_one<kAttnDecode, true, kFp8>(p, kv_map, smem, dev, s)
                         : launch_one<kAttnDecode, false, kFp8>(p, kv_map, smem, dev, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_attention(const Params &p, const CUtensorMap &kv_map, AttnMode mode, bool fp8,
                             cudaStream_t s) {
    const size_t smem = attention_smem_bytes(p.B, p.stages, p.cluster, fp8);
    const int dev = current_device();
    return fp8 ? launch_mode<true>(p, kv_map, mode, smem, dev, s)
               : launch_mode<false>(p, kv_map, mode, smem, dev, s);
}

cudaError_t launch_rope_table(const Params &p, cudaStream_t s) {
    const int n = p.B * kRotPairs;
    rope_table_kernel<<<(n + kRopeThreads - 1) / kRopeThreads, kRopeThreads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_append_rope(const Params &p, bool fp8, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.Hkv, p.B);
    cfg.blockDim = dim3(kAppendThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = p.pdl ? 1 : 0;
    return fp8 ? cudaLaunchKernelEx(&cfg, append_rope_kernel<true>, p)
               : cudaLaunchKernelEx(&cfg, append_rope_kernel<false>, p);
}

cudaError_t launch_merge(const Params &p, cudaStream_t s) {
    merge_kernel<<<p.B * p.Hkv, 128, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace qdec
