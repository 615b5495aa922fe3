// qdec_kernels.cu -- sm_103a kernels of libqdec.
//
// Work layout.  The KV work of one launch is the flat list of page tiles
// (sequence b, KV head g, page) in that order; a "segment" is the run of
// tiles of one (b, g).  CTA j of G takes tiles [j*W/G, (j+1)*W/G) of the W
// tiles, so every CTA streams the same number of pages whatever the mix of
// context lengths (the ragged batch needs no host-side planning and the grid
// never depends on the lengths, so a launch can be captured in a graph).
// The part of a segment one CTA holds is a "piece": it gets a local softmax
// state and, when the segment is split over several CTAs, its (o, lse)
// pair goes to the workspace and is merged with the exact log-sum-exp rule
// (blog "Qwen3 GPU optimisation", part 8, split-KV: local softmax per CTA,
// then a reduction).
//
// Inside a CTA one producer thread streams page tiles (K and V of one page
// and one KV head, 4 KiB each) from HBM into an 8-deep shared-memory ring
// with TMA, 128-byte swizzled; four consumer warps take tiles round-robin.
// Per tile a warp forms S^T = K q^T for the 4 query heads of the group and
// O^T += V^T P^T with bf16 mma.sync (fp32 accumulate).  q and P are fed as
// bf16 hi + lo pairs, so the products carry ~16 mantissa bits while K and V
// enter exactly; the softmax statistics stay in fp32.
#include "qdec_internal.h"
#include "qdec.h"

#include <math.h>

namespace qdec {
namespace {

constexpr float kNegInf = -INFINITY;
constexpr float kRescaleThreshold = 8.0f;          // log2 units: p <= 2^8 between rescales
constexpr unsigned long long kWaitTimeoutNs = 1000000000ull;
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
constexpr int kOffCs = kOffKvNew + 2 * kHeadDim * 2;             // float2 [D/2]
constexpr int kOffKcs = kOffCs + kRotPairs * 8;                  // double2 [D/2]
constexpr int kOffKx = kOffKcs + kRotPairs * 16;                 // double [D]
constexpr int kOffKss = kOffKx + kHeadDim * 8;                   // double [4]
constexpr int kPrologueBytes = kOffKss + 4 * 8;
// attention-only buffers
constexpr int kOffBar = kPrologueBytes;                          // full[S], empty[S]
constexpr int kOffSlotOk = kOffBar + 2 * kStages * 8;
constexpr int kOffMisc = kOffSlotOk + kStages * 4;               // abort, last, issued
constexpr int kOffPbuf = kOffMisc + 8 * 4;                       // bf16 [warps][8][16]
constexpr int kOffMs = kOffPbuf + kConsumerWarps * 8 * 16 * 2;   // float [warps][G]
constexpr int kOffLs = kOffMs + kConsumerWarps * kGroup * 4;     // float [warps][G]
constexpr int kOffOs = kOffLs + kConsumerWarps * kGroup * 4;     // float [warps][G][D]
constexpr int kOffPre = kOffOs + kConsumerWarps * kGroup * kHeadDim * 4;  // int [B+1]
constexpr int kOffSl = kOffPre + (kMaxBatch + 1) * 4;                     // int [B]
constexpr int kOffRing = (kOffSl + kMaxBatch * 4 + 1023) / 1024 * 1024;  // 128B-swizzle atoms
constexpr int kSmemUsed = kOffRing + kStages * kTileBytes;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack for aligning the base to 1024
static_assert(kOffKvNew % 16 == 0 && kOffKcs % 16 == 0 && kOffKx % 8 == 0 &&
              kOffBar % 8 == 0 && kOffOs % 16 == 0 && kOffPbuf % 4 == 0, "smem alignment");
static_assert(kSmemBytes * kCtasPerSm <= 227 * 1024, "two CTAs per SM must fit");

// ------------------------------------------------------------ PTX helpers --
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
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
__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for a barrier phase; give up after kWaitTimeoutNs or when another
// thread of the CTA has already given up.  Never spins without bound.
__device__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > kWaitTimeoutNs) return false;
    }
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
// D += A (16x16 bf16, row) * B (16x8 bf16, col), fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void consumer_sync() {  // the 128 consumer threads only
    asm volatile("bar.sync 1, 128;" ::: "memory");
}

__device__ __forceinline__ void flag_error(int32_t *err, int bits) {
    if (err) atomicOr(err, bits);
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}
__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}
__device__ __forceinline__ uint32_t pack_bf16(__nv_bfloat16 lo, __nv_bfloat16 hi) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(lo)) |
           (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
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

// Walks the pieces of one CTA's tile range in order.
struct Walk {
    int b, g, pg;
    long long f, hi;
};
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
__device__ void walk_start(Walk &w, const int *pre, int B, int Hkv, long long lo, long long hi) {
    w.f = lo;
    w.hi = hi;
    w.b = w.g = w.pg = 0;
    if (lo >= hi) return;
    const int b = seq_of(pre, B, Hkv, lo);
    const int n = pre[b + 1] - pre[b];
    const long long rem = lo - static_cast<long long>(Hkv) * pre[b];
    w.b = b;
    w.g = static_cast<int>(rem / n);
    w.pg = static_cast<int>(rem % n);
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

// ------------------------------------------------------------ row math --
// The new-token rows of (sequence b, KV head g): the 4 query rows 4g..4g+3
// and, when need_k, the key row g with the value row g.  Run by the 128
// consumer threads (warp w owns query row 4g + w; lane l holds dims 2l, 2l+1,
// 64+2l, 65+2l, i.e. both members of two rotate-half pairs).
//
// Query rows: RMSNorm and RoPE in fp32; the angle pos * theta^(-2i/D) is
// formed and reduced modulo 2 pi in double, then sin/cos are taken in fp32.
// Key row: RMSNorm and RoPE in double with double sin/cos, so the one bf16
// rounding on append matches a correctly rounded result of the exact math.
//
// Q_OUT = 0: scaled bf16 hi/lo operand rows into shared memory (qb);
// Q_OUT = 1: fp32 rows to p.q_rot_out (unscaled).
// kv_new receives bf16(k_rot) and v; the pool slot (b, L-1) receives both.
template <int Q_OUT>
__device__ void new_token_rows(const Params &p, int b, int g, int L, bool need_k, uint8_t *sm) {
    const int t = threadIdx.x, w = t >> 5, lane = t & 31;
    const int pos = p.positions[b];
    float2 *cs = reinterpret_cast<float2 *>(sm + kOffCs);
    double2 *kcs = reinterpret_cast<double2 *>(sm + kOffKcs);
    double *kx = reinterpret_cast<double *>(sm + kOffKx);
    double *kss = reinterpret_cast<double *>(sm + kOffKss);
    __nv_bfloat16 *kv_new = reinterpret_cast<__nv_bfloat16 *>(sm + kOffKvNew);

    // Phase A: per-row sums of squares, the rotation angles.
    const int hq = g * kGroup + w;
    const __nv_bfloat16 *qrow = p.q + b * p.q_stride + static_cast<int64_t>(hq) * kHeadDim;
    const __nv_bfloat162 qa = reinterpret_cast<const __nv_bfloat162 *>(qrow)[lane];
    const __nv_bfloat162 qb2 = reinterpret_cast<const __nv_bfloat162 *>(qrow + 64)[lane];
    float x[4] = {__low2float(qa), __high2float(qa), __low2float(qb2), __high2float(qb2)};
    const float ss = warp_sum(x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3]);
    const float r = rsqrtf(ss * (1.0f / kHeadDim) + p.eps);
    {
        const __nv_bfloat162 wa = reinterpret_cast<const __nv_bfloat162 *>(p.w_q)[lane];
        const __nv_bfloat162 wb = reinterpret_cast<const __nv_bfloat162 *>(p.w_q + 64)[lane];
        x[0] = x[0] * r * __low2float(wa);
        x[1] = x[1] * r * __high2float(wa);
        x[2] = x[2] * r * __low2float(wb);
        x[3] = x[3] * r * __high2float(wb);
    }
    if (t < kRotPairs) {
        const double th = static_cast<double>(pos) * p.inv_freq[t];
        const double kq = rint(th * kInvTwoPi);
        double red = fma(-kq, kTwoPiHi, th);
        red = fma(-kq, kTwoPiLo, red);
        float sn, cn;
        sincosf(static_cast<float>(red), &sn, &cn);
        cs[t] = make_float2(cn, sn);
    }
    double kxv = 0.0;
    if (need_k) {
        if (t >= kRotPairs) {
            const double th = static_cast<double>(pos) * p.inv_freq[t - kRotPairs];
            double sn, cn;
            sincos(th, &sn, &cn);
            kcs[t - kRotPairs] = make_double2(cn, sn);
        }
        const __nv_bfloat16 *krow =
            p.k + b * p.k_stride + static_cast<int64_t>(g) * kHeadDim;
        kxv = static_cast<double>(__bfloat162float(krow[t]));
        const double part = warp_sum(kxv * kxv);
        if (lane == 0) kss[w] = part;
    }
    consumer_sync();

    // Phase B: rotate the query rows; normalise the key row.
    {
        const float2 c0 = cs[2 * lane], c1 = cs[2 * lane + 1];
        const float y0 = x[0] * c0.x - x[2] * c0.y;
        const float y2 = x[2] * c0.x + x[0] * c0.y;
        const float y1 = x[1] * c1.x - x[3] * c1.y;
        const float y3 = x[3] * c1.x + x[1] * c1.y;
        if (Q_OUT == 0) {
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
    if (!need_k) return;
    {
        const double tot = kss[0] + kss[1] + kss[2] + kss[3];
        const double rk = 1.0 / sqrt(tot / kHeadDim + static_cast<double>(p.eps));
        kx[t] = kxv * rk * static_cast<double>(__bfloat162float(p.w_k[t]));
    }
    consumer_sync();

    // Phase C: rotate the key row (double), round once, append k and v.
    const int i = t & (kRotPairs - 1);
    const double2 c = kcs[i];
    const double y = t < kRotPairs ? kx[t] * c.x - kx[t + kRotPairs] * c.y
                                   : kx[t] * c.x + kx[t - kRotPairs] * c.y;
    const __nv_bfloat16 kb = __double2bfloat16(y);
    const __nv_bfloat16 vb = (p.v + b * p.v_stride + static_cast<int64_t>(g) * kHeadDim)[t];
    kv_new[t] = kb;
    kv_new[kHeadDim + t] = vb;
    const int slot = L - 1;
    const int page = p.block_table[static_cast<int64_t>(b) * p.max_blocks + slot / kPageSize];
    if (page >= 0 && page < p.num_pages) {
        const int64_t row =
            ((static_cast<int64_t>(page) * 2 * p.Hkv + g) * kPageSize + slot % kPageSize) *
            kHeadDim;
        p.pool[row + t] = kb;
        p.pool[row + static_cast<int64_t>(p.Hkv) * kPageSize * kHeadDim + t] = vb;
    } else if (t == 0) {
        flag_error(p.err, QDEC_FLAG_BAD_PAGE);
    }
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
        const float aA = st.mA == kNegInf ? 0.f : exp2f(st.mA - nA);
        const float aB = st.mB == kNegInf ? 0.f : exp2f(st.mB - nB);
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
    const float pA0 = exp2f(sA0 - bA), pA1 = exp2f(sA1 - bA);
    const float pB0 = exp2f(sB0 - bB), pB1 = exp2f(sB1 - bB);
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

// Log-sum-exp merge of the np pieces of segment sigma (piece ids sigma + j,
// j = j0 .. j0 + np - 1) into out.  128 threads: head t/32, dims 4(t%32)...
__device__ void merge_pieces(const Params &p, int sigma, int b, int g, int j0, int np) {
    const int t = threadIdx.x, h = t >> 5, d0 = (t & 31) * 4;
    float M = kNegInf;
    for (int j = 0; j < np; ++j)
        M = fmaxf(M, __ldcg(p.ws_lse + static_cast<int64_t>(sigma + j0 + j) * kGroup + h));
    float den = 0.f;
    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != kNegInf) {
        for (int j = 0; j < np; ++j) {
            const int64_t pid = sigma + j0 + j;
            const float e = exp2f(__ldcg(p.ws_lse + pid * kGroup + h) - M);
            const float4 o = __ldcg(
                reinterpret_cast<const float4 *>(p.ws_o + (pid * kGroup + h) * kHeadDim + d0));
            den += e;
            num.x += e * o.x;
            num.y += e * o.y;
            num.z += e * o.z;
            num.w += e * o.w;
        }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    __nv_bfloat16 *dst =
        p.out + (static_cast<int64_t>(b) * p.Hq + g * kGroup + h) * kHeadDim + d0;
    reinterpret_cast<uint2 *>(dst)[0] =
        make_uint2(pack_bf16(__float2bfloat16_rn(num.x * inv), __float2bfloat16_rn(num.y * inv)),
                   pack_bf16(__float2bfloat16_rn(num.z * inv), __float2bfloat16_rn(num.w * inv)));
}

// ------------------------------------------------------ attention kernel --
template <bool kFused>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    attention_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *ring = sm + kOffRing;
    const uint32_t full0 = smem_u32(sm + kOffBar);
    const uint32_t empty0 = full0 + kStages * 8;
    volatile int *slot_ok = reinterpret_cast<volatile int *>(sm + kOffSlotOk);
    volatile int *misc = reinterpret_cast<volatile int *>(sm + kOffMisc);  // 0 abort, 1 last, 2 issued
    int *pre = reinterpret_cast<int *>(sm + kOffPre);
    int *sl = reinterpret_cast<int *>(sm + kOffSl);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        misc[0] = 0;
        misc[1] = 0;
        misc[2] = 0;
        fence_mbar_init();
    }
    if (warp == 0) build_prefix(p, pre, sl, blockIdx.x == 0);
    __syncthreads();

    const long long W = static_cast<long long>(p.Hkv) * pre[p.B];
    if (W == 0) return;
    const int G = static_cast<int>(min(static_cast<long long>(p.grid), W));
    if (static_cast<int>(blockIdx.x) >= G) return;  // the whole CTA leaves together
    const long long lo = static_cast<long long>(blockIdx.x) * W / G;
    const long long hi = static_cast<long long>(blockIdx.x + 1) * W / G;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------ TMA producer --
        if (lane == 0) {
            Walk w;
            walk_start(w, pre, p.B, p.Hkv, lo, hi);
            uint32_t i = 0;
            bool stop = false;
            while (!stop && w.f < w.hi) {
                const int cnt = piece_len(w, pre);
                const int32_t *bt = p.block_table + static_cast<int64_t>(w.b) * p.max_blocks;
                for (int k = 0; k < cnt; ++k, ++i) {
                    const int slot = i % kStages;
                    const uint32_t full = full0 + 8 * slot;
                    if (i >= kStages &&
                        !mbar_wait_bounded(empty0 + 8 * slot, ((i / kStages) - 1) & 1, misc)) {
                        misc[0] = 1;
                        flag_error(p.err, QDEC_FLAG_TIMEOUT);
                        stop = true;
                        break;
                    }
                    const int page = bt[w.pg + k];
                    if (page >= 0 && page < p.num_pages) {
                        slot_ok[slot] = 1;
                        mbar_arrive_expect_tx(full, kTileBytes);
                        const int yk = (page * 2 * p.Hkv + w.g) * kPageSize;
                        const int yv = yk + p.Hkv * kPageSize;
                        const uint32_t dst = smem_u32(ring + slot * kTileBytes);
                        tma_load_2d(dst, &kv_map, 0, yk, full);
                        tma_load_2d(dst + kTileHalfBytes, &kv_map, 64, yk, full);
                        tma_load_2d(dst + kPlaneBytes, &kv_map, 0, yv, full);
                        tma_load_2d(dst + kPlaneBytes + kTileHalfBytes, &kv_map, 64, yv, full);
                    } else {
                        slot_ok[slot] = 0;
                        flag_error(p.err, QDEC_FLAG_BAD_PAGE);
                        mbar_arrive(full);
                    }
                }
                if (!stop) walk_next(w, pre, p.Hkv, cnt);
            }
            misc[2] = static_cast<int>(i);
        }
    } else {
        // ---------------------------------------------- consumer warps --
        __nv_bfloat16 *qb = reinterpret_cast<__nv_bfloat16 *>(sm + kOffQb);
        const __nv_bfloat16 *kv_new = reinterpret_cast<const __nv_bfloat16 *>(sm + kOffKvNew);
        __nv_bfloat16 *pbuf = reinterpret_cast<__nv_bfloat16 *>(sm + kOffPbuf) + warp * 8 * 16;
        float *ms = reinterpret_cast<float *>(sm + kOffMs);
        float *ls = reinterpret_cast<float *>(sm + kOffLs);
        float *os = reinterpret_cast<float *>(sm + kOffOs);
        const int tg = lane >> 2, c = lane & 3;

        Walk w;
        walk_start(w, pre, p.B, p.Hkv, lo, hi);
        uint32_t i = 0;
        while (w.f < w.hi) {
            const int cnt = piece_len(w, pre);
            const int b = w.b, g = w.g, pg0 = w.pg;
            const int L = sl[b];
            const int n = pre[b + 1] - pre[b];
            const bool has_last = pg0 + cnt == n;

            // prologue: the group's 4 query rows as bf16 hi/lo MMA operands
            if (kFused) {
                new_token_rows<0>(p, b, g, L, has_last, sm);
            } else {
                const float *src =
                    p.q_rot_in + (static_cast<int64_t>(b) * p.Hq + g * kGroup + warp) * kHeadDim;
                const float2 ya = reinterpret_cast<const float2 *>(src)[lane];
                const float2 yb = reinterpret_cast<const float2 *>(src + 64)[lane];
                const float ys[4] = {ya.x * p.qscale, ya.y * p.qscale, yb.x * p.qscale,
                                     yb.y * p.qscale};
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
            consumer_sync();
            uint32_t qf[8][2];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const __nv_bfloat16 *row = qb + tg * kQbStride + 16 * j + 2 * c;
                qf[j][0] = *reinterpret_cast<const uint32_t *>(row);
                qf[j][1] = *reinterpret_cast<const uint32_t *>(row + 8);
            }

            WarpState st;
            st.mA = st.mB = kNegInf;
            st.lA = st.lB = 0.f;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt)
                st.o[mt][0] = st.o[mt][1] = st.o[mt][2] = st.o[mt][3] = 0.f;

            for (int k = 0; k < cnt; ++k, ++i) {
                if (static_cast<int>(i & 3) != warp) continue;
                const int slot = i % kStages;
                const bool ok = mbar_wait_bounded(full0 + 8 * slot, (i / kStages) & 1, misc);
                if (!ok && lane == 0) {
                    misc[0] = 1;
                    flag_error(p.err, QDEC_FLAG_TIMEOUT);
                }
                const int pg = pg0 + k;
                const int ntok = min(kPageSize, L - pg * kPageSize);
                if (ok && slot_ok[slot]) {
                    uint8_t *tile = ring + slot * kTileBytes;
                    const bool patch = kFused && pg == n - 1;
                    if (patch || ntok < kPageSize) fix_tile(tile, ntok, patch, kv_new, lane);
                    const uint32_t ks = smem_u32(tile);
                    tile_math(ks, ks + kPlaneBytes, qf, ntok, lane, st, pbuf);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty0 + 8 * slot);
            }

            // epilogue: combine hi/lo columns, then the four warps' states
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
                    oA[16 * mt + tg] = st.o[mt][0];
                    oB[16 * mt + tg] = st.o[mt][1];
                    oA[16 * mt + tg + 8] = st.o[mt][2];
                    oB[16 * mt + tg + 8] = st.o[mt][3];
                }
                if (tg == 0) {
                    ms[warp * kGroup + hA] = st.mA;
                    ms[warp * kGroup + hB] = st.mB;
                    ls[warp * kGroup + hA] = st.lA;
                    ls[warp * kGroup + hB] = st.lB;
                }
            }
            consumer_sync();
            {
                const int h = tid >> 5, d0 = (tid & 31) * 4;
                float M = kNegInf;
#pragma unroll
                for (int q = 0; q < kConsumerWarps; ++q) M = fmaxf(M, ms[q * kGroup + h]);
                float den = 0.f;
                float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
                if (M != kNegInf) {
#pragma unroll
                    for (int q = 0; q < kConsumerWarps; ++q) {
                        const float mq = ms[q * kGroup + h];
                        const float e = mq == kNegInf ? 0.f : exp2f(mq - M);
                        const float4 o4 =
                            *reinterpret_cast<const float4 *>(os + (q * kGroup + h) * kHeadDim + d0);
                        den += e * ls[q * kGroup + h];
                        num.x += e * o4.x;
                        num.y += e * o4.y;
                        num.z += e * o4.z;
                        num.w += e * o4.w;
                    }
                }
                const float inv = den > 0.f ? 1.f / den : 0.f;
                const long long seg0 = static_cast<long long>(p.Hkv) * pre[b] +
                                       static_cast<long long>(g) * n;
                const int j0 = cta_of(seg0, W, G);
                const int np = cta_of(seg0 + n - 1, W, G) - j0 + 1;
                const int sigma = b * p.Hkv + g;
                if (np == 1) {
                    __nv_bfloat16 *dst =
                        p.out + (static_cast<int64_t>(b) * p.Hq + g * kGroup + h) * kHeadDim + d0;
                    reinterpret_cast<uint2 *>(dst)[0] = make_uint2(
                        pack_bf16(__float2bfloat16_rn(num.x * inv), __float2bfloat16_rn(num.y * inv)),
                        pack_bf16(__float2bfloat16_rn(num.z * inv), __float2bfloat16_rn(num.w * inv)));
                } else {
                    const int64_t pid = sigma + static_cast<int64_t>(blockIdx.x);
                    *reinterpret_cast<float4 *>(p.ws_o + (pid * kGroup + h) * kHeadDim + d0) =
                        make_float4(num.x * inv, num.y * inv, num.z * inv, num.w * inv);
                    if ((tid & 31) == 0)
                        p.ws_lse[pid * kGroup + h] = den > 0.f ? M + log2f(den) : kNegInf;
                    if (kFused) {
                        __threadfence();
                        consumer_sync();
                        if (tid == 0) {
                            const int prev = atomicAdd(p.ws_cnt + sigma, 1);
                            misc[1] = prev == np - 1;
                        }
                        consumer_sync();
                        if (misc[1]) {
                            __threadfence();
                            merge_pieces(p, sigma, b, g, j0, np);
                            if (tid == 0) p.ws_cnt[sigma] = 0;  // ready for the next launch
                        }
                    }
                }
            }
            walk_next(w, pre, p.Hkv, cnt);
        }
    }
    __syncthreads();
    // A wait that gave up may leave bulk copies in flight: let them land
    // (bounded) before the CTA's shared memory is released.
    if (tid == 0 && misc[0]) {
        const uint32_t issued = static_cast<uint32_t>(misc[2]);
        const uint32_t first = issued > kStages ? issued - kStages : 0;
        volatile int never = 0;
        for (uint32_t t = first; t < issued; ++t)
            mbar_wait_bounded(full0 + 8 * (t % kStages), (t / kStages) & 1, &never);
    }
}

// ---------------------------------------------------------- append kernel --
// Steps 1-3 for (KV head blockIdx.x, sequence blockIdx.y): q rows to
// q_rot_out, k and v into the pool.
__global__ void __launch_bounds__(128) append_rope_kernel(const __grid_constant__ Params p) {
    __shared__ __align__(16) uint8_t sm[kPrologueBytes];
    const int g = blockIdx.x, b = blockIdx.y;
    const int L = p.seq_lens[b];
    if (L < 1 || L > p.max_blocks * kPageSize) {
        if (threadIdx.x == 0 && g == 0) flag_error(p.err, QDEC_FLAG_BAD_SEQLEN);
        return;
    }
    new_token_rows<1>(p, b, g, L, true, sm);
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
    merge_pieces(p, sigma, b, g, j0, np);
}

bool g_attr_set[2][64];

}  // namespace

size_t attention_smem_bytes() { return kSmemBytes; }

static int current_device() {
    int d = 0;
    cudaGetDevice(&d);
    return d < 64 ? d : 63;
}

cudaError_t launch_attention(const Params &p, const CUtensorMap &kv_map, bool fused,
                             cudaStream_t s) {
    const int dev = current_device();
    if (!g_attr_set[fused][dev]) {
        cudaError_t e = fused ? cudaFuncSetAttribute(attention_kernel<true>,
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     kSmemBytes)
                              : cudaFuncSetAttribute(attention_kernel<false>,
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     kSmemBytes);
        if (e != cudaSuccess) return e;
        g_attr_set[fused][dev] = true;
    }
    if (fused)
        attention_kernel<true><<<p.grid, kThreads, kSmemBytes, s>>>(kv_map, p);
    else
        attention_kernel<false><<<p.grid, kThreads, kSmemBytes, s>>>(kv_map, p);
    return cudaGetLastError();
}

cudaError_t launch_append_rope(const Params &p, cudaStream_t s) {
    append_rope_kernel<<<dim3(p.Hkv, p.B), 128, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_merge(const Params &p, cudaStream_t s) {
    merge_kernel<<<p.B * p.Hkv, 128, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace qdec
