// qdec_api.cu -- host side of the libqdec C ABI: argument checks, workspace
// layout, the TMA descriptor of the KV pool, and kernel launches.  No call
// here allocates device memory; the only host-side arithmetic is the RoPE
// frequency table rope_theta^(-2i/D), a per-shape constant passed to the
// kernels by value.
#include "qdec_internal.h"
#include "qdec.h"

#include <math.h>

#include <algorithm>
#include <atomic>
#include <mutex>

namespace {

using qdec::Params;

constexpr int kVersion = 20000;  // 2.0.0: the prefill entry points gained a workspace and an angle table

// ----------------------------------------------------------- device info --
// Per-device attribute caches: calls may come from several host threads, so
// the entries are atomics (every writer stores the same value).
int cached_attribute(std::atomic<int> (&cache)[64], cudaDeviceAttr attr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, attr, dev) != cudaSuccess) return 0;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

int sm_count_of_current_device() {
    static std::atomic<int> cache[64];
    return cached_attribute(cache, cudaDevAttrMultiProcessorCount);
}

// ------------------------------------------------------------ validation --
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

qdec_status check_shape(const qdec_shape *s) {
    if (!s) return QDEC_ERR_INVALID_ARG;
    if (s->batch < 1 || s->num_q_heads < 1 || s->num_kv_heads < 1 || s->head_dim < 1 ||
        s->page_size < 1 || s->num_pages < 1 || s->max_blocks_per_seq < 1 ||
        s->max_seq_len < 1 || s->num_ctas < 0)
        return QDEC_ERR_INVALID_ARG;
    if ((s->launch_flags & ~(QDEC_LAUNCH_OVERLAP_PREVIOUS | QDEC_LAUNCH_PREFILL_PAGES_READY |
                             QDEC_LAUNCH_TEST_WITHHOLD_TILE)) != 0)
        return QDEC_ERR_INVALID_ARG;
    if (!(s->rope_theta > 0.f) || !(s->eps >= 0.f) || !(s->sm_scale >= 0.f) ||
        !isfinite(s->rope_theta) || !isfinite(s->eps) || !isfinite(s->sm_scale))
        return QDEC_ERR_INVALID_ARG;
    if (static_cast<int64_t>(s->max_seq_len) >
        static_cast<int64_t>(s->max_blocks_per_seq) * s->page_size)
        return QDEC_ERR_INVALID_ARG;
    if (s->head_dim != qdec::kHeadDim || s->page_size != qdec::kPageSize ||
        s->num_q_heads != qdec::kGroup * s->num_kv_heads || s->batch > qdec::kMaxBatch)
        return QDEC_ERR_UNSUPPORTED;
    // TMA row coordinates of the pool are 32-bit
    if (static_cast<int64_t>(s->num_pages) * 2 * s->num_kv_heads * qdec::kPageSize >= (1ll << 31))
        return QDEC_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(s->max_blocks_per_seq) * qdec::kPageSize >= (1ll << 31))
        return QDEC_ERR_UNSUPPORTED;
    return QDEC_OK;
}

qdec_status check_row_input(const void *p, int64_t stride, int rows) {
    if (!p) return QDEC_ERR_INVALID_ARG;
    if (!aligned16(p) || stride % 8 != 0 || stride < static_cast<int64_t>(rows) * qdec::kHeadDim)
        return QDEC_ERR_INVALID_ARG;
    return QDEC_OK;
}

int smem_per_sm_of_current_device() {
    static std::atomic<int> cache[64];
    return cached_attribute(cache, cudaDevAttrMaxSharedMemoryPerMultiprocessor);
}

// ----------------------------------------------------------------- plan --
int64_t max_tiles(const qdec_shape *s) {
    return static_cast<int64_t>(s->batch) * s->num_kv_heads *
           ((s->max_seq_len + qdec::kPageSize - 1) / qdec::kPageSize);
}

// Work layout of the attention kernel (see qdec_kernels.cu): a function of
// the shape and the device only, never of the lengths in seq_lens.
struct Plan {
    int grid;        // CTAs launched
    int stages;      // ring depth
    int cluster;     // 0 = flat partition, else CTAs per cluster
    int chunks;      // cluster layout: chunks (clusters) per segment
};

// Below this many tiles per CTA the per-CTA stream is too short to hide the
// global merge, so the cluster layout is used.
constexpr int64_t kFlatMinTilesPerCta = 32;

// Deepest ring (a multiple of the 4 consumer warps) that still lets the
// layout's CTAs per SM share it.
int ring_cap(const qdec_shape *s, int cluster, bool fp8) {
    int per_sm = smem_per_sm_of_current_device();
    if (per_sm <= 0) per_sm = 228 * 1024;
    const int w = qdec::kConsumerWarps;
    int cap = qdec::kMaxStages / w * w;
    while (cap > w &&
           static_cast<int64_t>(qdec::ctas_per_sm(cluster > 0, fp8)) *
                   static_cast<int64_t>(qdec::attention_smem_bytes(s->batch, cap, cluster, fp8) +
                                        1024) >
               static_cast<int64_t>(per_sm))
        cap -= w;
    return cap;
}

// Ring depth: a CTA's whole share of tiles when that is small (so a launch
// can prefetch everything before its inputs are ready), else the cap; always
// a multiple of the consumer warp count (see the attention kernel).
int clamp_stages(int64_t want, int cap) {
    const int w = qdec::kConsumerWarps;
    int64_t st = (want + w - 1) / w * w;
    if (st < w) st = w;
    return static_cast<int>(st < cap ? st : cap);
}

// CTAs of cluster size c that fit on the device at once (cached per device
// and pool type).
int64_t cluster_capacity(const qdec_shape *s, int c, int cap, bool fp8) {
    static std::mutex mu;
    static int cache[64][2][qdec::kMaxCluster + 1];
    static size_t cache_smem[64][2][qdec::kMaxCluster + 1];
    const size_t smem = qdec::attention_smem_bytes(s->batch, cap, c, fp8);
    const int t = fp8 ? 1 : 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = -1;
    int n = 0;
    if (dev >= 0) {
        std::lock_guard<std::mutex> lock(mu);
        n = cache_smem[dev][t][c] == smem ? cache[dev][t][c] : 0;
        if (n == 0) {
            // a failed query leaves no error behind, but an error the caller
            // has not read yet stays pending
            const cudaError_t pending = cudaPeekAtLastError();
            n = qdec::max_active_clusters(c, smem, fp8);
            if (pending == cudaSuccess) cudaGetLastError();
            if (n <= 0) n = -1;
            cache[dev][t][c] = n;
            cache_smem[dev][t][c] = smem;
        }
    }
    if (n > 0) return static_cast<int64_t>(n) * c;
    int sms = sm_count_of_current_device();
    if (sms <= 0) sms = 1;
    return static_cast<int64_t>(sms) * qdec::kCtasPerSm / c * c;  // no device: plain estimate
}

// allow_cluster = false for the three-call path, whose merge kernel reads
// the flat layout.  num_ctas > 0 forces the flat layout on that grid.
//
// Cluster layout: each (sequence, KV head) is cut into K chunks of C CTAs.
// Chunks meet through the workspace (a fence, an atomic and a second pass:
// the costly merge), CTAs of a cluster through distributed shared memory.
// So the fewest chunks K that still give enough CTAs to stream the pages:
// about kBytesPerCta each, or 60% of the resident CTAs, whichever is fewer
// (a smaller grid also leaves room for the next launch to start early).  For
// that K the largest cluster that fits on the device in one wave.
constexpr double kBytesPerCta = 96.0 * 1024;
constexpr double kGridShare = 0.6;

Plan plan_for(const qdec_shape *s, bool allow_cluster, bool fp8) {
    int sms = sm_count_of_current_device();
    if (sms <= 0) sms = 1;
    const int64_t target = static_cast<int64_t>(sms) * qdec::kCtasPerSm;
    const int64_t wmax = max_tiles(s);
    Plan pl{};
    const int64_t per_cta = (wmax + target - 1) / target;
    const int64_t segs = static_cast<int64_t>(s->batch) * s->num_kv_heads;
    const int64_t nmax = (s->max_seq_len + qdec::kPageSize - 1) / qdec::kPageSize;
    // Few segments: every one can have CTAs of its own within the grid share,
    // so the cluster layout's per-segment split adapts to the actual lengths
    // whatever the bound (an engine plans one graph for its longest context).
    const bool few_segments = static_cast<double>(segs) <= kGridShare * static_cast<double>(target);
    if (s->num_ctas == 0 && allow_cluster && (per_cta < kFlatMinTilesPerCta || few_segments)) {
        const double bytes =
            static_cast<double>(wmax) * (fp8 ? qdec::kFp8TileBytes : qdec::kTileBytes);
        const double want = std::min(kGridShare * static_cast<double>(target), bytes / kBytesPerCta);
        Plan widest{};
        for (int64_t k = 1; k <= nmax && pl.grid == 0; ++k) {
            if (segs * k > target) break;  // not even one CTA per chunk fits
            for (int c = qdec::kMaxCluster; c >= 1; --c) {
                if (c * k > nmax && c > 1) continue;  // every CTA gets a page
                const int64_t t = (nmax + c * k - 1) / (c * k);
                const int64_t grid = c * segs * k;
                const int cap = ring_cap(s, c, fp8);
                const int need = qdec::min_stages(c, fp8);
                if (cap < need || grid > cluster_capacity(s, c, cap, fp8)) continue;
                Plan cand{};
                cand.cluster = c;
                cand.chunks = static_cast<int>(k);
                cand.grid = static_cast<int>(grid);
                cand.stages = std::max(clamp_stages(t + 1, cap), need);
                if (grid > widest.grid) widest = cand;
                if (static_cast<double>(grid) >= want) pl = cand;
                break;  // the largest cluster that fits, for this k
            }
        }
        if (pl.grid == 0 && widest.grid > 0 && (per_cta < kFlatMinTilesPerCta / 2 || few_segments))
            pl = widest;
        if (pl.grid > 0) return pl;
    }
    // flat layout: a whole number of CTAs per SM for the pool type in the
    // fused kernel; the three-call path keeps two per SM for both types, as
    // its merge kernel (which knows no pool type) rebuilds the piece layout
    // from the grid
    const int64_t flat_target =
        static_cast<int64_t>(sms) * (allow_cluster ? qdec::ctas_per_sm(false, fp8) : qdec::kCtasPerSm);
    const int64_t g = s->num_ctas > 0 ? s->num_ctas : std::min(flat_target, wmax);
    pl.grid = static_cast<int>(g);
    pl.stages = clamp_stages((wmax + g - 1) / g, ring_cap(s, 0, fp8));
    return pl;
}

// The FP8 pool's scale windows need an even number of KV heads.
bool fp8_supported(const qdec_shape *s) { return s->num_kv_heads % 2 == 0; }

// Grid bound covering both layouts and both pool types (sizes the
// workspace, so one workspace serves every entry point).
int attention_grid(const qdec_shape *s) {
    int g = std::max(plan_for(s, true, false).grid, plan_for(s, false, false).grid);
    if (fp8_supported(s))
        g = std::max(g, std::max(plan_for(s, true, true).grid, plan_for(s, false, true).grid));
    return g;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// qdec_step on the flat layout (many segments: each CTA walks several) runs
// as two launches, the new-token kernel and then the attention in decode
// mode as its programmatic dependent: there the fused kernel's per-piece
// new-token work holds the consumer warps of a CTA while its ring fills,
// which costs more than the extra launch (measured on 64 ragged sequences:
// bf16 pool 182.9 -> 172.6 us per layer-step).  On the cluster layout (one
// piece per CTA, latency-bound) the single launch is faster.
bool step_in_two_launches(const qdec_shape *s, bool fp8) {
    return plan_for(s, true, fp8).cluster == 0;
}

struct WorkspaceLayout {
    size_t cnt, lse, o, o_end, qrot, total;
};

// counters [B*Hkv] int32 | partial lse [pieces][G] f32 | partial o [pieces][G][D] f32
// with pieces <= grid + B*Hkv for either layout (flat: each CTA adds at most
// one piece per segment it starts in, plus its first; cluster: one per
// cluster) | q_rot [B][Hq][D] f32 where qdec_step runs in two launches.
WorkspaceLayout workspace_layout(const qdec_shape *s) {
    const size_t segs = static_cast<size_t>(s->batch) * s->num_kv_heads;
    const size_t pieces = static_cast<size_t>(attention_grid(s)) + segs;
    WorkspaceLayout l;
    l.cnt = 0;
    l.lse = round256(segs * sizeof(int32_t));
    l.o = l.lse + round256(pieces * qdec::kGroup * sizeof(float));
    l.o_end = l.o + pieces * qdec::kGroup * qdec::kHeadDim * sizeof(float);
    l.qrot = round256(l.o_end);
    const bool two = step_in_two_launches(s, false) ||
                     (fp8_supported(s) && step_in_two_launches(s, true));
    l.total = l.qrot + (two ? static_cast<size_t>(s->batch) * s->num_q_heads * qdec::kHeadDim *
                                  sizeof(float)
                            : 0);
    return l;
}

// RoPE frequencies rope_theta^(-2i/D) in double, cached per theta.
void fill_inv_freq(double *dst, float theta) {
    static std::mutex mu;
    static float cached_theta = -1.f;
    static double table[qdec::kRotPairs];
    std::lock_guard<std::mutex> lock(mu);
    if (cached_theta != theta) {
        for (int i = 0; i < qdec::kRotPairs; ++i)
            table[i] = pow(static_cast<double>(theta), -2.0 * i / qdec::kHeadDim);
        cached_theta = theta;
    }
    for (int i = 0; i < qdec::kRotPairs; ++i) dst[i] = table[i];
}

void fill_common(Params &p, const qdec_shape *s, bool allow_cluster, bool fp8 = false) {
    p.B = s->batch;
    p.Hq = s->num_q_heads;
    p.Hkv = s->num_kv_heads;
    p.num_pages = s->num_pages;
    p.max_blocks = s->max_blocks_per_seq;
    p.eps = s->eps;
    const double scale =
        s->sm_scale > 0.f ? s->sm_scale : 1.0 / sqrt(static_cast<double>(s->head_dim));
    p.qscale = static_cast<float>(scale * 1.4426950408889634074);  // * log2(e)
    const Plan pl = plan_for(s, allow_cluster, fp8);
    p.grid = pl.grid;
    p.stages = pl.stages;
    p.cluster = pl.cluster;
    p.chunks = pl.chunks;
    p.pdl = (s->launch_flags & QDEC_LAUNCH_OVERLAP_PREVIOUS) != 0;
    p.withhold_first = (s->launch_flags & QDEC_LAUNCH_TEST_WITHHOLD_TILE) != 0;
    p.wait_cycles = p.withhold_first ? qdec::kTestWaitCycles : qdec::kWaitTimeoutCycles;
    fill_inv_freq(p.inv_freq, s->rope_theta);
}

void bind_workspace(Params &p, const qdec_shape *s, void *ws) {
    const WorkspaceLayout l = workspace_layout(s);
    uint8_t *base = static_cast<uint8_t *>(ws);
    p.ws_cnt = reinterpret_cast<int32_t *>(base + l.cnt);
    p.ws_lse = reinterpret_cast<float *>(base + l.lse);
    p.ws_o = reinterpret_cast<float *>(base + l.o);
    p.ws_pieces = static_cast<long long>((l.o_end - l.o) /
                                         (qdec::kGroup * qdec::kHeadDim * sizeof(float)));
}

// ------------------------------------------------------- TMA descriptor --
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// The pool as a 5-D tensor whose box is one page tile: dims (64 of D,
// token [16], half of D [2], plane K/V [2], page*2*Hkv + head), strides
// (2, 256, 128, Hkv*4096, 4096) bytes.  The plane and head dimensions
// address the same bytes two ways (the K/V plane step is Hkv heads), which
// the hardware allows; every box stays inside the pool because the last
// coordinate is page*2*Hkv + head with head < Hkv.  128-byte rows are
// swizzled so the tile math reads shared memory without bank conflicts.
qdec_status encode_pool_map(CUtensorMap *map, const qdec_shape *s, const void *pool) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return QDEC_ERR_CUDA;
    const cuuint64_t plane = static_cast<cuuint64_t>(qdec::kPageSize) * qdec::kHeadDim * 2;
    const cuuint64_t dims[5] = {64, static_cast<cuuint64_t>(qdec::kPageSize), 2, 2,
                                static_cast<cuuint64_t>(s->num_pages) * 2 * s->num_kv_heads};
    const cuuint64_t strides[4] = {qdec::kHeadDim * 2, 128,
                                   static_cast<cuuint64_t>(s->num_kv_heads) * plane, plane};
    const cuuint32_t box[5] = {64, static_cast<cuuint32_t>(qdec::kPageSize), 2, 2, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(pool), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? QDEC_OK : QDEC_ERR_CUDA;
}

// The same 5-D view of the bf16 pool with a box of one (page, plane, half
// of D) region: 16 tokens x 64 dims, 2 KiB (the tensor-core prefill brings
// each region of four pages side by side).
qdec_status encode_pool_region_map(CUtensorMap *map, const qdec_shape *s, const void *pool) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return QDEC_ERR_CUDA;
    const cuuint64_t plane = static_cast<cuuint64_t>(qdec::kPageSize) * qdec::kHeadDim * 2;
    const cuuint64_t dims[5] = {64, static_cast<cuuint64_t>(qdec::kPageSize), 2, 2,
                                static_cast<cuuint64_t>(s->num_pages) * 2 * s->num_kv_heads};
    const cuuint64_t strides[4] = {qdec::kHeadDim * 2, 128,
                                   static_cast<cuuint64_t>(s->num_kv_heads) * plane, plane};
    const cuuint32_t box[5] = {64, static_cast<cuuint32_t>(qdec::kPageSize), 1, 1, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(pool), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? QDEC_OK : QDEC_ERR_CUDA;
}

// The FP8 pool as a 4-D tensor whose box is one page tile: dims (128 bytes
// of D, token [16], plane K/V [2], page*2*Hkv + head), strides (128,
// Hkv*2048, 2048) bytes; 128-byte rows swizzled as in the bf16 map.
qdec_status encode_pool_map_fp8(CUtensorMap *map, const qdec_shape *s, const void *pool8) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return QDEC_ERR_CUDA;
    const cuuint64_t plane = static_cast<cuuint64_t>(qdec::kFp8PlaneBytes);
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(qdec::kHeadDim),
                                static_cast<cuuint64_t>(qdec::kPageSize), 2,
                                static_cast<cuuint64_t>(s->num_pages) * 2 * s->num_kv_heads};
    const cuuint64_t strides[3] = {qdec::kHeadDim,
                                   static_cast<cuuint64_t>(s->num_kv_heads) * plane, plane};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(qdec::kHeadDim),
                               static_cast<cuuint32_t>(qdec::kPageSize), 2, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(pool8), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? QDEC_OK : QDEC_ERR_CUDA;
}

// The FP8 pool's 4-D view with a box of one (page, plane): 16 tokens x 128
// codes, 2 KiB (the tensor-core prefill brings K and V separately).
qdec_status encode_pool_plane_map_fp8(CUtensorMap *map, const qdec_shape *s, const void *pool8) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return QDEC_ERR_CUDA;
    const cuuint64_t plane = static_cast<cuuint64_t>(qdec::kFp8PlaneBytes);
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(qdec::kHeadDim),
                                static_cast<cuuint64_t>(qdec::kPageSize), 2,
                                static_cast<cuuint64_t>(s->num_pages) * 2 * s->num_kv_heads};
    const cuuint64_t strides[3] = {qdec::kHeadDim,
                                   static_cast<cuuint64_t>(s->num_kv_heads) * plane, plane};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(qdec::kHeadDim),
                               static_cast<cuuint32_t>(qdec::kPageSize), 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(pool8), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? QDEC_OK : QDEC_ERR_CUDA;
}

// A row-major bf16 matrix [rows][cols] (row stride `stride` elements) as a
// 2-D tensor with box_rows x 64 boxes, 128-byte swizzled.
qdec_status encode_rows_map(CUtensorMap *map, const void *base, int64_t rows, int64_t cols,
                            int64_t stride, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return QDEC_ERR_CUDA;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(stride) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? QDEC_OK : QDEC_ERR_CUDA;
}

qdec_status cuda_status(cudaError_t e) { return e == cudaSuccess ? QDEC_OK : QDEC_ERR_CUDA; }

qdec_status check_new_token_args(const qdec_shape *shape, const qdec_bf16 *q, int64_t q_stride,
                                 const qdec_bf16 *k, int64_t k_stride, const qdec_bf16 *v,
                                 int64_t v_stride, const qdec_bf16 *q_norm_w,
                                 const qdec_bf16 *k_norm_w, const int32_t *positions,
                                 const int32_t *seq_lens, const int32_t *block_table) {
    qdec_status st = check_shape(shape);
    if (st != QDEC_OK) return st;
    if ((st = check_row_input(q, q_stride, shape->num_q_heads)) != QDEC_OK) return st;
    if ((st = check_row_input(k, k_stride, shape->num_kv_heads)) != QDEC_OK) return st;
    if ((st = check_row_input(v, v_stride, shape->num_kv_heads)) != QDEC_OK) return st;
    if (!q_norm_w || !k_norm_w || !positions || !seq_lens || !block_table)
        return QDEC_ERR_INVALID_ARG;
    if (!aligned16(q_norm_w) || !aligned16(k_norm_w)) return QDEC_ERR_INVALID_ARG;
    return QDEC_OK;
}

qdec_status check_workspace(const qdec_shape *shape, const void *ws, size_t bytes) {
    if (!ws || !aligned16(ws)) return QDEC_ERR_WORKSPACE;
    if (bytes < workspace_layout(shape).total) return QDEC_ERR_WORKSPACE;
    return QDEC_OK;
}

// The pool an entry point works on: bf16, or E4M3 codes with their scales.
struct PoolArg {
    const void *data;
    const float *scale;  // FP8 only
    bool fp8;
};

qdec_status check_pool(const qdec_shape *shape, const PoolArg &pool) {
    if (!pool.data || !aligned16(pool.data)) return QDEC_ERR_INVALID_ARG;
    if (!pool.fp8) return QDEC_OK;
    if (!fp8_supported(shape)) return QDEC_ERR_UNSUPPORTED;
    if (!pool.scale || !aligned16(pool.scale)) return QDEC_ERR_INVALID_ARG;
    return QDEC_OK;
}

void bind_pool(Params &p, const PoolArg &pool) {
    if (pool.fp8) {
        p.pool8 = static_cast<uint8_t *>(const_cast<void *>(pool.data));
        p.kv_scale = pool.scale;
    } else {
        p.pool = static_cast<__nv_bfloat16 *>(const_cast<void *>(pool.data));
    }
}

qdec_status encode_map(CUtensorMap *map, const qdec_shape *shape, const PoolArg &pool) {
    return pool.fp8 ? encode_pool_map_fp8(map, shape, pool.data)
                    : encode_pool_map(map, shape, pool.data);
}

void bind_new_token(Params &p, const qdec_bf16 *q, int64_t q_stride, const qdec_bf16 *k,
                    int64_t k_stride, const qdec_bf16 *v, int64_t v_stride,
                    const qdec_bf16 *q_norm_w, const qdec_bf16 *k_norm_w,
                    const int32_t *positions, const int32_t *seq_lens,
                    const int32_t *block_table, const void *rope_table) {
    p.q = reinterpret_cast<const __nv_bfloat16 *>(q);
    p.k = reinterpret_cast<const __nv_bfloat16 *>(k);
    p.v = reinterpret_cast<const __nv_bfloat16 *>(v);
    p.q_stride = q_stride;
    p.k_stride = k_stride;
    p.v_stride = v_stride;
    p.w_q = reinterpret_cast<const __nv_bfloat16 *>(q_norm_w);
    p.w_k = reinterpret_cast<const __nv_bfloat16 *>(k_norm_w);
    p.positions = positions;
    p.seq_lens = seq_lens;
    p.block_table = block_table;
    p.rope = static_cast<const qdec::RopeEntry *>(rope_table);
}

qdec_status append_rope_impl(const qdec_shape *shape, const qdec_bf16 *q, int64_t q_stride,
                             const qdec_bf16 *k, int64_t k_stride, const qdec_bf16 *v,
                             int64_t v_stride, const qdec_bf16 *q_norm_w,
                             const qdec_bf16 *k_norm_w, const int32_t *positions,
                             const int32_t *seq_lens, const int32_t *block_table,
                             const void *rope_table, const PoolArg &pool, float *q_rot,
                             int32_t *err_flag, void *stream) {
    qdec_status st = check_new_token_args(shape, q, q_stride, k, k_stride, v, v_stride, q_norm_w,
                                          k_norm_w, positions, seq_lens, block_table);
    if (st != QDEC_OK) return st;
    if ((st = check_pool(shape, pool)) != QDEC_OK) return st;
    if (rope_table && !aligned16(rope_table)) return QDEC_ERR_INVALID_ARG;
    if (!q_rot || !aligned16(q_rot)) return QDEC_ERR_INVALID_ARG;
    Params p{};
    fill_common(p, shape, false, pool.fp8);
    bind_new_token(p, q, q_stride, k, k_stride, v, v_stride, q_norm_w, k_norm_w, positions,
                   seq_lens, block_table, rope_table);
    bind_pool(p, pool);
    p.q_rot_out = q_rot;
    p.err = err_flag;
    return cuda_status(qdec::launch_append_rope(p, pool.fp8, static_cast<cudaStream_t>(stream)));
}

qdec_status attn_split_impl(const qdec_shape *shape, const float *q_rot, const PoolArg &pool,
                            const int32_t *block_table, const int32_t *seq_lens, void *workspace,
                            size_t workspace_bytes, qdec_bf16 *out, int32_t *err_flag,
                            void *stream) {
    qdec_status st = check_shape(shape);
    if (st != QDEC_OK) return st;
    if ((st = check_pool(shape, pool)) != QDEC_OK) return st;
    if (!q_rot || !block_table || !seq_lens || !out) return QDEC_ERR_INVALID_ARG;
    if (!aligned16(q_rot) || !aligned16(out)) return QDEC_ERR_INVALID_ARG;
    if ((st = check_workspace(shape, workspace, workspace_bytes)) != QDEC_OK) return st;
    Params p{};
    fill_common(p, shape, false, pool.fp8);
    p.q_rot_in = q_rot;
    p.seq_lens = seq_lens;
    p.block_table = block_table;
    bind_pool(p, pool);
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.err = err_flag;
    p.pdl = 0;  // reads what the append just wrote: no overlap
    bind_workspace(p, shape, workspace);
    CUtensorMap map;
    if ((st = encode_map(&map, shape, pool)) != QDEC_OK) return st;
    return cuda_status(
        qdec::launch_attention(p, map, qdec::kAttnSplit, pool.fp8,
                               static_cast<cudaStream_t>(stream)));
}

qdec_status step_impl(const qdec_shape *shape, const qdec_bf16 *q, int64_t q_stride,
                      const qdec_bf16 *k, int64_t k_stride, const qdec_bf16 *v, int64_t v_stride,
                      const qdec_bf16 *q_norm_w, const qdec_bf16 *k_norm_w,
                      const int32_t *positions, const int32_t *seq_lens,
                      const int32_t *block_table, const void *rope_table, const PoolArg &pool,
                      void *workspace, size_t workspace_bytes, qdec_bf16 *out,
                      int32_t *err_flag, void *stream) {
    qdec_status st = check_new_token_args(shape, q, q_stride, k, k_stride, v, v_stride, q_norm_w,
                                          k_norm_w, positions, seq_lens, block_table);
    if (st != QDEC_OK) return st;
    if ((st = check_pool(shape, pool)) != QDEC_OK) return st;
    if (rope_table && !aligned16(rope_table)) return QDEC_ERR_INVALID_ARG;
    if (!out || !aligned16(out)) return QDEC_ERR_INVALID_ARG;
    if ((st = check_workspace(shape, workspace, workspace_bytes)) != QDEC_OK) return st;
    Params p{};
    fill_common(p, shape, true, pool.fp8);
    bind_new_token(p, q, q_stride, k, k_stride, v, v_stride, q_norm_w, k_norm_w, positions,
                   seq_lens, block_table, rope_table);
    bind_pool(p, pool);
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.err = err_flag;
    bind_workspace(p, shape, workspace);
    CUtensorMap map;
    if ((st = encode_map(&map, shape, pool)) != QDEC_OK) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (step_in_two_launches(shape, pool.fp8)) {
        // q_rot in the workspace's last region; the append with the shape's
        // flags, the attention always as its programmatic dependent (it
        // reads q_rot and the appended slots only after the append is done)
        float *q_rot = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) +
                                                 workspace_layout(shape).qrot);
        Params pa = p;
        pa.q_rot_out = q_rot;
        // over an FP8 pool the new-token kernel starts only once the kernel
        // before it is done: launched early, its CTAs slowed the previous
        // layer's attention (64 ragged sequences: 220.8 against 131.0 us per
        // layer-step)
        if (pool.fp8) pa.pdl = 0;
        cudaError_t e = qdec::launch_append_rope(pa, pool.fp8, s);
        if (e != cudaSuccess) return cuda_status(e);
        Params pd = p;
        pd.q_rot_in = q_rot;
        pd.pdl = 1;
        return cuda_status(qdec::launch_attention(pd, map, qdec::kAttnDecode, pool.fp8, s));
    }
    return cuda_status(qdec::launch_attention(p, map, qdec::kAttnFused, pool.fp8, s));
}

qdec_status attn_decode_impl(const qdec_shape *shape, const float *q_rot, const PoolArg &pool,
                             const int32_t *block_table, const int32_t *seq_lens, void *workspace,
                             size_t workspace_bytes, qdec_bf16 *out, int32_t *err_flag,
                             void *stream) {
    qdec_status st = check_shape(shape);
    if (st != QDEC_OK) return st;
    if ((st = check_pool(shape, pool)) != QDEC_OK) return st;
    if (!q_rot || !block_table || !seq_lens || !out) return QDEC_ERR_INVALID_ARG;
    if (!aligned16(q_rot) || !aligned16(out)) return QDEC_ERR_INVALID_ARG;
    if ((st = check_workspace(shape, workspace, workspace_bytes)) != QDEC_OK) return st;
    Params p{};
    fill_common(p, shape, true, pool.fp8);
    p.q_rot_in = q_rot;
    p.seq_lens = seq_lens;
    p.block_table = block_table;
    bind_pool(p, pool);
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.err = err_flag;
    bind_workspace(p, shape, workspace);
    CUtensorMap map;
    if ((st = encode_map(&map, shape, pool)) != QDEC_OK) return st;
    return cuda_status(qdec::launch_attention(p, map, qdec::kAttnDecode, pool.fp8,
                                              static_cast<cudaStream_t>(stream)));
}

qdec_status prefill_append_impl(const qdec_shape *shape, int32_t num_tokens, const qdec_bf16 *q,
                                int64_t q_stride, const qdec_bf16 *k, int64_t k_stride,
                                const qdec_bf16 *v, int64_t v_stride, const qdec_bf16 *q_norm_w,
                                const qdec_bf16 *k_norm_w, const int32_t *positions,
                                const void *rope_table, const int32_t *qo_indptr,
                                const int32_t *seq_lens, const int32_t *block_table,
                                const PoolArg &pool, float *q_rot, int32_t *err_flag,
                                void *stream) {
    qdec_status st = check_new_token_args(shape, q, q_stride, k, k_stride, v, v_stride, q_norm_w,
                                          k_norm_w, positions, seq_lens, block_table);
    if (st != QDEC_OK) return st;
    if ((st = check_pool(shape, pool)) != QDEC_OK) return st;
    if (num_tokens < 0 || !qo_indptr || !q_rot || !aligned16(q_rot)) return QDEC_ERR_INVALID_ARG;
    if (rope_table && !aligned16(rope_table)) return QDEC_ERR_INVALID_ARG;
    Params p{};
    fill_common(p, shape, false, pool.fp8);
    // the table's rows are the chunk rows (r), not the sequences
    bind_new_token(p, q, q_stride, k, k_stride, v, v_stride, q_norm_w, k_norm_w, positions,
                   seq_lens, block_table, rope_table);
    bind_pool(p, pool);
    p.qo_indptr = qo_indptr;
    p.T = num_tokens;
    p.q_rot_out = q_rot;
    p.err = err_flag;
    return cuda_status(
        qdec::launch_prefill_append(p, pool.fp8, static_cast<cudaStream_t>(stream)));
}

// Scratch of the FP8 prefill's widened pool: every page slot of every
// sequence as 16-bit values (the bf16 pool's page size).
size_t prefill_fp8_scratch_bytes(const qdec_shape *s) {
    return static_cast<size_t>(s->batch) * s->max_blocks_per_seq * 2 * s->num_kv_heads *
           qdec::kPageSize * qdec::kHeadDim * 2;
}

qdec_status prefill_attn_impl(const qdec_shape *shape, int32_t num_tokens, const float *q_rot,
                              const int32_t *qo_indptr, const int32_t *seq_lens,
                              const int32_t *block_table, const PoolArg &pool, qdec_bf16 *out,
                              int32_t *err_flag, void *stream, void *workspace = nullptr,
                              size_t workspace_bytes = 0) {
    qdec_status st = check_shape(shape);
    if (st != QDEC_OK) return st;
    if ((st = check_pool(shape, pool)) != QDEC_OK) return st;
    if (num_tokens < 0 || !q_rot || !qo_indptr || !seq_lens || !block_table || !out)
        return QDEC_ERR_INVALID_ARG;
    if (!aligned16(q_rot) || !aligned16(out)) return QDEC_ERR_INVALID_ARG;
    Params p{};
    fill_common(p, shape, false, pool.fp8);
    p.q_rot_in = q_rot;
    p.qo_indptr = qo_indptr;
    p.T = num_tokens;
    p.seq_lens = seq_lens;
    p.block_table = block_table;
    bind_pool(p, pool);
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.err = err_flag;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    CUtensorMap map;
    if (pool.fp8 && workspace) {
        // dequantize the sequences' pages once, then attend over the scratch
        // as over a bf16 pool (the attention a programmatic dependent of the
        // dequantizing pass, whose output it reads only after its wait)
        if (!aligned16(workspace) || workspace_bytes < prefill_fp8_scratch_bytes(shape))
            return QDEC_ERR_WORKSPACE;
        qdec_shape ws_shape = *shape;
        ws_shape.num_pages = shape->batch * shape->max_blocks_per_seq;
        if ((st = encode_pool_region_map(&map, &ws_shape, workspace)) != QDEC_OK) return st;
        p.wide = static_cast<__nv_bfloat16 *>(workspace);
        Params pa = p;
        if (!(shape->launch_flags & QDEC_LAUNCH_PREFILL_PAGES_READY)) {
            cudaError_t e = qdec::launch_prefill_widen(p, cs);
            if (e != cudaSuccess) return cuda_status(e);
            pa.pdl = 1;
        }
        return cuda_status(qdec::launch_prefill_attention(pa, map, qdec::kPrefillPoolWide, cs));
    }
    if ((st = pool.fp8 ? encode_pool_plane_map_fp8(&map, shape, pool.data)
                       : encode_pool_region_map(&map, shape, pool.data)) != QDEC_OK)
        return st;
    return cuda_status(qdec::launch_prefill_attention(
        p, map, pool.fp8 ? qdec::kPrefillPoolFp8 : qdec::kPrefillPoolBf16, cs));
}

qdec_status qkv_impl(const qdec_shape *shape, int32_t hidden, const qdec_bf16 *x,
                     int64_t x_stride, const qdec_bf16 *w_packed, const qdec_bf16 *q_norm_w,
                     const qdec_bf16 *k_norm_w, const int32_t *positions, const int32_t *seq_lens,
                     const int32_t *block_table, const void *rope_table, const PoolArg &pool,
                     float *q_rot, int32_t *err_flag, void *stream) {
    qdec_status st = check_shape(shape);
    if (st != QDEC_OK) return st;
    if ((st = check_pool(shape, pool)) != QDEC_OK) return st;
    if (hidden < 64 || hidden % 64 != 0) return QDEC_ERR_UNSUPPORTED;
    if (!x || !w_packed || !q_norm_w || !k_norm_w || !positions || !seq_lens || !block_table ||
        !rope_table || !q_rot)
        return QDEC_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_packed) || !aligned16(q_norm_w) || !aligned16(k_norm_w) ||
        !aligned16(rope_table) || !aligned16(q_rot))
        return QDEC_ERR_INVALID_ARG;
    if (x_stride < hidden || x_stride % 8 != 0) return QDEC_ERR_INVALID_ARG;
    Params p{};
    fill_common(p, shape, false);
    p.hidden = hidden;
    qdec::qkv_geometry(shape->batch, hidden, p.qkv_rows, p.qkv_boxes, p.qkv_stages);
    p.w_q = reinterpret_cast<const __nv_bfloat16 *>(q_norm_w);
    p.w_k = reinterpret_cast<const __nv_bfloat16 *>(k_norm_w);
    p.positions = positions;
    p.seq_lens = seq_lens;
    p.block_table = block_table;
    p.rope = static_cast<const qdec::RopeEntry *>(rope_table);
    bind_pool(p, pool);
    p.q_rot_out = q_rot;
    p.err = err_flag;
    p.w_packed = reinterpret_cast<const __nv_bfloat16 *>(w_packed);
    CUtensorMap x_map;
    if ((st = encode_rows_map(&x_map, x, shape->batch, hidden, x_stride, p.qkv_rows)) != QDEC_OK)
        return st;
    return cuda_status(qdec::launch_qkv_append(p, x_map, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

size_t qdec_rope_table_bytes(const qdec_shape *shape) {
    if (check_shape(shape) != QDEC_OK) return 0;
    return static_cast<size_t>(shape->batch) * qdec::kRotPairs * sizeof(qdec::RopeEntry);
}

qdec_status qdec_rope_table(const qdec_shape *shape, const int32_t *positions, void *rope_table,
                            void *stream) {
    qdec_status st = check_shape(shape);
    if (st != QDEC_OK) return st;
    if (!positions || !rope_table || !aligned16(rope_table)) return QDEC_ERR_INVALID_ARG;
    Params p{};
    fill_common(p, shape, false);
    p.positions = positions;
    p.rope_out = static_cast<qdec::RopeEntry *>(rope_table);
    return cuda_status(qdec::launch_rope_table(p, static_cast<cudaStream_t>(stream)));
}

size_t qdec_prefill_rope_table_bytes(int32_t num_tokens) {
    return num_tokens > 0 ? static_cast<size_t>(num_tokens) * qdec::kRotPairs * sizeof(qdec::RopeEntry)
                          : 0;
}

qdec_status qdec_prefill_rope_table(const qdec_shape *shape, int32_t num_tokens,
                                    const int32_t *positions, void *rope_table, void *stream) {
    qdec_status st = check_shape(shape);
    if (st != QDEC_OK) return st;
    if (num_tokens < 0 || !positions || !rope_table || !aligned16(rope_table))
        return QDEC_ERR_INVALID_ARG;
    if (num_tokens == 0) return QDEC_OK;
    Params p{};
    fill_common(p, shape, false);
    p.B = num_tokens;  // one table row per chunk row
    p.positions = positions;
    p.rope_out = static_cast<qdec::RopeEntry *>(rope_table);
    return cuda_status(qdec::launch_rope_table(p, static_cast<cudaStream_t>(stream)));
}

int qdec_step_launches(const qdec_shape *shape, int fp8_pool) {
    if (check_shape(shape) != QDEC_OK) return 0;
    return step_in_two_launches(shape, fp8_pool != 0) ? 2 : 1;
}

size_t qdec_workspace_bytes(const qdec_shape *shape) {
    if (check_shape(shape) != QDEC_OK) return 0;
    return workspace_layout(shape).total;
}

qdec_status qdec_workspace_init(const qdec_shape *shape, void *workspace, size_t workspace_bytes,
                                void *stream) {
    qdec_status st = check_shape(shape);
    if (st != QDEC_OK) return st;
    if ((st = check_workspace(shape, workspace, workspace_bytes)) != QDEC_OK) return st;
    const size_t n = static_cast<size_t>(shape->batch) * shape->num_kv_heads * sizeof(int32_t);
    return cuda_status(cudaMemsetAsync(workspace, 0, n, static_cast<cudaStream_t>(stream)));
}

qdec_status qdec_append_rope(const qdec_shape *shape, const qdec_bf16 *q, int64_t q_stride,
                             const qdec_bf16 *k, int64_t k_stride, const qdec_bf16 *v,
                             int64_t v_stride, const qdec_bf16 *q_norm_w,
                             const qdec_bf16 *k_norm_w, const int32_t *positions,
                             const int32_t *seq_lens, const int32_t *block_table,
                             const void *rope_table, qdec_bf16 *kv_pool, float *q_rot,
                             int32_t *err_flag, void *stream) {
    return append_rope_impl(shape, q, q_stride, k, k_stride, v, v_stride, q_norm_w, k_norm_w,
                            positions, seq_lens, block_table, rope_table,
                            PoolArg{kv_pool, nullptr, false}, q_rot, err_flag, stream);
}

qdec_status qdec_append_rope_fp8(const qdec_shape *shape, const qdec_bf16 *q, int64_t q_stride,
                                 const qdec_bf16 *k, int64_t k_stride, const qdec_bf16 *v,
                                 int64_t v_stride, const qdec_bf16 *q_norm_w,
                                 const qdec_bf16 *k_norm_w, const int32_t *positions,
                                 const int32_t *seq_lens, const int32_t *block_table,
                                 const void *rope_table, uint8_t *kv_pool_fp8,
                                 const float *kv_scale, float *q_rot, int32_t *err_flag,
                                 void *stream) {
    return append_rope_impl(shape, q, q_stride, k, k_stride, v, v_stride, q_norm_w, k_norm_w,
                            positions, seq_lens, block_table, rope_table,
                            PoolArg{kv_pool_fp8, kv_scale, true}, q_rot, err_flag, stream);
}

qdec_status qdec_attn_split(const qdec_shape *shape, const float *q_rot, const qdec_bf16 *kv_pool,
                            const int32_t *block_table, const int32_t *seq_lens, void *workspace,
                            size_t workspace_bytes, qdec_bf16 *out, int32_t *err_flag,
                            void *stream) {
    return attn_split_impl(shape, q_rot, PoolArg{kv_pool, nullptr, false}, block_table, seq_lens,
                           workspace, workspace_bytes, out, err_flag, stream);
}

qdec_status qdec_attn_split_fp8(const qdec_shape *shape, const float *q_rot,
                                const uint8_t *kv_pool_fp8, const float *kv_scale,
                                const int32_t *block_table, const int32_t *seq_lens,
                                void *workspace, size_t workspace_bytes, qdec_bf16 *out,
                                int32_t *err_flag, void *stream) {
    return attn_split_impl(shape, q_rot, PoolArg{kv_pool_fp8, kv_scale, true}, block_table,
                           seq_lens, workspace, workspace_bytes, out, err_flag, stream);
}

qdec_status qdec_attn_decode(const qdec_shape *shape, const float *q_rot,
                             const qdec_bf16 *kv_pool, const int32_t *block_table,
                             const int32_t *seq_lens, void *workspace, size_t workspace_bytes,
                             qdec_bf16 *out, int32_t *err_flag, void *stream) {
    return attn_decode_impl(shape, q_rot, PoolArg{kv_pool, nullptr, false}, block_table,
                            seq_lens, workspace, workspace_bytes, out, err_flag, stream);
}

qdec_status qdec_attn_decode_fp8(const qdec_shape *shape, const float *q_rot,
                                 const uint8_t *kv_pool_fp8, const float *kv_scale,
                                 const int32_t *block_table, const int32_t *seq_lens,
                                 void *workspace, size_t workspace_bytes, qdec_bf16 *out,
                                 int32_t *err_flag, void *stream) {
    return attn_decode_impl(shape, q_rot, PoolArg{kv_pool_fp8, kv_scale, true}, block_table,
                            seq_lens, workspace, workspace_bytes, out, err_flag, stream);
}

qdec_status qdec_prefill_append_rope(const qdec_shape *shape, int32_t num_tokens,
                                     const qdec_bf16 *q, int64_t q_stride, const qdec_bf16 *k,
                                     int64_t k_stride, const qdec_bf16 *v, int64_t v_stride,
                                     const qdec_bf16 *q_norm_w, const qdec_bf16 *k_norm_w,
                                     const int32_t *positions, const void *rope_table,
                                     const int32_t *qo_indptr, const int32_t *seq_lens,
                                     const int32_t *block_table, qdec_bf16 *kv_pool, float *q_rot,
                                     int32_t *err_flag, void *stream) {
    return prefill_append_impl(shape, num_tokens, q, q_stride, k, k_stride, v, v_stride, q_norm_w,
                               k_norm_w, positions, rope_table, qo_indptr, seq_lens, block_table,
                               PoolArg{kv_pool, nullptr, false}, q_rot, err_flag, stream);
}

qdec_status qdec_prefill_append_rope_fp8(const qdec_shape *shape, int32_t num_tokens,
                                         const qdec_bf16 *q, int64_t q_stride,
                                         const qdec_bf16 *k, int64_t k_stride,
                                         const qdec_bf16 *v, int64_t v_stride,
                                         const qdec_bf16 *q_norm_w, const qdec_bf16 *k_norm_w,
                                         const int32_t *positions, const void *rope_table,
                                         const int32_t *qo_indptr, const int32_t *seq_lens,
                                         const int32_t *block_table, uint8_t *kv_pool_fp8,
                                         const float *kv_scale, float *q_rot, int32_t *err_flag,
                                         void *stream) {
    return prefill_append_impl(shape, num_tokens, q, q_stride, k, k_stride, v, v_stride, q_norm_w,
                               k_norm_w, positions, rope_table, qo_indptr, seq_lens, block_table,
                               PoolArg{kv_pool_fp8, kv_scale, true}, q_rot, err_flag, stream);
}

qdec_status qdec_prefill_attn(const qdec_shape *shape, int32_t num_tokens, const float *q_rot,
                              const int32_t *qo_indptr, const int32_t *seq_lens,
                              const int32_t *block_table, const qdec_bf16 *kv_pool,
                              qdec_bf16 *out, int32_t *err_flag, void *stream) {
    return prefill_attn_impl(shape, num_tokens, q_rot, qo_indptr, seq_lens, block_table,
                             PoolArg{kv_pool, nullptr, false}, out, err_flag, stream);
}

qdec_status qdec_prefill_attn_fp8(const qdec_shape *shape, int32_t num_tokens,
                                  const float *q_rot, const int32_t *qo_indptr,
                                  const int32_t *seq_lens, const int32_t *block_table,
                                  const uint8_t *kv_pool_fp8, const float *kv_scale,
                                  void *workspace, size_t workspace_bytes, qdec_bf16 *out,
                                  int32_t *err_flag, void *stream) {
    return prefill_attn_impl(shape, num_tokens, q_rot, qo_indptr, seq_lens, block_table,
                             PoolArg{kv_pool_fp8, kv_scale, true}, out, err_flag, stream,
                             workspace, workspace_bytes);
}

size_t qdec_prefill_fp8_workspace_bytes(const qdec_shape *shape) {
    if (check_shape(shape) != QDEC_OK) return 0;
    return prefill_fp8_scratch_bytes(shape);
}

qdec_status qdec_attn_merge(const qdec_shape *shape, const int32_t *seq_lens,
                            const void *workspace, size_t workspace_bytes, qdec_bf16 *out,
                            int32_t *err_flag, void *stream) {
    qdec_status st = check_shape(shape);
    if (st != QDEC_OK) return st;
    if (!seq_lens || !out || !aligned16(out)) return QDEC_ERR_INVALID_ARG;
    if ((st = check_workspace(shape, workspace, workspace_bytes)) != QDEC_OK) return st;
    Params p{};
    fill_common(p, shape, false);
    p.seq_lens = seq_lens;
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.err = err_flag;
    bind_workspace(p, shape, const_cast<void *>(workspace));
    return cuda_status(qdec::launch_merge(p, static_cast<cudaStream_t>(stream)));
}

qdec_status qdec_step(const qdec_shape *shape, const qdec_bf16 *q, int64_t q_stride,
                      const qdec_bf16 *k, int64_t k_stride, const qdec_bf16 *v, int64_t v_stride,
                      const qdec_bf16 *q_norm_w, const qdec_bf16 *k_norm_w,
                      const int32_t *positions, const int32_t *seq_lens,
                      const int32_t *block_table, const void *rope_table, qdec_bf16 *kv_pool,
                      void *workspace, size_t workspace_bytes, qdec_bf16 *out,
                      int32_t *err_flag, void *stream) {
    return step_impl(shape, q, q_stride, k, k_stride, v, v_stride, q_norm_w, k_norm_w, positions,
                     seq_lens, block_table, rope_table, PoolArg{kv_pool, nullptr, false},
                     workspace, workspace_bytes, out, err_flag, stream);
}

qdec_status qdec_step_fp8(const qdec_shape *shape, const qdec_bf16 *q, int64_t q_stride,
                          const qdec_bf16 *k, int64_t k_stride, const qdec_bf16 *v,
                          int64_t v_stride, const qdec_bf16 *q_norm_w, const qdec_bf16 *k_norm_w,
                          const int32_t *positions, const int32_t *seq_lens,
                          const int32_t *block_table, const void *rope_table,
                          uint8_t *kv_pool_fp8, const float *kv_scale, void *workspace,
                          size_t workspace_bytes, qdec_bf16 *out, int32_t *err_flag,
                          void *stream) {
    return step_impl(shape, q, q_stride, k, k_stride, v, v_stride, q_norm_w, k_norm_w, positions,
                     seq_lens, block_table, rope_table, PoolArg{kv_pool_fp8, kv_scale, true},
                     workspace, workspace_bytes, out, err_flag, stream);
}

qdec_status qdec_qkv_pack_weights(const qdec_shape *shape, int32_t hidden, const qdec_bf16 *w_qkv,
                                  qdec_bf16 *w_packed, void *stream) {
    qdec_status st = check_shape(shape);
    if (st != QDEC_OK) return st;
    if (hidden < 64 || hidden % 64 != 0) return QDEC_ERR_UNSUPPORTED;
    if (!w_qkv || !w_packed || !aligned16(w_qkv) || !aligned16(w_packed) || w_qkv == w_packed)
        return QDEC_ERR_INVALID_ARG;
    const int rows = (shape->num_q_heads + 2 * shape->num_kv_heads) * qdec::kHeadDim;
    return cuda_status(qdec::launch_qkv_pack(reinterpret_cast<const __nv_bfloat16 *>(w_qkv),
                                             reinterpret_cast<__nv_bfloat16 *>(w_packed), rows,
                                             hidden, static_cast<cudaStream_t>(stream)));
}

qdec_status qdec_qkv_append_rope(const qdec_shape *shape, int32_t hidden, const qdec_bf16 *x,
                                 int64_t x_stride, const qdec_bf16 *w_packed,
                                 const qdec_bf16 *q_norm_w, const qdec_bf16 *k_norm_w,
                                 const int32_t *positions, const int32_t *seq_lens,
                                 const int32_t *block_table, const void *rope_table,
                                 qdec_bf16 *kv_pool, float *q_rot, int32_t *err_flag,
                                 void *stream) {
    return qkv_impl(shape, hidden, x, x_stride, w_packed, q_norm_w, k_norm_w, positions, seq_lens,
                    block_table, rope_table, PoolArg{kv_pool, nullptr, false}, q_rot, err_flag,
                    stream);
}

qdec_status qdec_qkv_append_rope_fp8(const qdec_shape *shape, int32_t hidden, const qdec_bf16 *x,
                                     int64_t x_stride, const qdec_bf16 *w_packed,
                                     const qdec_bf16 *q_norm_w, const qdec_bf16 *k_norm_w,
                                     const int32_t *positions, const int32_t *seq_lens,
                                     const int32_t *block_table, const void *rope_table,
                                     uint8_t *kv_pool_fp8, const float *kv_scale, float *q_rot,
                                     int32_t *err_flag, void *stream) {
    return qkv_impl(shape, hidden, x, x_stride, w_packed, q_norm_w, k_norm_w, positions, seq_lens,
                    block_table, rope_table, PoolArg{kv_pool_fp8, kv_scale, true}, q_rot,
                    err_flag, stream);
}

qdec_status qdec_check_error(int32_t *err_flag, void *stream, int32_t *flags_out) {
    if (!err_flag) return QDEC_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t flags = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return QDEC_ERR_CUDA;
    if (cudaMemcpyAsync(&flags, err_flag, sizeof flags, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return QDEC_ERR_CUDA;
    if (cudaMemsetAsync(err_flag, 0, sizeof flags, s) != cudaSuccess) return QDEC_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return QDEC_ERR_CUDA;
    if (flags_out) *flags_out = flags;
    if (flags & QDEC_FLAG_TIMEOUT) return QDEC_ERR_TIMEOUT;
    if (flags & (QDEC_FLAG_BAD_PAGE | QDEC_FLAG_BAD_SEQLEN | QDEC_FLAG_BAD_INDEX))
        return QDEC_ERR_DEVICE_BOUNDS;
    return QDEC_OK;
}

const char *qdec_status_string(qdec_status status) {
    switch (status) {
        case QDEC_OK: return "ok";
        case QDEC_ERR_INVALID_ARG: return "invalid argument";
        case QDEC_ERR_UNSUPPORTED: return "unsupported shape";
        case QDEC_ERR_WORKSPACE: return "workspace missing or too small";
        case QDEC_ERR_CUDA: return "CUDA call failed";
        case QDEC_ERR_DEVICE_BOUNDS: return "device saw a block-table entry or seq_len out of range";
        case QDEC_ERR_TIMEOUT: return "a bounded device wait gave up";
    }
    return "unknown status";
}

int32_t qdec_version(void) { return kVersion; }

}  // extern "C"
