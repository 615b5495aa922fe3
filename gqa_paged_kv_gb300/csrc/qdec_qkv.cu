// qdec_qkv.cu -- the merged QKV projection fused with steps 1-3 (RMSNorm,
// NeoX RoPE, paged append), on sm_103a.
//
// The projection is one matrix W [(Hq + 2 Hkv) * D][hidden] (article "扔掉
// vLLM！从零构建 Qwen3-8B 推理引擎" (news.rkmt.cn), section 4.4.3: the q, k and v
// projections merged into one; rows: the query heads, then the key heads,
// then the value heads), applied to every sequence's hidden state x [B][hidden].
// Its epilogue keeps each head's 128 outputs unrounded (fp32) into the norm,
// the rotation and the append: query heads go to q_rot (fp32, unscaled, the
// input of qdec_attn_split), key heads are rounded once to bf16 after the
// rotation and value heads once as they are, into slot seq_lens[b] - 1.
//
// Layout: a cluster of 4 CTAs per output head; CTA r of the cluster computes
// head dims 16r .. 16r+15 and 64+16r .. 64+16r+15 (so every rotate-half pair
// stays inside one CTA) for 64 batch rows, over the whole hidden dimension.
// The weight is packed once (qdec_qkv_pack_weights) into the order the
// projection reads it: for every (head, cluster rank) the 32 rows it owns, in
// blocks of 64 hidden elements, each block 4 KiB contiguous with its
// 128-byte rows already swizzled for conflict-free matrix loads; a CTA's
// whole share is one contiguous run.  One producer warp streams stages of
// 1, 2 or 4 such blocks (one bulk copy; more for smaller batches) and the
// matching boxes of x (the batch rounded up to 16 rows, at most 64; rows past
// B read as zero, TMA) into a ring of about 96 KiB; four consumer warps each
// own 16 batch rows and run bf16 mma.sync (fp32 accumulate).  The
// RMSNorm needs the sum of squares over all 128 dims: each CTA leaves its
// share per row in shared memory and reads the peers' shares over
// distributed shared memory between two cluster-barrier phases.
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
constexpr int kQkvRows = 4 * 16;                            // batch rows per CTA (4 warps x m16)
constexpr int kQkvChunk = 64;                               // hidden elements per stage
constexpr int kQkvMaxStages = 16;
constexpr int kQkvWBox = 16 * kQkvChunk * 2;                // one 16-row W box, 2 KiB
constexpr int kQkvRingBytes = 96 * 1024;
// after the ring: barriers full[16], empty[16], the abort flag, row sums
constexpr int kQkvTailBytes = 2 * kQkvMaxStages * 8 + 16 + kQkvRows * 4;
// a stage: [packed W blocks, 4 KiB each: rows 16r.. then rows 64+16r..][x
// boxes], each piece starting on a 1024-byte boundary (rows % 16 == 0)
__host__ __device__ constexpr int qkv_stage_bytes(int rows, int boxes) {
    return boxes * (2 * kQkvWBox + rows * kQkvChunk * 2);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
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

// Address of row r, 16-byte chunk c of a 128-byte-swizzled box at `base`.
__device__ __forceinline__ uint32_t swz(uint32_t base, int r, int c) {
    return base + r * 128 + ((c ^ (r & 7)) << 4);
}

__global__ void __launch_bounds__(kThreads, 2)
    qkv_append_kernel(const __grid_constant__ CUtensorMap x_map, const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int head = blockIdx.x / kQkvCluster, rank = blockIdx.x % kQkvCluster;
    const int row0 = blockIdx.y * kQkvRows;
    const int NB = p.qkv_boxes;
    const int nchunks = p.hidden / (kQkvChunk * NB);
    const int NS = p.qkv_stages;
    const int stage_bytes = qkv_stage_bytes(p.qkv_rows, NB);
    uint8_t *tail = sm + NS * stage_bytes;
    const uint32_t full0 = smem_u32(tail);
    const uint32_t empty0 = full0 + kQkvMaxStages * 8;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tail + 2 * kQkvMaxStages * 8);
    float *ss = reinterpret_cast<float *>(tail + 2 * kQkvMaxStages * 8 + 16);
    if (NS < 1 || NS > kQkvMaxStages || p.qkv_rows < 16 || p.qkv_rows > kQkvRows ||
        p.qkv_rows % 16 != 0 || NB < 1 || NB > 4 || p.hidden % (kQkvChunk * NB) != 0) {
        if (tid == 0) flag_error(p.err, QDEC_FLAG_BAD_INDEX);
        return;  // uniform over the cluster: every CTA sees the same parameters
    }

    if (p.pdl && tid == 0) launch_dependents();  // the next kernel waits for our completion
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kConsumerWarps);  // every warp takes every chunk
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------ TMA producer --
        if (lane == 0) {
            // this CTA's packed blocks: (head * 4 + rank) * (hidden / 64) onwards
            const __nv_bfloat16 *wsrc =
                p.w_packed + static_cast<int64_t>(head * kQkvCluster + rank) * p.hidden * 32;
            // With an overlapped launch the weight (which no kernel writes) of
            // the first stages goes out before the dependency wait; the hidden
            // states only after it.
            const int pre = p.pdl ? min(NS, nchunks) : 0;
            for (int c = 0; c < pre; ++c) {
                const uint32_t full = full0 + 8 * c;
                mbar_arrive_expect_tx(full, stage_bytes);
                bulk_load(smem_u32(sm + c * stage_bytes),
                          wsrc + static_cast<int64_t>(c) * NB * 32 * kQkvChunk, NB * 2 * kQkvWBox,
                          full);
            }
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
                    bulk_load(dst, wsrc + static_cast<int64_t>(c) * NB * 32 * kQkvChunk,
                              NB * 2 * kQkvWBox, full);
                }
                for (int j = 0; j < NB; ++j)
                    tma_load_2d(dst + 2 * NB * kQkvWBox + j * p.qkv_rows * kQkvChunk * 2, &x_map,
                                (c * NB + j) * kQkvChunk, row0, full);
            }
        }
        __syncwarp();
        cluster_sync_all();  // row sums published
        cluster_sync_all();  // peers done reading them
    } else {
        // ------------------------------------------- consumer warps --
        // warp w: batch rows row0 + 16w .. +15; n-tiles 0, 1: dims 16r + 0..15,
        // n-tiles 2, 3: dims 64 + 16r + 0..15
        const int g = lane >> 2, t = lane & 3;
        const bool live = row0 + 16 * warp < p.B;
        float acc[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
        const int mi = lane >> 3, r8 = lane & 7;
        const int arow = 16 * warp + (mi & 1) * 8 + r8;  // x row this lane addresses
        const int brow = (mi >> 1) * 8 + r8;             // W row within a 16-row box
        if (p.pdl) grid_dependency_wait();  // the tables, q_rot and the pool of earlier kernels

        // the epilogue's lookups for rows g and g + 8, made while the weight
        // streams: the append slot (-1: skip the row) and the norm weights
        const int Hq = p.Hq, Hkv = p.Hkv;
        const int kind = head < Hq ? 0 : (head < Hq + Hkv ? 1 : 2);  // q, k or v head
        const int kvh = kind == 1 ? head - Hq : head - Hq - Hkv;
        int64_t slot[2] = {-1, -1};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int b = row0 + 16 * warp + g + 8 * half;
            if (!live || b >= p.B) continue;
            const int L = p.seq_lens[b];
            if (L < 1 || L > p.max_blocks * kPageSize) {
                if (t == 0 && head == 0 && rank == 0) flag_error(p.err, QDEC_FLAG_BAD_SEQLEN);
                continue;
            }
            if (kind == 0) {
                slot[half] = 0;
                continue;
            }
            const int page =
                p.block_table[static_cast<int64_t>(b) * p.max_blocks + (L - 1) / kPageSize];
            if (page < 0 || page >= p.num_pages) {
                if (t == 0 && rank == 0 && kind == 1 && kvh == 0)
                    flag_error(p.err, QDEC_FLAG_BAD_PAGE);
                continue;
            }
            slot[half] =
                ((static_cast<int64_t>(page) * 2 * Hkv + kvh) * kPageSize + (L - 1) % kPageSize) *
                kHeadDim;
        }
        uint32_t wn2[2][2];  // norm weight pairs (d, d+1), (d+64, d+65) of n-tiles 0, 1
        {
            const __nv_bfloat16 *wn = kind == 0 ? p.w_q : p.w_k;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int d = 16 * rank + 8 * nt + 2 * t;
                wn2[nt][0] = kind == 2 ? 0u : *reinterpret_cast<const uint32_t *>(wn + d);
                wn2[nt][1] = kind == 2 ? 0u : *reinterpret_cast<const uint32_t *>(wn + d + 64);
            }
        }
        for (int c = 0; c < nchunks; ++c) {
            const int s = c % NS;
            const bool ok = mbar_wait_bounded(full0 + 8 * s, (c / NS) & 1, abort_flag,
                                              p.wait_cycles);
            if (!ok) {
                if (lane == 0) {
                    *abort_flag = 1;
                    flag_error(p.err, QDEC_FLAG_TIMEOUT);
                }
                break;
            }
            for (int j = 0; j < NB && live; ++j) {
                const uint32_t sb = smem_u32(sm + s * stage_bytes);
                // packed block j: rows 0..15 dims 16r.., rows 16..31 dims 64 + 16r..
                const uint32_t wa = sb + j * 2 * kQkvWBox, wbb = wa + kQkvWBox;
                const uint32_t xb = sb + 2 * NB * kQkvWBox + j * p.qkv_rows * kQkvChunk * 2;
#pragma unroll
                for (int kk = 0; kk < kQkvChunk / 16; ++kk) {
                    uint32_t a[4], b01[4], b23[4];
                    ldmatrix_x4(a, swz(xb, arow, 2 * kk + (mi >> 1)));
                    ldmatrix_x4(b01, swz(wa, brow, 2 * kk + (mi & 1)));
                    ldmatrix_x4(b23, swz(wbb, brow, 2 * kk + (mi & 1)));
                    mma_bf16(acc[0], a, b01[0], b01[1]);
                    mma_bf16(acc[1], a, b01[2], b01[3]);
                    mma_bf16(acc[2], a, b23[0], b23[1]);
                    mma_bf16(acc[3], a, b23[2], b23[3]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * s);
        }
        // this CTA's share of each row's sum of squares (rows g and g + 8)
        float sA = 0.f, sB = 0.f;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            sA += acc[nt][0] * acc[nt][0] + acc[nt][1] * acc[nt][1];
            sB += acc[nt][2] * acc[nt][2] + acc[nt][3] * acc[nt][3];
        }
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {
            sA += __shfl_xor_sync(kFull, sA, o);
            sB += __shfl_xor_sync(kFull, sB, o);
        }
        if (t == 0) {
            ss[16 * warp + g] = sA;
            ss[16 * warp + g + 8] = sB;
        }
        cluster_sync_all();  // every CTA's shares are in place
        float totA = 0.f, totB = 0.f;
#pragma unroll
        for (int q = 0; q < kQkvCluster; ++q) {
            const float *peer = cluster_peer(ss, q);
            totA += peer[16 * warp + g];
            totB += peer[16 * warp + g + 8];
        }
        cluster_sync_all();  // nobody leaves while a peer may still read

#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int b = row0 + 16 * warp + g + 8 * half;
            if (*abort_flag || slot[half] < 0) continue;
            const float tot = half ? totB : totA;
            const int64_t kslot = slot[half];
            const float rn = rsqrtf(tot * (1.0f / kHeadDim) + p.eps);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int d = 16 * rank + 8 * nt + 2 * t;  // dims d, d+1 and d+64, d+65
                const float x1a = acc[nt][2 * half], x1b = acc[nt][2 * half + 1];
                const float x2a = acc[nt + 2][2 * half], x2b = acc[nt + 2][2 * half + 1];
                if (kind == 2) {
                    __nv_bfloat16 *vdst = p.pool + kslot + static_cast<int64_t>(Hkv) * kPageSize *
                                                               kHeadDim;
                    *reinterpret_cast<uint32_t *>(vdst + d) = pack2_bf16(x1a, x1b);
                    *reinterpret_cast<uint32_t *>(vdst + d + 64) = pack2_bf16(x2a, x2b);
                    continue;
                }
                const float2 w1 = bf16x2_to_float2(wn2[nt][0]), w2 = bf16x2_to_float2(wn2[nt][1]);
                const float n1a = x1a * rn * w1.x, n1b = x1b * rn * w1.y;
                const float n2a = x2a * rn * w2.x, n2b = x2b * rn * w2.y;
                const RopeEntry ea = p.rope[static_cast<int64_t>(b) * kRotPairs + d];
                const RopeEntry eb = p.rope[static_cast<int64_t>(b) * kRotPairs + d + 1];
                const float y1a = n1a * ea.c_hi - n2a * ea.s_hi, y2a = n2a * ea.c_hi + n1a * ea.s_hi;
                const float y1b = n1b * eb.c_hi - n2b * eb.s_hi, y2b = n2b * eb.c_hi + n1b * eb.s_hi;
                if (kind == 0) {
                    float *dst = p.q_rot_out + (static_cast<int64_t>(b) * Hq + head) * kHeadDim;
                    *reinterpret_cast<float2 *>(dst + d) = make_float2(y1a, y1b);
                    *reinterpret_cast<float2 *>(dst + d + 64) = make_float2(y2a, y2b);
                } else {
                    __nv_bfloat16 *kdst = p.pool + kslot;
                    *reinterpret_cast<uint32_t *>(kdst + d) = pack2_bf16(y1a, y1b);
                    *reinterpret_cast<uint32_t *>(kdst + d + 64) = pack2_bf16(y2a, y2b);
                }
            }
        }
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

// Packing: destination 16-byte unit u lies in block u / 256 (4 KiB), row
// (u / 8) % 32 of the block, position u % 8, which holds source chunk
// (u % 8) ^ (row % 8) of that row (the 128-byte swizzle).  Block index =
// (head * 4 + rank) * (hidden / 64) + k-block; block rows 0-15 are weight rows
// head * 128 + 16 rank + i, rows 16-31 are head * 128 + 64 + 16 rank + i.
__global__ void qkv_pack_kernel(const __nv_bfloat16 *w, __nv_bfloat16 *wp, int rows, int hidden) {
    const int64_t total = static_cast<int64_t>(rows) * hidden / 8;
    const int nk = hidden / kQkvChunk;
    for (int64_t u = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; u < total;
         u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t block = u / 256;
        const int rho = static_cast<int>((u / 8) % 32), pos = static_cast<int>(u % 8);
        const int q = pos ^ (rho & 7);
        const int kb = static_cast<int>(block % nk);
        const int64_t hr = block / nk;  // head * 4 + rank
        const int head = static_cast<int>(hr / kQkvCluster), rank = static_cast<int>(hr % kQkvCluster);
        const int row = head * kHeadDim + (rho < 16 ? 16 * rank + rho : 64 + 16 * rank + rho - 16);
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
    rows = B >= kQkvRows ? kQkvRows : (B + 15) / 16 * 16;
    boxes = rows <= 16 ? 4 : (rows <= 32 ? 2 : 1);
    while (boxes > 1 && hidden % (kQkvChunk * boxes) != 0) boxes /= 2;
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
            const cudaError_t e = cudaFuncSetAttribute(
                qkv_append_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kQkvSmemMax);
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
    return cudaLaunchKernelEx(&cfg, qkv_append_kernel, x_map, p);
}

}  // namespace qdec
