// qdec_internal.h -- what the host API (qdec_api.cu) and the kernels
// (qdec_kernels.cu) of libqdec share.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qdec {

// Shapes the kernels are written for.
constexpr int kHeadDim = 128;       // D
constexpr int kPageSize = 16;       // P (tokens per page)
constexpr int kGroup = 4;           // query heads per KV head
constexpr int kMaxBatch = 1024;     // sequence prefix sums live in shared memory
constexpr int kRotPairs = kHeadDim / 2;

// Attention kernel geometry.
constexpr int kConsumerWarps = 4;                          // tile math
constexpr int kThreads = (kConsumerWarps + 1) * 32;        // + one TMA producer warp
constexpr int kMaxStages = 24;                             // ring of page tiles (runtime depth)
constexpr int kTileHalfBytes = kPageSize * 64 * 2;         // 16 rows x 64 dims bf16 = 2 KiB
constexpr int kPlaneBytes = 2 * kTileHalfBytes;            // one (page, plane, head) = 4 KiB
constexpr int kTileBytes = 2 * kPlaneBytes;                // K + V = 8 KiB
// FP8 (E4M3) pool: one byte per element, so a (page, plane, head) is 16
// rows of 128 bytes and a page tile K + V is 4 KiB.  Each ring slot also
// holds the tile's K and V scale (two floats the producer stores with the
// page lookup, so a tile is one copy).
constexpr int kFp8PlaneBytes = kPageSize * kHeadDim;       // 2 KiB
constexpr int kFp8TileBytes = 2 * kFp8PlaneBytes;          // 4 KiB
constexpr int kFp8SlotExtra = 16;                          // per ring slot
// Cluster layout: the largest cluster whose peers' pieces get their own
// receive buffer; larger clusters receive in rank 0's drained ring.
constexpr int kMaxDirectRecv = 6;
constexpr int kCtasPerSm = 2;
// The FP8 flat layout (long tile ranges, half-size tiles) runs three CTAs per
// SM: more tiles in flight per SM at 128 registers a thread.
constexpr int kCtasPerSmFp8Flat = 3;
constexpr int ctas_per_sm(bool cluster, bool fp8) {
    return (!cluster && fp8) ? kCtasPerSmFp8Flat : kCtasPerSm;
}
constexpr int kMaxCluster = 8;                             // portable cluster size

// Budget of a bounded wait (SM cycles): ~2 s at the 2.07 GHz maximum clock;
// ~10 ms under the withheld-tile test hook.
constexpr long long kWaitTimeoutCycles = 4000000000ll;
constexpr long long kTestWaitCycles = 20000000ll;

// One RoPE angle of one sequence: cos and sin as unevaluated float pairs
// (hi + lo), i.e. about 48 significant bits.
struct RopeEntry {
    float c_hi, c_lo, s_hi, s_lo;
};

// Everything a launch needs, passed by value (__grid_constant__).
struct Params {
    int B, Hq, Hkv, num_pages, max_blocks;
    float eps;
    float qscale;            // sm_scale * log2(e): scores come out in log2 units
    const __nv_bfloat16 *q, *k, *v;
    int64_t q_stride, k_stride, v_stride;   // elements between sequences
    const __nv_bfloat16 *w_q, *w_k;
    const int32_t *positions, *seq_lens, *block_table;
    const RopeEntry *rope;   // [B][D/2] per-step table, or null: angles computed in-kernel
    RopeEntry *rope_out;     // rope-table kernel output
    __nv_bfloat16 *pool;
    uint8_t *pool8;          // E4M3 pool (FP8 entry points), same layout as pool
    const float *kv_scale;   // FP8: [num_pages][2][Hkv] scale of each (page, plane, head)
    const float *q_rot_in;   // split kernel (unfused): normed + rotated q rows
    float *q_rot_out;        // append kernel: normed + rotated q rows
    float *ws_o;             // [pieces][G][D] partial outputs (normalised)
    float *ws_lse;           // [pieces][G] partial log2-sum-exp
    int32_t *ws_cnt;         // [B * Hkv] arrival counters (fused merge)
    __nv_bfloat16 *out;      // [B][Hq][D]
    int32_t *err;            // device error flag (may be null)
    int grid;                // attention grid size the piece layout is built for
    int stages;              // ring depth: a multiple of kConsumerWarps, <= kMaxStages
    int pdl;                 // launched as a programmatic dependent of the previous kernel
    int cluster;             // 0: flat tile partition; C > 0: segment chunks on C-CTA clusters
    int chunks;              // cluster mode: chunks (clusters) per segment
    long long ws_pieces;     // partial slots the workspace holds (device bounds checks)
    long long wait_cycles;   // budget of every bounded wait, in SM cycles
    int withhold_first;      // test hook: CTA-local tile 0 is never copied (see qdec.h)
    int hidden;              // QKV projection: hidden size (a multiple of 64)
    int qkv_rows;            // QKV projection: hidden-state rows per stage (16, 32, 48 or 64)
    int qkv_stages;          // QKV projection: ring depth
    int qkv_boxes;           // QKV projection: 64-element blocks along hidden per stage
    const __nv_bfloat16 *w_packed;  // QKV projection: the weight in the packed order
    const int32_t *qo_indptr;  // prefill: [B+1] packed chunk rows of each sequence
    __nv_bfloat16 *wide;       // prefill over FP8: the dequantised bf16 scratch pool
    int T;                     // prefill: rows the caller's buffers hold (qo_indptr[B] <= T)
    double inv_freq[kRotPairs];  // rope_theta^(-2i/D), i < D/2
};

// Dynamic shared memory of the attention kernel for batch B, `stages` ring
// slots, the given layout (cluster = 0: flat; C > 0: C-CTA clusters) and
// pool element type (fp8: E4M3, else bf16).
size_t attention_smem_bytes(int B, int stages, int cluster, bool fp8);

// Smallest ring depth the cluster layout of C CTAs needs: with C above
// kMaxDirectRecv rank 0 receives its peers' pieces in its drained ring.
int min_stages(int cluster, bool fp8);

// Clusters of `cluster` CTAs (each with `smem` bytes of dynamic shared
// memory) that can be resident at once on the current device (0 if unknown).
int max_active_clusters(int cluster, size_t smem, bool fp8);

cudaError_t launch_rope_table(const Params &p, cudaStream_t s);
cudaError_t launch_append_rope(const Params &p, bool fp8, cudaStream_t s);
// What one attention launch does around step 4:
//   kAttnSplit  q_rot in; pieces of split segments left in the workspace for
//               the merge kernel (flat layout only)
//   kAttnFused  steps 1-4: new-token rows normed, rotated and appended in the
//               kernel; the last piece of a split segment merges it
//   kAttnDecode q_rot in (the slot already appended); the last piece merges
enum AttnMode : int { kAttnSplit = 0, kAttnFused = 1, kAttnDecode = 2 };

cudaError_t launch_attention(const Params &p, const CUtensorMap &kv_map, AttnMode mode, bool fp8,
                             cudaStream_t s);
cudaError_t launch_merge(const Params &p, cudaStream_t s);

// Chunked prefill (qdec_prefill.cu): steps 1-3 for every chunk row, and the
// causal paged attention of the chunk on the 5th-generation tensor core.
// Pool kinds of the attention: a bf16 pool (kv_map: one (page, plane, half
// of D) region per box), an FP8 pool converted as it arrives (one (page,
// plane) per box), or an FP8 pool dequantised beforehand by
// launch_prefill_widen into the bf16 scratch p.wide (the bf16 region map
// over that scratch).
constexpr int kPrefillPoolBf16 = 0, kPrefillPoolFp8 = 1, kPrefillPoolWide = 2;
cudaError_t launch_prefill_append(const Params &p, bool fp8, cudaStream_t s);
cudaError_t launch_prefill_attention(const Params &p, const CUtensorMap &kv_map, int pool,
                                     cudaStream_t s);
cudaError_t launch_prefill_widen(const Params &p, cudaStream_t s);

// The merged QKV projection fused with steps 1-3 (qdec_qkv.cu): the weight
// comes packed (qdec_qkv_pack_weights), x_map views x [B][hidden] with boxes
// of 64 elements x p.qkv_rows rows, 128-byte swizzled.
cudaError_t launch_qkv_append(const Params &p, const CUtensorMap &x_map, cudaStream_t s);
// Packs W [rows][hidden] (rows = (Hq + 2 Hkv) * 128) into the order the
// projection streams it.
cudaError_t launch_qkv_pack(const __nv_bfloat16 *w, __nv_bfloat16 *w_packed, int rows,
                            int hidden, cudaStream_t s);
// Stage geometry of the projection for batch B and hidden size: the hidden-
// state rows (B rounded up to 16, at most 64), 64-element boxes along hidden
// per stage (4 for up to 16 rows, 2 up to 32, else 1, so that each weight
// row is read in runs of up to 512 bytes), and as many stages as about
// 96 KiB hold.
void qkv_geometry(int B, int hidden, int &rows, int &boxes, int &stages);

}  // namespace qdec
