/*
 * qdec.h -- C ABI of libqdec: the attention block of one GQA decode
 * layer-step over a paged bf16 (or FP8 E4M3) KV cache, on one NVIDIA GB300
 * (sm_103a).
 *
 * What the block computes (for every sequence b of the batch, with
 * L_b = seq_lens[b] tokens including the new one, G = 4 query heads per KV
 * head, D = 128, page size P = 16):
 *
 *   1. QK RMSNorm -- every new-token head row x (Hq query rows, Hkv key rows)
 *      becomes x * rsqrt(mean(x^2) + eps) * w, with one weight vector w_q for
 *      the query rows and one w_k for the key rows.  (Blog "GPU 算子与执行优化：从 26 到 100 token/s 的推理引擎破茧之路" (yuzheng310.github.io),
 *      part 6 (第六部分): fused RMSNorm after the Q/K projection.)
 *   2. NeoX RoPE -- rotate-half at position positions[b]: for i < D/2 the pair
 *      (i, i + D/2) turns by pos * rope_theta^(-2i/D).  (Same blog, part 6,
 *      fused NeoX RoPE with interleave=False.)
 *   3. Paged append -- slot t = L_b - 1 lives in page block_table[b][t / P],
 *      row t % P; it receives bf16(k_rot) (round-to-nearest-even) and v (bits
 *      copied).  (Essay "推理引擎里面发生了什么" (locsic.com),
 *      section "PagedAttention：vLLM 的解法": 16-token blocks reached through
 *      a per-request block table.)
 *   4. Split-KV GQA decode attention -- query head h reads KV head h / G;
 *      out = softmax(q_rot K^T * sm_scale) V over the L_b tokens, the new one
 *      included.  The KV sequence of each (b, KV head) is cut into pieces
 *      processed by different CTAs, each piece yields a local softmax, and
 *      the pieces are reduced with the exact log-sum-exp merge.  (Blog part 8,
 *      split-KV; article "扔掉 vLLM！从零构建 Qwen3-8B 推理引擎" (news.rkmt.cn),
 *      section 4.4.2, grouped decode.)
 *
 * Pool layout (one pool per layer; the blog's part-4 shape with K and V in
 * one tensor):   kv_pool[num_pages][2][Hkv][P][D] bf16, plane 0 = K, 1 = V.
 * Every (page, plane, head) tile is 4 KiB contiguous.
 *
 * Conventions shared by every call:
 *   - bf16 tensors are passed as qdec_bf16 (raw IEEE bfloat16 bits).
 *   - Every pointer except `shape` and `err_flag`-less calls is a DEVICE
 *     pointer on the current CUDA device; the caller allocates and owns all
 *     of them.  The library never allocates or frees device memory and holds
 *     no per-call state; it caches only per-device attributes.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call is asynchronous on that stream; only
 *     qdec_check_error synchronises.
 *   - Host-detectable errors return a status and launch nothing.  A failed
 *     launch returns QDEC_ERR_CUDA.  Device-detected faults (a block-table
 *     entry outside the pool, a seq_len outside [1, max_blocks_per_seq * P],
 *     a bounded wait that ran out, an internal index that fails its bounds
 *     check) never trap: the kernel skips the affected
 *     work, ORs a QDEC_FLAG_* bit into *err_flag (when err_flag is not NULL)
 *     and the outputs of the affected sequences are unspecified.
 *   - Alignment: q, k, v, kv_pool, out, q_rot and workspace must be 16-byte
 *     aligned; q_stride, k_stride and v_stride (elements between consecutive
 *     sequences) must be multiples of 8.  Within a sequence the heads of q
 *     (and of k, of v) are contiguous rows of D elements, so q/k/v may be
 *     strided views of one fused qkv buffer [B][Hq + 2 Hkv][D].
 *   - The 36 layers of a model share block_table, seq_lens and positions;
 *     each layer brings its own kv_pool and norm weights.
 */
#ifndef QDEC_H
#define QDEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t qdec_bf16;

typedef enum {
    QDEC_OK = 0,
    QDEC_ERR_INVALID_ARG = 1,    /* null pointer, bad size, misalignment       */
    QDEC_ERR_UNSUPPORTED = 2,    /* shape outside what the kernels implement    */
    QDEC_ERR_WORKSPACE = 3,      /* workspace missing or smaller than required  */
    QDEC_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed           */
    QDEC_ERR_DEVICE_BOUNDS = 5,  /* qdec_check_error: device saw bad page/len   */
    QDEC_ERR_TIMEOUT = 6         /* qdec_check_error: a bounded wait gave up    */
} qdec_status;

/* qdec_shape.launch_flags */
#define QDEC_LAUNCH_OVERLAP_PREVIOUS 1
/* qdec_prefill_attn_fp8 with a workspace: the workspace already holds the
 * dequantized pages of this call's sequences, written by an earlier
 * qdec_prefill_attn_fp8 call with the same shape, qo_indptr, seq_lens,
 * block_table and workspace, and neither the pool's pages of those
 * sequences nor kv_scale have changed since (e.g. attending several query
 * sets over one context): the dequantizing pass is skipped and the call is
 * one launch.  Other calls ignore it. */
#define QDEC_LAUNCH_PREFILL_PAGES_READY 2
/* Test hook for the failure path, not for production use: in every CTA of
 * the paged attention kernels (qdec_step, qdec_attn_split, qdec_attn_decode,
 * qdec_prefill_attn and their FP8 forms) the first page tile is never
 * copied, and in every CTA of the QKV projection the first stage of weight
 * and hidden states, so the wait for it runs out (after ~10 ms instead of
 * ~2 s), the kernel stops its copies, lets those in flight land and returns;
 * qdec_check_error then reports QDEC_ERR_TIMEOUT.  Outputs of such a call
 * are undefined; the device stays usable.  The calls whose kernels wait on
 * nothing (rope table, append, merge, weight packing) ignore it.  No
 * counterpart in the pages. */
#define QDEC_LAUNCH_TEST_WITHHOLD_TILE (1 << 30)
/* qdec_step may be launched as a programmatic dependent of the kernel before
 * it on the stream: it starts streaming cached KV pages (reading seq_lens,
 * block_table and kv_pool) while that kernel is still finishing, and waits
 * for it before reading q, k, v, positions, the norm weights, the rope table
 * or writing anything.  Set it only when the immediately preceding kernel
 * does not write seq_lens, block_table or kv_pool pages other than the
 * append slots of this step (e.g. the previous layer's qdec_step).
 * (Where qdec_step runs as two launches, see there, the first reads seq_lens
 * before that wait, the second is always a programmatic dependent of the
 * first.)  qdec_append_rope with the flag reads seq_lens before the wait and
 * everything else after it.
 * qdec_attn_decode with the flag waits for the previous kernel before it
 * reads anything but its launch parameters.  qdec_qkv_append_rope with the
 * flag streams the first stages of its (packed) weight before that wait and
 * waits before it reads x, the tables or the norm weights or writes anything,
 * so the weight must not be written by the kernel before it. */

/* Bits a kernel ORs into *err_flag. */
#define QDEC_FLAG_BAD_PAGE   1   /* block-table entry outside [0, num_pages)   */
#define QDEC_FLAG_BAD_SEQLEN 2   /* seq_len outside [1, max_blocks_per_seq*P]  */
#define QDEC_FLAG_TIMEOUT    4   /* an mbarrier wait exceeded its time limit   */
#define QDEC_FLAG_BAD_INDEX  8   /* an internal index failed its bounds check  */

/* Problem description.  Supported: head_dim 128, page_size 16,
 * num_q_heads == 4 * num_kv_heads, 1 <= batch <= 1024. */
typedef struct {
    int32_t batch;               /* B                                            */
    int32_t num_q_heads;         /* Hq                                           */
    int32_t num_kv_heads;        /* Hkv                                          */
    int32_t head_dim;            /* D (128)                                      */
    int32_t page_size;           /* P (16)                                       */
    int32_t num_pages;           /* pages in kv_pool (device bounds checks)      */
    int32_t max_blocks_per_seq;  /* row stride of block_table                    */
    int32_t max_seq_len;         /* host upper bound of seq_lens; sizes the grid */
    float rope_theta;            /* RoPE base, e.g. 1e6                          */
    float eps;                   /* RMSNorm epsilon, e.g. 1e-6                   */
    float sm_scale;              /* softmax scale; 0 selects 1/sqrt(head_dim)    */
    int32_t num_ctas;            /* attention grid size; 0 = automatic (a whole
                                    number of CTAs per SM).  Results do not
                                    depend on it beyond fp32 rounding.          */
    int32_t launch_flags;        /* QDEC_LAUNCH_* bits                           */
} qdec_shape;

/* Bytes of device workspace that qdec_attn_split / qdec_attn_merge /
 * qdec_step need for `shape` on the current device (0 on an invalid shape).
 * The workspace holds the per-piece partial results (o, lse) of the split
 * and one arrival counter per (sequence, KV head). */
size_t qdec_workspace_bytes(const qdec_shape *shape);

/* Bytes of the per-step RoPE table for `shape` (B * D/2 entries of 16 B). */
size_t qdec_rope_table_bytes(const qdec_shape *shape);

/* cos and sin of every RoPE angle positions[b] * rope_theta^(-2i/D) of the
 * step, each kept as an unevaluated pair of floats (about 48 bits), into
 * rope_table (device, qdec_rope_table_bytes).  The angles depend on the
 * positions only, so one table serves all layers of a decode step (the
 * blog's part 3: build per-step metadata once, share it across the 36
 * layers).  Pass it to qdec_step / qdec_append_rope; recompute it whenever
 * positions change. */
qdec_status qdec_rope_table(const qdec_shape *shape, const int32_t *positions,
                            void *rope_table, void *stream);

/* Zero the arrival counters of a fresh workspace.  Call once after
 * allocating it (the kernels leave the counters at zero again when they
 * finish), and again after any call that reported a device error. */
qdec_status qdec_workspace_init(const qdec_shape *shape, void *workspace,
                                size_t workspace_bytes, void *stream);

/* Steps 1-3 for every sequence: RMSNorm + NeoX RoPE of the new q and k rows,
 * then the append of bf16(k_rot) and v into kv_pool at slot seq_lens[b]-1.
 *   q [B][Hq][D] (sequence stride q_stride), k, v [B][Hkv][D] (k_stride,
 *   v_stride); q_norm_w, k_norm_w [D]; positions, seq_lens [B] int32;
 *   block_table [B][max_blocks_per_seq] int32; rope_table from qdec_rope_table
 *   for these positions, or NULL (the angles are then computed in the kernel,
 *   partly in slow fp64); kv_pool as above (written at one slot per
 *   (sequence, KV head) only); q_rot [B][Hq][D] fp32 output, the normed and
 *   rotated query rows, unscaled and unrounded. */
qdec_status qdec_append_rope(const qdec_shape *shape,
                             const qdec_bf16 *q, int64_t q_stride,
                             const qdec_bf16 *k, int64_t k_stride,
                             const qdec_bf16 *v, int64_t v_stride,
                             const qdec_bf16 *q_norm_w, const qdec_bf16 *k_norm_w,
                             const int32_t *positions, const int32_t *seq_lens,
                             const int32_t *block_table, const void *rope_table,
                             qdec_bf16 *kv_pool, float *q_rot, int32_t *err_flag,
                             void *stream);

/* Step 4, first half: split-KV attention of q_rot (from qdec_append_rope)
 * over the pool.  A (sequence, KV head) handled by one piece gets its bf16
 * output written to `out` [B][Hq][D] directly; the others leave partial
 * (o, lse) pairs in the workspace for qdec_attn_merge. */
qdec_status qdec_attn_split(const qdec_shape *shape, const float *q_rot,
                            const qdec_bf16 *kv_pool, const int32_t *block_table,
                            const int32_t *seq_lens, void *workspace,
                            size_t workspace_bytes, qdec_bf16 *out,
                            int32_t *err_flag, void *stream);

/* Step 4, second half: log-sum-exp merge of the partials qdec_attn_split left
 * in the workspace (same shape and seq_lens), bf16 result into `out`. */
qdec_status qdec_attn_merge(const qdec_shape *shape, const int32_t *seq_lens,
                            const void *workspace, size_t workspace_bytes,
                            qdec_bf16 *out, int32_t *err_flag, void *stream);

/* Step 4 whole in ONE launch: split-KV attention of q_rot (from
 * qdec_append_rope or qdec_qkv_append_rope, whose append this launch must
 * follow on the stream) over the pool, and the log-sum-exp merge of every
 * split (sequence, KV head) by the last of its pieces to finish, bf16 result
 * into out [B][Hq][D].  The work plan (cluster or flat layout) is
 * qdec_step's; the workspace counters must be zero on entry
 * (qdec_workspace_init once; every launch leaves them zero).  With
 * QDEC_LAUNCH_OVERLAP_PREVIOUS the launch may start while the previous kernel
 * on the stream finishes; it reads q_rot, the pool and writes out only after
 * that kernel has completed.  Errors as qdec_attn_split. */
qdec_status qdec_attn_decode(const qdec_shape *shape, const float *q_rot,
                             const qdec_bf16 *kv_pool, const int32_t *block_table,
                             const int32_t *seq_lens, void *workspace,
                             size_t workspace_bytes, qdec_bf16 *out,
                             int32_t *err_flag, void *stream);

/* The whole layer-step (steps 1-4).  In ONE kernel launch where the work
 * plan is the cluster layout (few (sequence, KV head) segments): every CTA
 * norms and rotates the four query rows of the (sequence, KV head) it works
 * on, the CTA that holds the last page of a (sequence, KV head) also norms,
 * rotates and appends the new key/value, and the last CTA to finish a split
 * (sequence, KV head) merges its pieces.  On the flat layout (many
 * segments, each CTA walking several) in TWO: the kernel of
 * qdec_append_rope (q_rot kept in the workspace), then the attention of
 * qdec_attn_decode as its programmatic dependent -- there the per-segment
 * new-token work inside the attention kernel costs more than the second
 * launch.  (Over an FP8 pool the first of the two is never launched as a
 * programmatic dependent, whatever the flags: started early, its CTAs slowed
 * the previous attention.)  qdec_step_launches tells which.  Either way the grid
 * depends on the shape only (one captured graph serves every length).  Same
 * arguments as qdec_append_rope plus the workspace and `out`; no q_rot
 * buffer is needed.  The workspace counters must be zero on entry
 * (qdec_workspace_init once).  See QDEC_LAUNCH_OVERLAP_PREVIOUS for
 * overlapping consecutive layers. */
qdec_status qdec_step(const qdec_shape *shape,
                      const qdec_bf16 *q, int64_t q_stride,
                      const qdec_bf16 *k, int64_t k_stride,
                      const qdec_bf16 *v, int64_t v_stride,
                      const qdec_bf16 *q_norm_w, const qdec_bf16 *k_norm_w,
                      const int32_t *positions, const int32_t *seq_lens,
                      const int32_t *block_table, const void *rope_table,
                      qdec_bf16 *kv_pool, void *workspace, size_t workspace_bytes,
                      qdec_bf16 *out, int32_t *err_flag, void *stream);

/* Kernel launches of one qdec_step (fp8_pool = 0) or qdec_step_fp8
 * (fp8_pool != 0) call for this shape on the current device: 1 or 2; 0 for
 * an invalid shape.  Host only, no device work. */
int qdec_step_launches(const qdec_shape *shape, int fp8_pool);

/* The merged QKV projection fused with steps 1-3 (article "扔掉 vLLM！从零
 * 构建 Qwen3-8B 推理引擎" (news.rkmt.cn), section 4.4.3: the q, k and v
 * projections as one matrix), in place of qdec_append_rope when the layer's
 * input is the hidden state:
 *   qkv = W x[b]  for every sequence b, with
 *   x [B][hidden] bf16 (row stride x_stride elements, a multiple of 8),
 *   W = w_qkv [(Hq + 2 Hkv) * 128][hidden] bf16, row-major: rows h*128 .. +127
 *     are query head h, then the key heads, then the value heads (no bias),
 *     passed in the packed order qdec_qkv_pack_weights writes (once per
 *     model load);
 *   hidden a multiple of 64.
 * The projection is kept unrounded (fp32 accumulate) into RMSNorm + NeoX RoPE
 * of the q and k heads and the append: q_rot [B][Hq][128] fp32 (as
 * qdec_append_rope writes it, for qdec_attn_split / qdec_attn_merge), bf16 of
 * the rotated k and of v into slot seq_lens[b]-1 of kv_pool (bf16 pool).
 * rope_table (from qdec_rope_table) is required.  Errors as qdec_append_rope;
 * hidden not a multiple of 64 gives QDEC_ERR_UNSUPPORTED. */
qdec_status qdec_qkv_append_rope(const qdec_shape *shape, int32_t hidden,
                                 const qdec_bf16 *x, int64_t x_stride,
                                 const qdec_bf16 *w_packed,
                                 const qdec_bf16 *q_norm_w, const qdec_bf16 *k_norm_w,
                                 const int32_t *positions, const int32_t *seq_lens,
                                 const int32_t *block_table, const void *rope_table,
                                 qdec_bf16 *kv_pool, float *q_rot, int32_t *err_flag,
                                 void *stream);

/* Rearranges w_qkv (row-major, as above) into w_packed (a separate buffer of
 * the same size, 16-byte aligned): per (output head, block of 64 hidden
 * elements) 16 KiB, the head's 128 rows in four 4 KiB sub-blocks (sub-block i:
 * dims 16i .. 16i+15, then 64+16i .. 64+16i+15), each 128-byte row swizzled,
 * so each CTA of the projection streams one contiguous run.  A device-side
 * copy on `stream`; run it once per weight. */
qdec_status qdec_qkv_pack_weights(const qdec_shape *shape, int32_t hidden,
                                  const qdec_bf16 *w_qkv, qdec_bf16 *w_packed, void *stream);

/* ------------------------------------------------------- chunked prefill --
 * The step that fills the pool (article "扔掉 vLLM！从零构建 Qwen3-8B 推理引擎"
 * (news.rkmt.cn), section 4.4.1: FlashAttention-2 prefill, queries in blocks
 * that see only keys at or before them).  A chunk of n_b new tokens per
 * sequence (n_b may be 0), packed as rows qo_indptr[b] .. qo_indptr[b+1]-1
 * (qo_indptr [B+1] int32, qo_indptr[0] = 0, non-decreasing, qo_indptr[B] <=
 * num_tokens); chunk row j of sequence b becomes token t = seq_lens[b] - n_b
 * + j of it (seq_lens counted after the chunk, n_b <= seq_lens[b]).  The
 * block table must map every page up to token seq_lens[b] - 1.  Sequences
 * whose chunk is malformed are skipped and flagged QDEC_FLAG_BAD_SEQLEN.
 * shape->batch = B sequences; shape->num_ctas is ignored.  With
 * QDEC_LAUNCH_OVERLAP_PREVIOUS, qdec_prefill_attn (bf16 or FP8 pool) may
 * start while the previous kernel on the stream finishes: it reads
 * qo_indptr, seq_lens and the block table at once, and waits for that kernel
 * before it reads q_rot, the pool or kv_scale or writes out (set the flag only
 * when the previous kernel writes none of the first three); the append
 * ignores the flag (it starts after the previous kernel).
 * FP8-pool forms follow the FP8 section below. */

/* The RoPE angles of num_tokens chunk rows (row r at positions[r]) into
 * rope_table (device, 16-byte aligned, qdec_prefill_rope_table_bytes):
 * computed once per step, they serve every layer's qdec_prefill_append_rope
 * (the angles depend on the positions only), as qdec_rope_table does for
 * decode.  One launch. */
size_t qdec_prefill_rope_table_bytes(int32_t num_tokens);
qdec_status qdec_prefill_rope_table(const qdec_shape *shape, int32_t num_tokens,
                                    const int32_t *positions, void *rope_table, void *stream);

/* Steps 1-3 for every chunk row r: RMSNorm + NeoX RoPE at positions[r] of
 * its query rows (q [num_tokens][Hq][D], row stride q_stride) into q_rot
 * [num_tokens][Hq][D] fp32 (unscaled), and of its key rows; bf16(k_rot) and v
 * (k, v [num_tokens][Hkv][D], row strides k_stride, v_stride) into slot t of
 * its sequence.  positions [num_tokens] int32.  rope_table: NULL (each row's
 * angles computed in the kernel) or the rows' angles from
 * qdec_prefill_rope_table over the same positions (the same bits, fewer
 * instructions per layer).  Errors as qdec_append_rope. */
qdec_status qdec_prefill_append_rope(const qdec_shape *shape, int32_t num_tokens,
                                     const qdec_bf16 *q, int64_t q_stride,
                                     const qdec_bf16 *k, int64_t k_stride,
                                     const qdec_bf16 *v, int64_t v_stride,
                                     const qdec_bf16 *q_norm_w, const qdec_bf16 *k_norm_w,
                                     const int32_t *positions, const void *rope_table,
                                     const int32_t *qo_indptr,
                                     const int32_t *seq_lens, const int32_t *block_table,
                                     qdec_bf16 *kv_pool, float *q_rot, int32_t *err_flag,
                                     void *stream);

/* Causal paged attention of the chunk: q_rot row r (query head h) of
 * sequence b attends to tokens 0 .. t of b through KV head h / (Hq / Hkv),
 * softmax scale shape->sm_scale (0: 1/sqrt(D)); bf16 out [num_tokens][Hq][D]
 * (rows past qo_indptr[B] untouched).  Run after qdec_prefill_append_rope on
 * the same stream.  One launch; no workspace. */
qdec_status qdec_prefill_attn(const qdec_shape *shape, int32_t num_tokens, const float *q_rot,
                              const int32_t *qo_indptr, const int32_t *seq_lens,
                              const int32_t *block_table, const qdec_bf16 *kv_pool,
                              qdec_bf16 *out, int32_t *err_flag, void *stream);

/* ------------------------------------------------------------ FP8 KV pool --
 * The same block over a KV cache held in FP8 (essay "推理引擎里面发生了什么"
 * (locsic.com), section on quantization: an FP8 KV cache halves its memory
 * and traffic at a negligible quality cost; the format and the scale
 * granularity are not given there, the choices below are this library's):
 *   kv_pool_fp8[num_pages][2][Hkv][P][D] uint8 -- OCP E4M3 codes (sign, 4
 *     exponent bits with bias 7, 3 mantissa bits, subnormals, NaN =
 *     S.1111.111, no infinity, largest finite 448), the bf16 pool's layout
 *     with one byte per element (a (page, plane, head) tile is 2 KiB);
 *   kv_scale[num_pages][2][Hkv] float -- one scale per (page, plane, KV
 *     head): an element's value is e4m3(code) * scale.  The caller sets a
 *     page's scales (positive, finite) before the page is first written and
 *     owns them like the block table; the library only reads them.
 * The append quantizes the row the bf16 entry points would store:
 *   K code = E4M3_RNE_satfinite(fp32(bf16(k_rot)) / scale_K),
 *   V code = E4M3_RNE_satfinite(fp32(v) / scale_V),
 * each division rounded once to fp32, then round-to-nearest-even to E4M3 with
 * magnitudes beyond 448 saturating to +-448.  The attention computes with the
 * dequantized values (scores and the output in fp32, as in the bf16 path);
 * out stays bf16 [B][Hq][D].  Requires num_kv_heads even (UNSUPPORTED
 * otherwise); kv_pool_fp8 and kv_scale must be 16-byte aligned.  The
 * workspace (qdec_workspace_bytes) and qdec_attn_merge serve both pool types. */

/* qdec_append_rope with an FP8 pool: writes the codes of slot seq_lens[b]-1
 * of every (sequence, KV head); kv_scale is read only. */
qdec_status qdec_append_rope_fp8(const qdec_shape *shape,
                                 const qdec_bf16 *q, int64_t q_stride,
                                 const qdec_bf16 *k, int64_t k_stride,
                                 const qdec_bf16 *v, int64_t v_stride,
                                 const qdec_bf16 *q_norm_w, const qdec_bf16 *k_norm_w,
                                 const int32_t *positions, const int32_t *seq_lens,
                                 const int32_t *block_table, const void *rope_table,
                                 uint8_t *kv_pool_fp8, const float *kv_scale, float *q_rot,
                                 int32_t *err_flag, void *stream);

/* qdec_attn_split over an FP8 pool; finish with qdec_attn_merge. */
qdec_status qdec_attn_split_fp8(const qdec_shape *shape, const float *q_rot,
                                const uint8_t *kv_pool_fp8, const float *kv_scale,
                                const int32_t *block_table, const int32_t *seq_lens,
                                void *workspace, size_t workspace_bytes, qdec_bf16 *out,
                                int32_t *err_flag, void *stream);

/* qdec_attn_decode over an FP8 pool. */
qdec_status qdec_attn_decode_fp8(const qdec_shape *shape, const float *q_rot,
                                 const uint8_t *kv_pool_fp8, const float *kv_scale,
                                 const int32_t *block_table, const int32_t *seq_lens,
                                 void *workspace, size_t workspace_bytes, qdec_bf16 *out,
                                 int32_t *err_flag, void *stream);

/* Chunked prefill over an FP8 pool: qdec_prefill_append_rope storing the
 * chunk rows' codes (the append rule above, each row with the scales of its
 * slot's (page, plane, head)), and qdec_prefill_attn over the dequantized
 * pool.  kv_scale is read only.
 * qdec_prefill_attn_fp8 with a workspace (device memory, 16-byte aligned, at
 * least qdec_prefill_fp8_workspace_bytes(shape) bytes, caller-owned, no
 * initialisation needed) first dequantizes every page of the chunks'
 * sequences once into it, each value code x scale rounded to bf16 (a
 * relative error of at most 2^-8, against the 2^-4 of the E4M3 code), then
 * runs the bf16-pool attention over that copy: two launches, each page
 * dequantized once instead of once per 64-row query block, and no scale in
 * the softmax (the faster form).  With workspace NULL (workspace_bytes
 * ignored) each block converts the codes it reads exactly to f16 and
 * applies the scales in the softmax: one launch, no memory.  The two agree
 * to within the bf16 rounding of the dequantized values;
 * QDEC_ERR_WORKSPACE if the workspace is too small or misaligned. */
qdec_status qdec_prefill_append_rope_fp8(const qdec_shape *shape, int32_t num_tokens,
                                         const qdec_bf16 *q, int64_t q_stride,
                                         const qdec_bf16 *k, int64_t k_stride,
                                         const qdec_bf16 *v, int64_t v_stride,
                                         const qdec_bf16 *q_norm_w, const qdec_bf16 *k_norm_w,
                                         const int32_t *positions, const void *rope_table,
                                         const int32_t *qo_indptr,
                                         const int32_t *seq_lens, const int32_t *block_table,
                                         uint8_t *kv_pool_fp8, const float *kv_scale,
                                         float *q_rot, int32_t *err_flag, void *stream);
qdec_status qdec_prefill_attn_fp8(const qdec_shape *shape, int32_t num_tokens,
                                  const float *q_rot, const int32_t *qo_indptr,
                                  const int32_t *seq_lens, const int32_t *block_table,
                                  const uint8_t *kv_pool_fp8, const float *kv_scale,
                                  void *workspace, size_t workspace_bytes, qdec_bf16 *out,
                                  int32_t *err_flag, void *stream);
/* Bytes of the workspace that qdec_prefill_attn_fp8 dequantizes into:
 * batch * max_blocks_per_seq pages of 2 * Hkv * 16 * 128 bf16 values
 * (0 for an invalid shape).  Host only. */
size_t qdec_prefill_fp8_workspace_bytes(const qdec_shape *shape);

/* qdec_qkv_append_rope with an FP8 pool: the projected key and value rows,
 * rounded to bf16 as the bf16 pool would hold them, are divided by their
 * slot's scales and rounded to E4M3 (the append rule above). */
qdec_status qdec_qkv_append_rope_fp8(const qdec_shape *shape, int32_t hidden,
                                     const qdec_bf16 *x, int64_t x_stride,
                                     const qdec_bf16 *w_packed,
                                     const qdec_bf16 *q_norm_w, const qdec_bf16 *k_norm_w,
                                     const int32_t *positions, const int32_t *seq_lens,
                                     const int32_t *block_table, const void *rope_table,
                                     uint8_t *kv_pool_fp8, const float *kv_scale, float *q_rot,
                                     int32_t *err_flag, void *stream);

/* qdec_step over an FP8 pool: steps 1-4, the new key and value quantized
 * into their slot as above; one or two launches by the same rule as
 * qdec_step (qdec_step_launches with fp8_pool != 0 tells which).  Same
 * launch flags, workspace and error reporting as qdec_step. */
qdec_status qdec_step_fp8(const qdec_shape *shape,
                          const qdec_bf16 *q, int64_t q_stride,
                          const qdec_bf16 *k, int64_t k_stride,
                          const qdec_bf16 *v, int64_t v_stride,
                          const qdec_bf16 *q_norm_w, const qdec_bf16 *k_norm_w,
                          const int32_t *positions, const int32_t *seq_lens,
                          const int32_t *block_table, const void *rope_table,
                          uint8_t *kv_pool_fp8, const float *kv_scale, void *workspace,
                          size_t workspace_bytes, qdec_bf16 *out, int32_t *err_flag,
                          void *stream);

/* qdec_step without a caller-provided workspace, for callers that cannot
 * allocate device memory (e.g. a serving loop that must not call
 * cudaMalloc/cudaFree once running, or a plugin whose host runtime owns all
 * device allocations).  No counterpart in the pages: it is a deployment
 * convenience, not part of the method.  The scratch is a fixed array of
 * QDEC_STATIC_SCRATCH_BYTES in the library's own device memory, reserved on
 * every device that loads the library and held until the process exits.
 *   - Same arguments as qdec_step minus workspace/workspace_bytes; the caller
 *     still passes every input and output.  Allocates nothing.
 *   - Returns QDEC_ERR_WORKSPACE when the shape needs more scratch than
 *     QDEC_STATIC_SCRATCH_BYTES (qdec_workspace_bytes tells how much).
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - Every call, on any stream, uses the same array, which keeps the
 *     previous call's contents; each call clears the counters it needs on its
 *     stream before the kernel runs.  Calls that can overlap on the GPU (other
 *     streams, other threads) race on the array: serialise them.
 *   - That clearing is a memset on the stream between the previous kernel
 *     and this call's kernel, so QDEC_LAUNCH_OVERLAP_PREVIOUS does not let the
 *     kernel start before the previous one ends through this entry point. */
#define QDEC_STATIC_SCRATCH_BYTES (4u << 20)
qdec_status qdec_step_static_scratch(const qdec_shape *shape,
                                     const qdec_bf16 *q, int64_t q_stride,
                                     const qdec_bf16 *k, int64_t k_stride,
                                     const qdec_bf16 *v, int64_t v_stride,
                                     const qdec_bf16 *q_norm_w, const qdec_bf16 *k_norm_w,
                                     const int32_t *positions, const int32_t *seq_lens,
                                     const int32_t *block_table, const void *rope_table,
                                     qdec_bf16 *kv_pool, qdec_bf16 *out, int32_t *err_flag,
                                     void *stream);

/* Synchronise `stream`, read *err_flag (device), clear it, and map it to a
 * status: QDEC_OK, QDEC_ERR_DEVICE_BOUNDS or QDEC_ERR_TIMEOUT (QDEC_ERR_CUDA
 * if the stream itself failed).  The raw bits go to *flags_out if not NULL. */
qdec_status qdec_check_error(int32_t *err_flag, void *stream, int32_t *flags_out);

/* Static, human-readable name of a status. */
const char *qdec_status_string(qdec_status status);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t qdec_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QDEC_H */
