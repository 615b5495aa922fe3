/*
 * qdec_oracle.c -- plain, slow, fp64 CPU oracle for one GQA decode-attention
 * layer-step over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference leg use it.  It shares no code, header, table or
 * constant with the CUDA library; the two meet only in the caller's buffers.
 *
 * Every step is written from its definition, single-threaded, in double:
 *
 *   RMSNorm   -- blog "GPU 算子与执行优化：从 26 到 100 token/s 的推理引擎破茧之路" (yuzheng310.github.io), part 6 (fusing
 *               Norm and RoPE): y = x * rsqrt(mean(x^2) + eps) * w, computed
 *               per head row after the Q/K projection.
 *   NeoX RoPE -- same blog, part 6, fused NeoX RoPE (interleave=False, i.e.
 *               rotate-half): pairs (i, i + D/2) are rotated by
 *               theta_i = pos * rope_theta^(-2i/D).
 *   append    -- essay "推理引擎里面发生了什么" (locsic.com),
 *               PagedAttention section: a request maps logical blocks of 16
 *               tokens to physical blocks through its block table.
 *   attention -- same essay, "standard attention" (S = QK^T, P = softmax(S),
 *               O = PV) restricted to one query row, with the 1/sqrt(d_head)
 *               scale and the GQA head mapping g = h / heads_per_group of the
 *               article "扔掉 vLLM！从零构建 Qwen3-8B 推理引擎" (news.rkmt.cn),
 *               section 4.4.2.
 *   split/merge -- blog part 8: one head's KV sequence is cut into parts,
 *               each part gets a local softmax, the parts are then reduced.
 *               The reduction is the exact log-sum-exp merge.
 *   prefill   -- engine article, section 4.4.1 (FlashAttention-2 prefill):
 *               a chunk of new tokens per sequence is normed, rotated and
 *               appended like the decode token, then every chunk query row
 *               attends causally (keys at or before its own index); the
 *               blockwise computation there is exact, so the oracle is plain
 *               causal softmax attention.  Its printed loop takes a softmax
 *               per key block and adds the blocks, which is not attention;
 *               the plain reading is taken.
 *   QKV projection -- engine article, section 4.4.3 (fused QKV): one merged
 *               matrix W [(Hq + 2 Hkv) D][hidden] (rows: the q heads, then the
 *               k heads, then the v heads) gives qkv = W x for each sequence;
 *               fused with steps 1-3 the projection stays unrounded (double
 *               here) into the norm, the rotation and the append.
 *   FP8 KV    -- essay, section on quantization: the KV cache held in FP8
 *               (half the bytes).  Codes are OCP E4M3; every (page, plane,
 *               KV head) carries one fp32 scale, value = e4m3(code) * scale.
 *               The append quantizes the bf16 row it would otherwise store:
 *               code = RNE_e4m3_satfinite(fp32(row) / scale), the division
 *               rounded once to fp32.
 *
 * Pool layout (the reading adopted for the shape the blog prints in part 4,
 * [num_blocks, num_heads, block_size, head_dim], with K and V in one tensor):
 *   pool[num_pages][2 (0 = K, 1 = V)][Hkv][P][D], bf16 stored as uint16.
 *
 * Parity pins: every function here is pinned by tests/test_oracle.py against
 * closed forms, invariants and brute force (see that file's header).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- bf16 -- */

/* bf16 is the top half of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static uint16_t float_bits_hi(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* Round a double straight to bf16, round-to-nearest-even (one rounding, no
 * detour through binary32).  bf16: 8 exponent bits, 7 stored mantissa bits,
 * so a value in [2^(e-1), 2^e) has spacing 2^(e-8); below the smallest
 * normal 2^-126 the spacing stays 2^-133. */
uint16_t oracle_double_to_bf16(double x)
{
    if (isnan(x))
        return (uint16_t)(signbit(x) ? 0xFFC0u : 0x7FC0u);
    if (isinf(x) || x == 0.0)
        return float_bits_hi((float)x);  /* exact: +-inf, +-0 */
    int e;
    (void)frexp(x, &e);                  /* |x| in [2^(e-1), 2^e) */
    if (e < -125)
        e = -125;
    double ulp = ldexp(1.0, e - 8);
    double r = nearbyint(x / ulp) * ulp; /* default mode: nearest-even */
    if (fabs(r) >= ldexp(1.0, 128))
        return (uint16_t)(r > 0 ? 0x7F80u : 0xFF80u);
    return float_bits_hi((float)r);      /* r is exact in bf16 */
}

/* ------------------------------------------------------------- RMSNorm -- */

/* y = x * 1/sqrt(mean(x^2) + eps) * w, eps inside the root. */
void oracle_rmsnorm(const double *x, const double *w, int D, double eps, double *y)
{
    double ss = 0.0;
    for (int i = 0; i < D; ++i)
        ss += x[i] * x[i];
    double r = 1.0 / sqrt(ss / (double)D + eps);
    for (int i = 0; i < D; ++i)
        y[i] = x[i] * r * w[i];
}

/* ----------------------------------------------------------- NeoX RoPE -- */

/* Rotate-half RoPE: for i < D/2, angle a = pos * theta^(-2i/D),
 *   y[i]       = x[i] cos a - x[i+D/2] sin a
 *   y[i+D/2]   = x[i+D/2] cos a + x[i] sin a          */
void oracle_rope_neox(const double *x, int D, double pos, double theta, double *y)
{
    int half = D / 2;
    for (int i = 0; i < half; ++i) {
        double inv_freq = pow(theta, -2.0 * (double)i / (double)D);
        double a = pos * inv_freq;
        double c = cos(a), s = sin(a);
        double x1 = x[i], x2 = x[i + half];
        y[i] = x1 * c - x2 * s;
        y[i + half] = x2 * c + x1 * s;
    }
}

/* ------------------------------------------------------- pool addressing -- */

typedef struct {
    int B, Hq, Hkv, D, P, num_pages, max_blocks;
} oracle_dims;

/* Element offset of token row `t` of sequence `b`, head `h`, plane kv
 * (0 = K, 1 = V) in the pool, through the block table.  Returns -1 if the
 * block table entry is outside the pool. */
static long pool_row(const oracle_dims *d, const int32_t *block_table, int b, int t,
                     int kv, int h)
{
    int32_t page = block_table[(long)b * d->max_blocks + t / d->P];
    if (page < 0 || page >= d->num_pages)
        return -1;
    return ((((long)page * 2 + kv) * d->Hkv + h) * d->P + (t % d->P)) * (long)d->D;
}

/* ------------------------------------------------------------ attention -- */

/* One query row against tokens [t0, t1) of sequence b, KV head g:
 *   s_t = scale * <q, K_t>;  m = max s;  w_t = exp(s_t - m)
 *   out = sum w_t V_t / sum w_t;  lse = m + log(sum w_t).
 * Returns 0, or -1 on a block-table entry outside the pool. */
static int attend_range(const oracle_dims *d, const uint16_t *pool,
                        const int32_t *block_table, int b, int g, const double *q,
                        double scale, int t0, int t1, double *out, double *lse)
{
    int D = d->D;
    int n = t1 - t0;
    double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double m = -INFINITY;
    for (int t = t0; t < t1; ++t) {
        long row = pool_row(d, block_table, b, t, 0, g);
        if (row < 0) {
            free(s);
            return -1;
        }
        double dot = 0.0;
        for (int i = 0; i < D; ++i)
            dot += q[i] * oracle_bf16_to_double(pool[row + i]);
        s[t - t0] = scale * dot;
        if (s[t - t0] > m)
            m = s[t - t0];
    }
    double l = 0.0;
    for (int i = 0; i < D; ++i)
        out[i] = 0.0;
    for (int t = t0; t < t1; ++t) {
        double w = exp(s[t - t0] - m);
        l += w;
        long row = pool_row(d, block_table, b, t, 1, g);
        for (int i = 0; i < D; ++i)
            out[i] += w * oracle_bf16_to_double(pool[row + i]);
    }
    for (int i = 0; i < D; ++i)
        out[i] /= l;
    *lse = m + log(l);
    free(s);
    return 0;
}

/* Attention of every query head of every sequence over its whole context,
 * with q_rot given in double (already normed and rotated).
 *   q_rot [B][Hq][D]; out [B][Hq][D]; lse [B][Hq]. */
int oracle_attention(int B, int Hq, int Hkv, int D, int P, int num_pages,
                     int max_blocks, const uint16_t *pool, const int32_t *block_table,
                     const int32_t *seq_lens, const double *q_rot, double scale,
                     double *out, double *lse)
{
    oracle_dims d = {B, Hq, Hkv, D, P, num_pages, max_blocks};
    int G = Hq / Hkv;
    for (int b = 0; b < B; ++b) {
        int L = seq_lens[b];
        if (L < 1 || L > max_blocks * P)
            return -2;
        for (int h = 0; h < Hq; ++h) {
            int g = h / G;
            long o = ((long)b * Hq + h) * D;
            if (attend_range(&d, pool, block_table, b, g, q_rot + o, scale, 0, L, out + o,
                             lse + (long)b * Hq + h))
                return -1;
        }
    }
    return 0;
}

/* Split mode: sequence b is cut into chunks of `chunk_pages` pages; each
 * chunk gives a partial (o_s, lse_s); the partials are merged exactly:
 *   M = max_s lse_s;  out = sum_s e^(lse_s - M) o_s / sum_s e^(lse_s - M);
 *   lse = M + log(sum_s e^(lse_s - M)).
 * Exists to pin the merge: for any chunking it must equal oracle_attention. */
int oracle_attention_split(int B, int Hq, int Hkv, int D, int P, int num_pages,
                           int max_blocks, const uint16_t *pool,
                           const int32_t *block_table, const int32_t *seq_lens,
                           const double *q_rot, double scale, int chunk_pages,
                           double *out, double *lse)
{
    oracle_dims d = {B, Hq, Hkv, D, P, num_pages, max_blocks};
    int G = Hq / Hkv;
    if (chunk_pages < 1)
        return -3;
    double *o_s = (double *)malloc(sizeof(double) * (size_t)D);
    for (int b = 0; b < B; ++b) {
        int L = seq_lens[b];
        if (L < 1 || L > max_blocks * P) {
            free(o_s);
            return -2;
        }
        int chunk = chunk_pages * P;
        int S = (L + chunk - 1) / chunk;
        for (int h = 0; h < Hq; ++h) {
            int g = h / G;
            long o = ((long)b * Hq + h) * D;
            double *lse_s = (double *)malloc(sizeof(double) * (size_t)S);
            double *o_all = (double *)malloc(sizeof(double) * (size_t)S * D);
            double M = -INFINITY;
            for (int s = 0; s < S; ++s) {
                int t0 = s * chunk, t1 = t0 + chunk < L ? t0 + chunk : L;
                if (attend_range(&d, pool, block_table, b, g, q_rot + o, scale, t0, t1,
                                 o_all + (long)s * D, &lse_s[s])) {
                    free(lse_s);
                    free(o_all);
                    free(o_s);
                    return -1;
                }
                if (lse_s[s] > M)
                    M = lse_s[s];
            }
            double den = 0.0;
            for (int i = 0; i < D; ++i)
                o_s[i] = 0.0;
            for (int s = 0; s < S; ++s) {
                double w = exp(lse_s[s] - M);
                den += w;
                for (int i = 0; i < D; ++i)
                    o_s[i] += w * o_all[(long)s * D + i];
            }
            for (int i = 0; i < D; ++i)
                out[o + i] = o_s[i] / den;
            lse[(long)b * Hq + h] = M + log(den);
            free(lse_s);
            free(o_all);
        }
    }
    free(o_s);
    return 0;
}

/* ---------------------------------------------------------- layer-step -- */

/* One decode layer-step, in the order the blog's decode path runs it:
 *   1. per head row: RMSNorm (q rows with w_q, k rows with w_k), then NeoX
 *      RoPE at positions[b];
 *   2. append: slot t = seq_lens[b] - 1 of sequence b receives bf16(k_rot)
 *      (one round-to-nearest-even) and v (bits copied) for every KV head;
 *   3. attention of every q head over tokens 0..seq_lens[b]-1, the new token
 *      included (it reads the rounded k just written);
 * Inputs are bf16 (uint16) and converted exactly to double.
 *   q [B][Hq][D], k,v [B][Hkv][D], w_q,w_k [D], positions,seq_lens [B],
 *   block_table [B][max_blocks], pool as described at the top (updated).
 * Outputs (double): q_rot [B][Hq][D], k_rot [B][Hkv][D] (unrounded),
 *   out [B][Hq][D], lse [B][Hq].  scale <= 0 selects 1/sqrt(D).
 * Returns 0; -1 block-table entry outside the pool; -2 bad seq_len;
 * -4 Hq not a multiple of Hkv or odd D. */
int oracle_decode_layer(int B, int Hq, int Hkv, int D, int P, int num_pages,
                        int max_blocks, const uint16_t *q, const uint16_t *k,
                        const uint16_t *v, const uint16_t *w_q, const uint16_t *w_k,
                        const int32_t *positions, const int32_t *seq_lens,
                        const int32_t *block_table, uint16_t *pool, double rope_theta,
                        double eps, double scale, double *q_rot, double *k_rot,
                        double *out, double *lse)
{
    if (Hkv < 1 || Hq % Hkv != 0 || D % 2 != 0)
        return -4;
    oracle_dims d = {B, Hq, Hkv, D, P, num_pages, max_blocks};
    if (scale <= 0.0)
        scale = 1.0 / sqrt((double)D);
    double *x = (double *)malloc(sizeof(double) * (size_t)D);
    double *xn = (double *)malloc(sizeof(double) * (size_t)D);
    double *wq = (double *)malloc(sizeof(double) * (size_t)D);
    double *wk = (double *)malloc(sizeof(double) * (size_t)D);
    for (int i = 0; i < D; ++i) {
        wq[i] = oracle_bf16_to_double(w_q[i]);
        wk[i] = oracle_bf16_to_double(w_k[i]);
    }
    int rc = 0;
    for (int b = 0; b < B && rc == 0; ++b) {
        int L = seq_lens[b];
        if (L < 1 || L > max_blocks * P) {
            rc = -2;
            break;
        }
        double pos = (double)positions[b];
        /* step 1: q rows */
        for (int h = 0; h < Hq; ++h) {
            long o = ((long)b * Hq + h) * D;
            for (int i = 0; i < D; ++i)
                x[i] = oracle_bf16_to_double(q[o + i]);
            oracle_rmsnorm(x, wq, D, eps, xn);
            oracle_rope_neox(xn, D, pos, rope_theta, q_rot + o);
        }
        /* steps 1-2: k rows, then the append of k and v */
        for (int h = 0; h < Hkv; ++h) {
            long o = ((long)b * Hkv + h) * D;
            for (int i = 0; i < D; ++i)
                x[i] = oracle_bf16_to_double(k[o + i]);
            oracle_rmsnorm(x, wk, D, eps, xn);
            oracle_rope_neox(xn, D, pos, rope_theta, k_rot + o);
            long rk = pool_row(&d, block_table, b, L - 1, 0, h);
            long rv = pool_row(&d, block_table, b, L - 1, 1, h);
            if (rk < 0 || rv < 0) {
                rc = -1;
                break;
            }
            for (int i = 0; i < D; ++i) {
                pool[rk + i] = oracle_double_to_bf16(k_rot[o + i]);
                pool[rv + i] = v[o + i];
            }
        }
    }
    /* step 3 (after every append, as in a batched layer) */
    if (rc == 0)
        rc = oracle_attention(B, Hq, Hkv, D, P, num_pages, max_blocks, pool, block_table,
                              seq_lens, q_rot, scale, out, lse);
    free(x);
    free(xn);
    free(wq);
    free(wk);
    return rc;
}

/* ------------------------------------------------------------ fp8 e4m3 -- */

/* E4M3 as the OCP 8-bit floating point format defines it: a sign bit, four
 * exponent bits with bias 7 and three mantissa bits.  Exponent field 0 holds
 * the subnormals m/8 * 2^-6; exponent and mantissa fields all ones is NaN;
 * there is no infinity, so the largest finite value is 1.75 * 2^8 = 448. */
double oracle_e4m3_to_double(uint8_t c)
{
    int neg = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
    double mag;
    if (e == 0xF && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);
    else
        mag = ldexp(8.0 + m, e - 10);
    return neg ? -mag : mag;
}

/* Round a binary32 value to E4M3, nearest-even, saturating: a magnitude at or
 * beyond the largest finite 448 (infinity included) gives +-448, NaN gives
 * the NaN pattern 0x7F, the sign of zero is kept.  Spacing: 2^(e-4) in
 * [2^(e-1), 2^e), never below the subnormal step 2^-9. */
uint8_t oracle_float_to_e4m3_satfinite(float xf)
{
    double x = (double)xf;
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    if (a == 0.0)
        return sign;
    int e;
    (void)frexp(a, &e);                    /* a in [2^(e-1), 2^e) */
    if (e < -5)
        e = -5;
    double ulp = ldexp(1.0, e - 4);
    double r = nearbyint(a / ulp) * ulp;   /* default mode: nearest-even */
    if (r < ldexp(1.0, -6))                /* subnormal (or zero) */
        return (uint8_t)(sign | (int)(r / ldexp(1.0, -9)));
    int er;
    (void)frexp(r, &er);                   /* r in [2^(er-1), 2^er) */
    int field = er - 1 + 7;
    int m = (int)((r / ldexp(1.0, er - 1) - 1.0) * 8.0);
    return (uint8_t)(sign | (field << 3) | m);
}

/* Offset of the scale of (page of token t of sequence b, plane kv, head h):
 * kv_scale[num_pages][2][Hkv].  -1 if the block-table entry is outside the
 * pool. */
static long scale_index(const oracle_dims *d, const int32_t *block_table, int b, int t,
                        int kv, int h)
{
    int32_t page = block_table[(long)b * d->max_blocks + t / d->P];
    if (page < 0 || page >= d->num_pages)
        return -1;
    return ((long)page * 2 + kv) * d->Hkv + h;
}

/* attend_range over an FP8 pool: row elements are e4m3(code) * scale (exact
 * in double), then the same scores, softmax and weighted sum. */
static int attend_range_fp8(const oracle_dims *d, const uint8_t *pool8, const float *kv_scale,
                            const int32_t *block_table, int b, int g, const double *q,
                            double scale, int t0, int t1, double *out, double *lse)
{
    int D = d->D;
    int n = t1 - t0;
    double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double m = -INFINITY;
    for (int t = t0; t < t1; ++t) {
        long row = pool_row(d, block_table, b, t, 0, g);
        long si = scale_index(d, block_table, b, t, 0, g);
        if (row < 0 || si < 0) {
            free(s);
            return -1;
        }
        double sk = (double)kv_scale[si];
        double dot = 0.0;
        for (int i = 0; i < D; ++i)
            dot += q[i] * (oracle_e4m3_to_double(pool8[row + i]) * sk);
        s[t - t0] = scale * dot;
        if (s[t - t0] > m)
            m = s[t - t0];
    }
    double l = 0.0;
    for (int i = 0; i < D; ++i)
        out[i] = 0.0;
    for (int t = t0; t < t1; ++t) {
        double w = exp(s[t - t0] - m);
        l += w;
        long row = pool_row(d, block_table, b, t, 1, g);
        double sv = (double)kv_scale[scale_index(d, block_table, b, t, 1, g)];
        for (int i = 0; i < D; ++i)
            out[i] += w * (oracle_e4m3_to_double(pool8[row + i]) * sv);
    }
    for (int i = 0; i < D; ++i)
        out[i] /= l;
    *lse = m + log(l);
    free(s);
    return 0;
}

/* oracle_attention over an FP8 pool (pool8 laid out like the bf16 pool, one
 * byte per element) with its scales kv_scale[num_pages][2][Hkv]. */
int oracle_attention_fp8(int B, int Hq, int Hkv, int D, int P, int num_pages,
                         int max_blocks, const uint8_t *pool8, const float *kv_scale,
                         const int32_t *block_table, const int32_t *seq_lens,
                         const double *q_rot, double scale, double *out, double *lse)
{
    oracle_dims d = {B, Hq, Hkv, D, P, num_pages, max_blocks};
    int G = Hq / Hkv;
    for (int b = 0; b < B; ++b) {
        int L = seq_lens[b];
        if (L < 1 || L > max_blocks * P)
            return -2;
        for (int h = 0; h < Hq; ++h) {
            int g = h / G;
            long o = ((long)b * Hq + h) * D;
            if (attend_range_fp8(&d, pool8, kv_scale, block_table, b, g, q_rot + o, scale, 0,
                                 L, out + o, lse + (long)b * Hq + h))
                return -1;
        }
    }
    return 0;
}

/* oracle_decode_layer with an FP8 pool: the same norm and rotation, then the
 * append stores, for every element of the new row,
 *   K: RNE_e4m3_satfinite(fp32(bf16(k_rot)) / scale_K)
 *   V: RNE_e4m3_satfinite(fp32(v) / scale_V)
 * with the scales of the (page, plane, head) the slot lies in (the scales
 * are inputs and are not changed), then the attention over the FP8 pool. */
int oracle_decode_layer_fp8(int B, int Hq, int Hkv, int D, int P, int num_pages,
                            int max_blocks, const uint16_t *q, const uint16_t *k,
                            const uint16_t *v, const uint16_t *w_q, const uint16_t *w_k,
                            const int32_t *positions, const int32_t *seq_lens,
                            const int32_t *block_table, uint8_t *pool8,
                            const float *kv_scale, double rope_theta, double eps,
                            double scale, double *q_rot, double *k_rot, double *out,
                            double *lse)
{
    if (Hkv < 1 || Hq % Hkv != 0 || D % 2 != 0)
        return -4;
    oracle_dims d = {B, Hq, Hkv, D, P, num_pages, max_blocks};
    if (scale <= 0.0)
        scale = 1.0 / sqrt((double)D);
    double *x = (double *)malloc(sizeof(double) * (size_t)D);
    double *xn = (double *)malloc(sizeof(double) * (size_t)D);
    double *wq = (double *)malloc(sizeof(double) * (size_t)D);
    double *wk = (double *)malloc(sizeof(double) * (size_t)D);
    for (int i = 0; i < D; ++i) {
        wq[i] = oracle_bf16_to_double(w_q[i]);
        wk[i] = oracle_bf16_to_double(w_k[i]);
    }
    int rc = 0;
    for (int b = 0; b < B && rc == 0; ++b) {
        int L = seq_lens[b];
        if (L < 1 || L > max_blocks * P) {
            rc = -2;
            break;
        }
        double pos = (double)positions[b];
        for (int h = 0; h < Hq; ++h) {
            long o = ((long)b * Hq + h) * D;
            for (int i = 0; i < D; ++i)
                x[i] = oracle_bf16_to_double(q[o + i]);
            oracle_rmsnorm(x, wq, D, eps, xn);
            oracle_rope_neox(xn, D, pos, rope_theta, q_rot + o);
        }
        for (int h = 0; h < Hkv; ++h) {
            long o = ((long)b * Hkv + h) * D;
            for (int i = 0; i < D; ++i)
                x[i] = oracle_bf16_to_double(k[o + i]);
            oracle_rmsnorm(x, wk, D, eps, xn);
            oracle_rope_neox(xn, D, pos, rope_theta, k_rot + o);
            long rk = pool_row(&d, block_table, b, L - 1, 0, h);
            long rv = pool_row(&d, block_table, b, L - 1, 1, h);
            long sk = scale_index(&d, block_table, b, L - 1, 0, h);
            long sv = scale_index(&d, block_table, b, L - 1, 1, h);
            if (rk < 0 || rv < 0 || sk < 0 || sv < 0) {
                rc = -1;
                break;
            }
            for (int i = 0; i < D; ++i) {
                float kf = (float)oracle_bf16_to_double(oracle_double_to_bf16(k_rot[o + i]));
                float vf = (float)oracle_bf16_to_double(v[o + i]);
                pool8[rk + i] = oracle_float_to_e4m3_satfinite(kf / kv_scale[sk]);
                pool8[rv + i] = oracle_float_to_e4m3_satfinite(vf / kv_scale[sv]);
            }
        }
    }
    if (rc == 0)
        rc = oracle_attention_fp8(B, Hq, Hkv, D, P, num_pages, max_blocks, pool8, kv_scale,
                                  block_table, seq_lens, q_rot, scale, out, lse);
    free(x);
    free(xn);
    free(wq);
    free(wk);
    return rc;
}

/* ------------------------------------------------------ QKV projection -- */

/* The merged QKV projection fused with steps 1-3, for every sequence b:
 *   qkv[j] = sum_i W[j][i] * x[b][i]          (double, no rounding)
 * rows j of query head h: h*D .. h*D+D-1; key head g: (Hq+g)*D ..; value
 * head g: (Hq+Hkv+g)*D ..; then RMSNorm + NeoX RoPE of the q and k rows at
 * positions[b], and the append of bf16(k_rot) and bf16(v) (each rounded once,
 * nearest-even) into slot seq_lens[b]-1.
 *   x [B][hidden], W [(Hq+2Hkv)*D][hidden], w_q, w_k [D] (bf16 as uint16).
 * Outputs (double): q_rot [B][Hq][D], k_rot and v [B][Hkv][D] (unrounded).
 * Returns 0, -1 (block-table entry outside the pool), -2 (bad seq_len),
 * -4 (Hq not a multiple of Hkv, or odd D). */
int oracle_qkv_append(int B, int Hq, int Hkv, int D, int P, int num_pages, int max_blocks,
                      int hidden, const uint16_t *x, const uint16_t *w_qkv,
                      const uint16_t *w_q, const uint16_t *w_k, const int32_t *positions,
                      const int32_t *seq_lens, const int32_t *block_table, uint16_t *pool,
                      double rope_theta, double eps, double *q_rot, double *k_rot,
                      double *v_out)
{
    if (Hkv < 1 || Hq % Hkv != 0 || D % 2 != 0)
        return -4;
    oracle_dims d = {B, Hq, Hkv, D, P, num_pages, max_blocks};
    int rows = (Hq + 2 * Hkv) * D;
    double *qkv = (double *)malloc(sizeof(double) * (size_t)rows);
    double *xd = (double *)malloc(sizeof(double) * (size_t)hidden);
    double *xn = (double *)malloc(sizeof(double) * (size_t)D);
    double *wq = (double *)malloc(sizeof(double) * (size_t)D);
    double *wk = (double *)malloc(sizeof(double) * (size_t)D);
    for (int i = 0; i < D; ++i) {
        wq[i] = oracle_bf16_to_double(w_q[i]);
        wk[i] = oracle_bf16_to_double(w_k[i]);
    }
    int rc = 0;
    for (int b = 0; b < B && rc == 0; ++b) {
        int L = seq_lens[b];
        if (L < 1 || L > max_blocks * P) {
            rc = -2;
            break;
        }
        double pos = (double)positions[b];
        for (int i = 0; i < hidden; ++i)
            xd[i] = oracle_bf16_to_double(x[(long)b * hidden + i]);
        for (int j = 0; j < rows; ++j) {
            double acc = 0.0;
            for (int i = 0; i < hidden; ++i)
                acc += oracle_bf16_to_double(w_qkv[(long)j * hidden + i]) * xd[i];
            qkv[j] = acc;
        }
        for (int h = 0; h < Hq; ++h) {
            oracle_rmsnorm(qkv + (long)h * D, wq, D, eps, xn);
            oracle_rope_neox(xn, D, pos, rope_theta, q_rot + ((long)b * Hq + h) * D);
        }
        for (int g = 0; g < Hkv; ++g) {
            long o = ((long)b * Hkv + g) * D;
            oracle_rmsnorm(qkv + (long)(Hq + g) * D, wk, D, eps, xn);
            oracle_rope_neox(xn, D, pos, rope_theta, k_rot + o);
            for (int i = 0; i < D; ++i)
                v_out[o + i] = qkv[(long)(Hq + Hkv + g) * D + i];
            long rk = pool_row(&d, block_table, b, L - 1, 0, g);
            long rv = pool_row(&d, block_table, b, L - 1, 1, g);
            if (rk < 0 || rv < 0) {
                rc = -1;
                break;
            }
            for (int i = 0; i < D; ++i) {
                pool[rk + i] = oracle_double_to_bf16(k_rot[o + i]);
                pool[rv + i] = oracle_double_to_bf16(v_out[o + i]);
            }
        }
    }
    free(qkv);
    free(xd);
    free(xn);
    free(wq);
    free(wk);
    return rc;
}

/* ------------------------------------------------------------- prefill -- */

/* A chunk of new tokens per sequence (chunked prefill): sequence b brings
 * n_b = qo_indptr[b+1] - qo_indptr[b] tokens, packed as rows
 * qo_indptr[b] .. qo_indptr[b+1]-1 of q, k, v; they become tokens
 * L_b - n_b .. L_b - 1 of the sequence (L_b = seq_lens[b], counted after the
 * chunk).  Validates the chunk layout: -2 if qo_indptr[0] != 0, a chunk is
 * negative or longer than its sequence, or L_b is outside [1, max_blocks*P]. */
static int prefill_check(int B, int P, int max_blocks, const int32_t *qo_indptr,
                         const int32_t *seq_lens)
{
    if (qo_indptr[0] != 0)
        return -2;
    for (int b = 0; b < B; ++b) {
        int n = qo_indptr[b + 1] - qo_indptr[b], L = seq_lens[b];
        if (n < 0 || L < 1 || L > max_blocks * P || n > L)
            return -2;
    }
    return 0;
}

/* Steps 1-2 for every chunk token (row r of sequence b, index
 * t = L_b - n_b + (r - qo_indptr[b])): RMSNorm and NeoX RoPE at positions[r]
 * of its q rows and k rows, then slot t of sequence b receives bf16(k_rot)
 * (one round-to-nearest-even) and v (bits copied).
 *   q [T][Hq][D], k,v [T][Hkv][D], positions [T] (T = qo_indptr[B]);
 *   outputs q_rot [T][Hq][D], k_rot [T][Hkv][D] (double, unrounded). */
int oracle_prefill_append(int B, int Hq, int Hkv, int D, int P, int num_pages, int max_blocks,
                          const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          const uint16_t *w_q, const uint16_t *w_k, const int32_t *positions,
                          const int32_t *qo_indptr, const int32_t *seq_lens,
                          const int32_t *block_table, uint16_t *pool, double rope_theta,
                          double eps, double *q_rot, double *k_rot)
{
    if (Hkv < 1 || Hq % Hkv != 0 || D % 2 != 0)
        return -4;
    int rc = prefill_check(B, P, max_blocks, qo_indptr, seq_lens);
    if (rc)
        return rc;
    oracle_dims d = {B, Hq, Hkv, D, P, num_pages, max_blocks};
    double *x = (double *)malloc(sizeof(double) * (size_t)D);
    double *xn = (double *)malloc(sizeof(double) * (size_t)D);
    double *wq = (double *)malloc(sizeof(double) * (size_t)D);
    double *wk = (double *)malloc(sizeof(double) * (size_t)D);
    for (int i = 0; i < D; ++i) {
        wq[i] = oracle_bf16_to_double(w_q[i]);
        wk[i] = oracle_bf16_to_double(w_k[i]);
    }
    for (int b = 0; b < B && rc == 0; ++b) {
        int n = qo_indptr[b + 1] - qo_indptr[b], L = seq_lens[b];
        for (int j = 0; j < n && rc == 0; ++j) {
            int r = qo_indptr[b] + j, t = L - n + j;
            double pos = (double)positions[r];
            for (int h = 0; h < Hq; ++h) {
                long o = ((long)r * Hq + h) * D;
                for (int i = 0; i < D; ++i)
                    x[i] = oracle_bf16_to_double(q[o + i]);
                oracle_rmsnorm(x, wq, D, eps, xn);
                oracle_rope_neox(xn, D, pos, rope_theta, q_rot + o);
            }
            for (int h = 0; h < Hkv; ++h) {
                long o = ((long)r * Hkv + h) * D;
                for (int i = 0; i < D; ++i)
                    x[i] = oracle_bf16_to_double(k[o + i]);
                oracle_rmsnorm(x, wk, D, eps, xn);
                oracle_rope_neox(xn, D, pos, rope_theta, k_rot + o);
                long rk = pool_row(&d, block_table, b, t, 0, h);
                long rv = pool_row(&d, block_table, b, t, 1, h);
                if (rk < 0 || rv < 0) {
                    rc = -1;
                    break;
                }
                for (int i = 0; i < D; ++i) {
                    pool[rk + i] = oracle_double_to_bf16(k_rot[o + i]);
                    pool[rv + i] = v[o + i];
                }
            }
        }
    }
    free(x);
    free(xn);
    free(wq);
    free(wk);
    return rc;
}

/* Step 4 for the chunk: causal attention.  Query row r of sequence b (chunk
 * token at index t = L_b - n_b + (r - qo_indptr[b])) attends over tokens
 * 0..t of its sequence, i.e. attend_range(.., 0, t + 1) with its KV head
 * g = h / (Hq / Hkv) -- engine article, 4.4.1 (blockwise causal prefill
 * attention: a query block sees only keys at or before it; computed by
 * blocks it is exactly this softmax attention).
 *   q_rot [T][Hq][D] double; out [T][Hq][D]; lse [T][Hq]. */
int oracle_prefill_attention(int B, int Hq, int Hkv, int D, int P, int num_pages,
                             int max_blocks, const uint16_t *pool, const int32_t *block_table,
                             const int32_t *qo_indptr, const int32_t *seq_lens,
                             const double *q_rot, double scale, double *out, double *lse)
{
    if (Hkv < 1 || Hq % Hkv != 0)
        return -4;
    int rc = prefill_check(B, P, max_blocks, qo_indptr, seq_lens);
    if (rc)
        return rc;
    oracle_dims d = {B, Hq, Hkv, D, P, num_pages, max_blocks};
    int G = Hq / Hkv;
    for (int b = 0; b < B; ++b) {
        int n = qo_indptr[b + 1] - qo_indptr[b], L = seq_lens[b];
        for (int j = 0; j < n; ++j) {
            int r = qo_indptr[b] + j, t = L - n + j;
            for (int h = 0; h < Hq; ++h) {
                long o = ((long)r * Hq + h) * D;
                if (attend_range(&d, pool, block_table, b, h / G, q_rot + o, scale, 0, t + 1,
                                 out + o, lse + (long)r * Hq + h))
                    return -1;
            }
        }
    }
    return 0;
}

/* oracle_prefill_append with an FP8 pool: the same norm and rotation of every
 * chunk row; slot t of its sequence receives, for every element,
 *   K: RNE_e4m3_satfinite(fp32(bf16(k_rot)) / scale_K)
 *   V: RNE_e4m3_satfinite(fp32(v) / scale_V)
 * with the scales of the (page, plane, head) the slot lies in (inputs, read
 * only) -- the decode step's FP8 append applied to each chunk row. */
int oracle_prefill_append_fp8(int B, int Hq, int Hkv, int D, int P, int num_pages,
                              int max_blocks, const uint16_t *q, const uint16_t *k,
                              const uint16_t *v, const uint16_t *w_q, const uint16_t *w_k,
                              const int32_t *positions, const int32_t *qo_indptr,
                              const int32_t *seq_lens, const int32_t *block_table,
                              uint8_t *pool8, const float *kv_scale, double rope_theta,
                              double eps, double *q_rot, double *k_rot)
{
    if (Hkv < 1 || Hq % Hkv != 0 || D % 2 != 0)
        return -4;
    int rc = prefill_check(B, P, max_blocks, qo_indptr, seq_lens);
    if (rc)
        return rc;
    oracle_dims d = {B, Hq, Hkv, D, P, num_pages, max_blocks};
    double *x = (double *)malloc(sizeof(double) * (size_t)D);
    double *xn = (double *)malloc(sizeof(double) * (size_t)D);
    double *wq = (double *)malloc(sizeof(double) * (size_t)D);
    double *wk = (double *)malloc(sizeof(double) * (size_t)D);
    for (int i = 0; i < D; ++i) {
        wq[i] = oracle_bf16_to_double(w_q[i]);
        wk[i] = oracle_bf16_to_double(w_k[i]);
    }
    for (int b = 0; b < B && rc == 0; ++b) {
        int n = qo_indptr[b + 1] - qo_indptr[b], L = seq_lens[b];
        for (int j = 0; j < n && rc == 0; ++j) {
            int r = qo_indptr[b] + j, t = L - n + j;
            double pos = (double)positions[r];
            for (int h = 0; h < Hq; ++h) {
                long o = ((long)r * Hq + h) * D;
                for (int i = 0; i < D; ++i)
                    x[i] = oracle_bf16_to_double(q[o + i]);
                oracle_rmsnorm(x, wq, D, eps, xn);
                oracle_rope_neox(xn, D, pos, rope_theta, q_rot + o);
            }
            for (int h = 0; h < Hkv; ++h) {
                long o = ((long)r * Hkv + h) * D;
                for (int i = 0; i < D; ++i)
                    x[i] = oracle_bf16_to_double(k[o + i]);
                oracle_rmsnorm(x, wk, D, eps, xn);
                oracle_rope_neox(xn, D, pos, rope_theta, k_rot + o);
                long rk = pool_row(&d, block_table, b, t, 0, h);
                long rv = pool_row(&d, block_table, b, t, 1, h);
                long sk = scale_index(&d, block_table, b, t, 0, h);
                long sv = scale_index(&d, block_table, b, t, 1, h);
                if (rk < 0 || rv < 0 || sk < 0 || sv < 0) {
                    rc = -1;
                    break;
                }
                for (int i = 0; i < D; ++i) {
                    float kf = (float)oracle_bf16_to_double(oracle_double_to_bf16(k_rot[o + i]));
                    float vf = (float)oracle_bf16_to_double(v[o + i]);
                    pool8[rk + i] = oracle_float_to_e4m3_satfinite(kf / kv_scale[sk]);
                    pool8[rv + i] = oracle_float_to_e4m3_satfinite(vf / kv_scale[sv]);
                }
            }
        }
    }
    free(x);
    free(xn);
    free(wq);
    free(wk);
    return rc;
}

/* oracle_prefill_attention over an FP8 pool: query row r attends over tokens
 * 0..t of its sequence, the keys and values dequantized exactly. */
int oracle_prefill_attention_fp8(int B, int Hq, int Hkv, int D, int P, int num_pages,
                                 int max_blocks, const uint8_t *pool8, const float *kv_scale,
                                 const int32_t *block_table, const int32_t *qo_indptr,
                                 const int32_t *seq_lens, const double *q_rot, double scale,
                                 double *out, double *lse)
{
    if (Hkv < 1 || Hq % Hkv != 0)
        return -4;
    int rc = prefill_check(B, P, max_blocks, qo_indptr, seq_lens);
    if (rc)
        return rc;
    oracle_dims d = {B, Hq, Hkv, D, P, num_pages, max_blocks};
    int G = Hq / Hkv;
    for (int b = 0; b < B; ++b) {
        int n = qo_indptr[b + 1] - qo_indptr[b], L = seq_lens[b];
        for (int j = 0; j < n; ++j) {
            int r = qo_indptr[b] + j, t = L - n + j;
            for (int h = 0; h < Hq; ++h) {
                long o = ((long)r * Hq + h) * D;
                if (attend_range_fp8(&d, pool8, kv_scale, block_table, b, h / G, q_rot + o,
                                     scale, 0, t + 1, out + o, lse + (long)r * Hq + h))
                    return -1;
            }
        }
    }
    return 0;
}

/* oracle_qkv_append with an FP8 pool: the projection, norm and rotation as
 * above into the bf16 rows the bf16 pool would receive (bf16(k_rot),
 * bf16(v)), then for every element of slot seq_lens[b]-1
 *   code = RNE_e4m3_satfinite(fp32(bf16 row) / scale)
 * with the scales of the slot's (page, plane, head) -- the FP8 append rule
 * of the decode step.  kv_scale is read only. */
int oracle_qkv_append_fp8(int B, int Hq, int Hkv, int D, int P, int num_pages, int max_blocks,
                          int hidden, const uint16_t *x, const uint16_t *w_qkv,
                          const uint16_t *w_q, const uint16_t *w_k, const int32_t *positions,
                          const int32_t *seq_lens, const int32_t *block_table, uint8_t *pool8,
                          const float *kv_scale, double rope_theta, double eps, double *q_rot,
                          double *k_rot, double *v_out)
{
    oracle_dims d = {B, Hq, Hkv, D, P, num_pages, max_blocks};
    size_t n = (size_t)num_pages * 2 * (size_t)Hkv * (size_t)P * (size_t)D;
    uint16_t *rows = (uint16_t *)calloc(n, sizeof(uint16_t));
    int rc = oracle_qkv_append(B, Hq, Hkv, D, P, num_pages, max_blocks, hidden, x, w_qkv, w_q,
                               w_k, positions, seq_lens, block_table, rows, rope_theta, eps,
                               q_rot, k_rot, v_out);
    for (int b = 0; b < B && rc == 0; ++b) {
        int L = seq_lens[b];
        for (int g = 0; g < Hkv; ++g) {
            for (int kv = 0; kv < 2; ++kv) {
                long r = pool_row(&d, block_table, b, L - 1, kv, g);
                long si = scale_index(&d, block_table, b, L - 1, kv, g);
                if (r < 0 || si < 0) {
                    rc = -1;
                    break;
                }
                for (int i = 0; i < D; ++i)
                    pool8[r + i] = oracle_float_to_e4m3_satfinite(
                        (float)oracle_bf16_to_double(rows[r + i]) / kv_scale[si]);
            }
        }
    }
    free(rows);
    return rc;
}
