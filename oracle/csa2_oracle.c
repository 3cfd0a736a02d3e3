/*
 * csa2_oracle.c -- TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain, slow CPU statement of what the CSA2 decode path over an FP4 main
 * KV cache computes, in fp64, used only as the parity reference for the CUDA
 * library.  Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load it.  It shares no source, header, table or constant with the
 * CUDA library; it is compiled with plain gcc, no SIMD intrinsics, no
 * fast-math, and runs single-threaded.
 *
 * Sources (web pages about the DeepSeek-V4.1-Flash technical report):
 *  [ENG]  "DeepSeek-V4.1-Flash：把 KV Cache 压缩到极限的百万上下文 MoE",
 *         sections "架构三件套 / CSA2——条目×序列×层三维联合压缩",
 *         "Hierarchical Sparse Indexer——索引成本变常数" and
 *         "效率组件四件", item 4 "FP4 主 KV Cache".
 *  [HUNT] "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression",
 *         the summary paragraph on Compressed Sparse Attention 2 (CSA2).
 *  [55ZB] "552B参数干掉1.6T：DeepSeek V4.1 Flash技术深度解析", the CSA2
 *         paragraph (three static layer modes) and the DeepSelect paragraph.
 *
 * What the pages leave open is read as follows (each reading is marked
 * READING below): element formats follow the OCP FP8 E4M3 ("fn") and
 * E2M1 definitions the pages name; the indexer score is
 * sum_h w_h * ReLU(q_h . k) over 4 heads of dim 64 (the pages give no
 * formula); attention is MLA-style: K = all D channels, V = the first dv.
 *
 * Parity pins: every function here is pinned by tests under tests/ that
 * check it against closed forms, library routines or brute force.
 */
#include <fenv.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_EXPORT __attribute__((visibility("default")))

enum { ORC_BF16 = 0, ORC_FP8_E4M3 = 1, ORC_FP32 = 2 };
enum { ORC_FULL = 0, ORC_REINDEX = 1, ORC_REUSE = 2 };

/* Round to nearest integer, ties to even (the C library's default
 * rounding mode, checked by orc_rounding_mode_ok()). */
static double rne(double x) { return nearbyint(x); }

ORC_EXPORT int orc_rounding_mode_ok(void) { return fegetround() == FE_TONEAREST; }

/* ------------------------------------------------------------------ */
/* Element formats.  [ENG] "效率组件四件" item 4: the main KV cache holds   */
/* E2M1 values with one E4M3 scale per 16 channels, no global scale.  */
/* ------------------------------------------------------------------ */

/* OCP FP8 E4M3 ("fn"): 1 sign, 4 exponent bits (bias 7), 3 mantissa
 * bits, no infinities; S.1111.111 is NaN.  Subnormals are m * 2^-9. */
ORC_EXPORT double orc_e4m3_value(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xF;
    int m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* E2M1: 1 sign (bit 3), 2 exponent bits (bias 1), 1 mantissa bit.
 * Magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
ORC_EXPORT double orc_e2m1_value(uint8_t c)
{
    int sign = (c >> 3) & 1;
    int e = (c >> 1) & 3;
    int m = c & 1;
    double v;
    if (e == 0)
        v = 0.5 * m;
    else
        v = ldexp(1.0 + m / 2.0, e - 1);
    return sign ? -v : v;
}

/* Encode a non-negative real onto the E4M3 grid: round to nearest, ties to
 * the even mantissa, saturating to the largest finite value 448 (0x7E).
 * Works binade by binade as the format is defined. */
ORC_EXPORT uint8_t orc_e4m3_encode_pos(double a)
{
    int e2;
    double n;
    if (!(a > 0.0)) return 0x00;              /* zero (and the caller never passes NaN) */
    if (a >= 448.0) return 0x7E;              /* satfinite */
    if (a < ldexp(1.0, -6)) {
        /* subnormal binade: spacing 2^-9; n == 8 is the smallest normal */
        n = rne(a / ldexp(1.0, -9));
        return (uint8_t)n;                    /* codes 0..8, all consistent */
    }
    /* normal: a = f * 2^e2 with f in [0.5, 1) -> significand 2f in [1, 2) */
    (void)frexp(a, &e2);
    {
        int e = e2 - 1;                       /* a in [2^e, 2^(e+1)) */
        double sig = ldexp(a, -e);            /* in [1, 2) */
        int E;
        n = rne((sig - 1.0) * 8.0);           /* 0..8 */
        if (n == 8.0) { n = 0.0; e += 1; }
        E = e + 7;
        if (E > 15 || (E == 15 && n == 7.0)) return 0x7E;
        return (uint8_t)((E << 3) | (int)n);
    }
}

/* Encode a non-negative ratio r onto the E2M1 magnitudes: round to nearest,
 * ties to the even code, r > 6 saturates to code 7 (value 6). */
ORC_EXPORT uint8_t orc_e2m1_encode_mag(double r)
{
    if (!(r > 0.0)) return 0;
    if (r >= 6.0) return 7;
    if (r < 1.0) return (uint8_t)rne(r / 0.5);               /* 0,1,2      */
    if (r < 2.0) return (uint8_t)(2 + rne((r - 1.0) / 0.5)); /* 2,3,4      */
    if (r < 4.0) return (uint8_t)(4 + rne(r - 2.0));         /* 4,5,6      */
    return (uint8_t)(6 + rne((r - 4.0) / 2.0));              /* 6,7        */
}

/* bf16 bit pattern -> exact real value. */
static double bf16_value(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

ORC_EXPORT double orc_bf16_value(uint16_t h) { return bf16_value(h); }

static double elem_value(const void *base, int dt, int64_t i)
{
    if (dt == ORC_BF16) return bf16_value(((const uint16_t *)base)[i]);
    if (dt == ORC_FP8_E4M3) return orc_e4m3_value(((const uint8_t *)base)[i]);
    return (double)((const float *)base)[i];
}

/* ------------------------------------------------------------------ */
/* Step 1: quantise post-RoPE KV rows to FP4.                          */
/* [ENG] "效率组件四件" item 4 ("RoPE 后量化": quantise after RoPE);      */
/* [HUNT] CSA2 paragraph (E2M1, one E4M3 scale per 16 channels).      */
/* ------------------------------------------------------------------ */

/*
 * For row r and 16-channel group g (channels 16g .. 16g+15):
 *   amax  = max |x_c|                            (bf16 values, exact)
 *   s     = E4M3_RNE_sat(amax / 6)                READING: 6 is the largest
 *                                                 E2M1 magnitude, so amax
 *                                                 maps to the top of the grid
 *   code  = sign(x_c) << 3 | E2M1_RNE_sat(|x_c| / s)   (magnitude 0 if s == 0)
 * Codes are packed two per byte: channel 2i in the low nibble of byte i,
 * channel 2i+1 in the high nibble.  Output planes: codes [slots, D/2] and
 * scales [slots, D/16]; row r goes to slot dst_slot[r] (or r).
 * READING: the code's sign bit is the input's sign bit, also for values
 * that round to zero.  Returns 0, or -1 on a non-finite input or bad D.
 */
ORC_EXPORT int orc_quantize_kv_fp4(const uint16_t *kv, int64_t rows, int D, int64_t row_stride,
                                   const int64_t *dst_slot, uint8_t *codes, uint8_t *scales)
{
    int ngroups;
    int64_t r;
    if (D <= 0 || D % 16 != 0) return -1;
    ngroups = D / 16;
    for (r = 0; r < rows; ++r) {
        const uint16_t *x = kv + r * row_stride;
        int64_t slot = dst_slot ? dst_slot[r] : r;
        uint8_t *crow = codes + slot * (int64_t)(D / 2);
        uint8_t *srow = scales + slot * (int64_t)ngroups;
        int g, c;
        for (g = 0; g < ngroups; ++g) {
            double amax = 0.0, s;
            uint8_t sbyte;
            for (c = 16 * g; c < 16 * g + 16; ++c) {
                double v = bf16_value(x[c]);
                if (!isfinite(v)) return -1;
                if (fabs(v) > amax) amax = fabs(v);
            }
            sbyte = orc_e4m3_encode_pos(amax / 6.0);
            s = orc_e4m3_value(sbyte);
            srow[g] = sbyte;
            for (c = 16 * g; c < 16 * g + 16; ++c) {
                uint8_t sign = (x[c] >> 15) & 1;
                uint8_t mag = (s > 0.0) ? orc_e2m1_encode_mag(fabs(bf16_value(x[c])) / s) : 0;
                uint8_t code = (uint8_t)((sign << 3) | mag);
                if ((c & 1) == 0)
                    crow[c / 2] = code;
                else
                    crow[c / 2] |= (uint8_t)(code << 4);
            }
        }
    }
    return 0;
}

/*
 * RoPE on the append path, then the quantiser ("DeepSeek-V4.1-Flash：把 KV
 * Cache 压缩到极限的百万上下文 MoE", 效率组件四件 item 4: the FP4 main KV is
 * quantised after RoPE).  The pages fix neither the rotation layout nor how
 * the angles are evaluated; READING: interleaved pairs (2i, 2i+1) of the last
 * rope_dim channels, rotated by a caller-supplied fp32 table cos_sin[pos][i] =
 * (cos, sin), evaluated in fp32 without fused multiply-add:
 *     a' = (a*c) - (b*s),  b' = (a*s) + (b*c)   (every product and sum rounded to fp32)
 * then rounded to bf16 (nearest, ties to even).  Other channels pass through.
 * out_bits may alias nothing; returns 0, or -1 on a bad shape or position.
 */
static uint16_t f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)(u >> 16);   /* inf / NaN: truncate */
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

ORC_EXPORT int orc_rope_bf16(const uint16_t *kv, int64_t rows, int D, int64_t row_stride, const int32_t *pos,
                             const float *cos_sin, int64_t n_pos, int rope_dim, uint16_t *out)
{
    int64_t r;
    if (D <= 0 || rope_dim <= 0 || rope_dim > D || rope_dim % 2 != 0) return -1;
    for (r = 0; r < rows; ++r) {
        const uint16_t *x = kv + r * row_stride;
        uint16_t *y = out + r * (int64_t)D;
        const int64_t p = pos[r];
        int c, i;
        if (p < 0 || p >= n_pos) return -1;
        for (c = 0; c < D - rope_dim; ++c) y[c] = x[c];
        for (i = 0; i < rope_dim / 2; ++i) {
            const float cs = cos_sin[(p * (rope_dim / 2) + i) * 2];
            const float sn = cos_sin[(p * (rope_dim / 2) + i) * 2 + 1];
            const float a = bf16_to_f32(x[D - rope_dim + 2 * i]);
            const float b = bf16_to_f32(x[D - rope_dim + 2 * i + 1]);
            const float ac = a * cs, bs = b * sn, as = a * sn, bc = b * cs;
            const float ra = ac - bs, rb = as + bc;
            y[D - rope_dim + 2 * i] = f32_to_bf16_rne(ra);
            y[D - rope_dim + 2 * i + 1] = f32_to_bf16_rne(rb);
        }
    }
    return 0;
}

/* Dequantised value of channel c of a stored entry (codes row, scales row). */
static double fp4_value(const uint8_t *crow, const uint8_t *srow, int c)
{
    uint8_t byte = crow[c / 2];
    uint8_t code = (c & 1) ? (byte >> 4) : (byte & 0xF);
    return orc_e2m1_value(code) * orc_e4m3_value(srow[c / 16]);
}

ORC_EXPORT void orc_dequant_fp4(const uint8_t *codes, const uint8_t *scales, int64_t rows, int D,
                                double *out)
{
    int64_t r;
    int c;
    for (r = 0; r < rows; ++r)
        for (c = 0; c < D; ++c)
            out[r * D + c] = fp4_value(codes + r * (D / 2), scales + r * (D / 16), c);
}

/* ------------------------------------------------------------------ */
/* Step 2: indexer scores.                                             */
/* The pages give no indexer formula.  READING: the lightning-indexer  */
/* form score = sum_{h<4} w_h * ReLU(sum_{d<64} q_hd * k_d), one 64-dim */
/* key per compressed entry shared by the 4 indexer heads, no scaling. */
/* Full mode scores every entry j < kv_len; Reindex mode scores only   */
/* the candidates 8*pool[p] + i of the hierarchical pool, using the    */
/* source layer's keys with this layer's own q and w                   */
/* ([ENG] "Hierarchical Sparse Indexer"; [HUNT] CSA2 paragraph).        */
/* Masked or invalid candidates score -inf.                            */
/* ------------------------------------------------------------------ */

#define ORC_IDX_HEADS 4
#define ORC_IDX_DIM 64

static void score_one(const void *q, int q_dt, int64_t qoff, const float *w, int64_t woff,
                      const void *k, int k_dt, int64_t koff, double *score, double *mag)
{
    double s = 0.0, m = 0.0;
    int h, d;
    for (h = 0; h < ORC_IDX_HEADS; ++h) {
        double dot = 0.0, adot = 0.0;
        for (d = 0; d < ORC_IDX_DIM; ++d) {
            double qv = elem_value(q, q_dt, qoff + h * ORC_IDX_DIM + d);
            double kv = elem_value(k, k_dt, koff + d);
            dot += qv * kv;
            adot += fabs(qv * kv);
        }
        s += (double)w[woff + h] * (dot > 0.0 ? dot : 0.0);
        m += fabs((double)w[woff + h]) * adot;
    }
    *score = s;
    if (mag) *mag = m;
}

/*
 * q: [B, T, 4, 64] (bf16 or fp8), w: fp32 [B, T, 4], k: [B, N, 64],
 * kv_len: int32 [B*T].  FULL: out [B, T, N].  REINDEX: pool int32
 * [B, T, P], out [B, T, 8P] in pool-local order l = 8p + i.
 * mag (nullable) receives sum_h |w_h| sum_d |q_hd k_d| per output, the
 * conditioning of the score used by the tolerance.
 */
ORC_EXPORT int orc_index_score(int mode, int B, int T, int64_t N, const void *q, int q_dt,
                               const float *w, const void *k, int k_dt, const int32_t *kv_len,
                               const int32_t *pool, int P, double *out, double *mag)
{
    int b, t;
    if (mode == ORC_REUSE) return 0;
    if (mode == ORC_REINDEX && !pool) return -1;
    for (b = 0; b < B; ++b) {
        for (t = 0; t < T; ++t) {
            int64_t bt = (int64_t)b * T + t;
            int64_t len = kv_len[bt] < N ? kv_len[bt] : N;
            int64_t qoff = bt * ORC_IDX_HEADS * ORC_IDX_DIM;
            int64_t woff = bt * ORC_IDX_HEADS;
            if (mode == ORC_FULL) {
                int64_t j;
                for (j = 0; j < N; ++j) {
                    double *o = out + bt * N + j;
                    double *mg = mag ? mag + bt * N + j : NULL;
                    if (j < len)
                        score_one(q, q_dt, qoff, w, woff, k, k_dt, ((int64_t)b * N + j) * ORC_IDX_DIM, o, mg);
                    else {
                        *o = -INFINITY;
                        if (mg) *mg = 0.0;
                    }
                }
            } else {
                int p, i;
                for (p = 0; p < P; ++p) {
                    int32_t blk = pool[bt * P + p];
                    for (i = 0; i < 8; ++i) {
                        int64_t l = (int64_t)p * 8 + i;
                        int64_t j = (int64_t)blk * 8 + i;
                        double *o = out + bt * (int64_t)P * 8 + l;
                        double *mg = mag ? mag + bt * (int64_t)P * 8 + l : NULL;
                        if (blk >= 0 && j < len)
                            score_one(q, q_dt, qoff, w, woff, k, k_dt, ((int64_t)b * N + j) * ORC_IDX_DIM, o, mg);
                        else {
                            *o = -INFINITY;
                            if (mg) *mg = 0.0;
                        }
                    }
                }
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Selection: the K largest finite values of a row.                    */
/* READING: ties go to the lower position; -inf is never selected; if   */
/* fewer than K candidates are finite, all of them are returned and the */
/* rest of the output is -1.  The output is in descending score order.  */
/* ------------------------------------------------------------------ */

typedef struct { double v; int64_t i; } vi_t;

static int cmp_desc(const void *a, const void *b)
{
    const vi_t *x = (const vi_t *)a, *y = (const vi_t *)b;
    if (x->v > y->v) return -1;
    if (x->v < y->v) return 1;
    return (x->i < y->i) ? -1 : (x->i > y->i);
}

/* Returns the number selected, writes candidate indices to out[0..K). */
static int64_t select_topk(const double *v, int64_t M, int64_t K, int64_t *out)
{
    vi_t *buf = (vi_t *)malloc((size_t)(M > 0 ? M : 1) * sizeof(vi_t));
    int64_t n = 0, i;
    if (!buf) return -1;
    for (i = 0; i < M; ++i)
        if (v[i] > -INFINITY) { buf[n].v = v[i]; buf[n].i = i; ++n; }
    qsort(buf, (size_t)n, sizeof(vi_t), cmp_desc);
    for (i = 0; i < K; ++i) out[i] = (i < n) ? buf[i].i : -1;
    free(buf);
    return n < K ? n : K;
}

/*
 * Step 3: the hierarchical candidate pool ([ENG] "Hierarchical Sparse
 * Indexer": at most 2048 blocks of 8 positions).  READING: a block is
 * the aligned run of G = 8 positions [8*beta, 8*beta + 8); its score is
 * the max over its valid positions (j < kv_len); the pool is the
 * Top-min(P, #blocks with a finite score) blocks.
 * scores: fp32 [B, T, N]; out: int32 [B, T, P] block ids, -1 padded.
 */
ORC_EXPORT int orc_build_pool(int B, int T, int64_t N, const float *scores, const int32_t *kv_len,
                              int P, int G, int32_t *out)
{
    int64_t nbmax = (N + G - 1) / G;
    double *bs = (double *)malloc((size_t)(nbmax > 0 ? nbmax : 1) * sizeof(double));
    int64_t *sel = (int64_t *)malloc((size_t)(P > 0 ? P : 1) * sizeof(int64_t));
    int64_t bt;
    if (!bs || !sel) { free(bs); free(sel); return -1; }
    for (bt = 0; bt < (int64_t)B * T; ++bt) {
        int64_t len = kv_len[bt] < N ? kv_len[bt] : N;
        int64_t beta, j;
        int p;
        for (beta = 0; beta < nbmax; ++beta) {
            double m = -INFINITY;
            for (j = beta * G; j < beta * G + G && j < len; ++j) {
                double v = (double)scores[bt * N + j];
                if (v > m) m = v;
            }
            bs[beta] = m;
        }
        if (select_topk(bs, nbmax, P, sel) < 0) { free(bs); free(sel); return -1; }
        for (p = 0; p < P; ++p) out[bt * P + p] = (int32_t)sel[p];
    }
    free(bs);
    free(sel);
    return 0;
}

/*
 * Step 4: Top-K selection ([ENG] CSA2 section: Top-512; [55ZB]
 * DeepSelect paragraph names it the sparse attention's Top-K kernel).
 * FULL: candidates are positions j < min(kv_len, M) of scores [B, T, M].
 * REINDEX: candidates are pool-local l = 8p + i of scores [B, T, 8P];
 * a selected l is reported as the global position 8*pool[p] + i.
 * REUSE: no work, idx untouched (the layer reuses its source's indices).
 * out idx: int32 [B, T, K], -1 padded, descending score order.
 */
ORC_EXPORT int orc_topk(int mode, int B, int T, int64_t M, const float *scores,
                        const int32_t *kv_len, const int32_t *pool, int P, int K, int32_t *idx)
{
    double *v;
    int64_t *sel, bt;
    if (mode == ORC_REUSE) return 0;
    if (mode == ORC_REINDEX && (!pool || M != (int64_t)P * 8)) return -1;
    v = (double *)malloc((size_t)(M > 0 ? M : 1) * sizeof(double));
    sel = (int64_t *)malloc((size_t)(K > 0 ? K : 1) * sizeof(int64_t));
    if (!v || !sel) { free(v); free(sel); return -1; }
    for (bt = 0; bt < (int64_t)B * T; ++bt) {
        int64_t j;
        int s;
        for (j = 0; j < M; ++j) {
            double x = (double)scores[bt * M + j];
            if (mode == ORC_FULL) {
                int64_t len = kv_len ? kv_len[bt] : M;
                if (j >= len) x = -INFINITY;
            } else if (pool[bt * P + j / 8] < 0) {
                x = -INFINITY;
            }
            v[j] = x;
        }
        select_topk(v, M, K, sel);
        for (s = 0; s < K; ++s) {
            int64_t l = sel[s];
            if (l < 0)
                idx[bt * K + s] = -1;
            else if (mode == ORC_FULL)
                idx[bt * K + s] = (int32_t)l;
            else
                idx[bt * K + s] = (int32_t)((int64_t)pool[bt * P + l / 8] * 8 + l % 8);
        }
    }
    free(v);
    free(sel);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Step 5: sparse attention over the selected FP4 entries.             */
/* READING (MLA-style, the pages give no formula): for query row       */
/* (b, t, h), with the valid selected entries J (idx != -1):           */
/*   z_j = sm_scale * sum_{c<D} q[c] * Khat[j][c]                       */
/*   lse = log sum_j exp(z_j),  o[c] = sum_j exp(z_j - lse) Khat[j][c]  */
/* for c < dv (V is the first dv channels of the same entry).          */
/* Khat is the dequantised entry.  An empty J gives o = 0, lse = -inf. */
/* Reuse layers call this with their source layer's idx unchanged      */
/* ([ENG] CSA2 section; [55ZB] CSA2 paragraph).                         */
/* Returns the number of out-of-range indices seen (they are skipped).  */
/* ------------------------------------------------------------------ */
ORC_EXPORT int64_t orc_sparse_attn(int B, int T, int H, int D, int dv, const uint16_t *q,
                                   const uint8_t *codes, const uint8_t *scales, int64_t N,
                                   const int32_t *idx, int K, const int32_t *kv_len,
                                   double sm_scale, double *out, double *lse)
{
    double *kh = (double *)malloc((size_t)(K > 0 ? K : 1) * (size_t)D * sizeof(double));
    double *z = (double *)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
    int64_t bad = 0, bt;
    if (!kh || !z) { free(kh); free(z); return -1; }
    for (bt = 0; bt < (int64_t)B * T; ++bt) {
        int64_t b = bt / T;
        int64_t len = kv_len ? (kv_len[bt] < N ? kv_len[bt] : N) : N;
        int nv = 0, s, h, c;
        /* dequantise the valid selected entries of this query token */
        for (s = 0; s < K; ++s) {
            int64_t j = idx[bt * K + s];
            if (j == -1) continue;
            if (j < 0 || j >= len) { ++bad; continue; }
            for (c = 0; c < D; ++c)
                kh[(int64_t)nv * D + c] = fp4_value(codes + (b * N + j) * (D / 2),
                                                    scales + (b * N + j) * (D / 16), c);
            ++nv;
        }
        for (h = 0; h < H; ++h) {
            const uint16_t *qr = q + (bt * H + h) * (int64_t)D;
            double *o = out + (bt * H + h) * (int64_t)dv;
            double m = -INFINITY, sum = 0.0, l;
            int i;
            for (c = 0; c < dv; ++c) o[c] = 0.0;
            if (nv == 0) {
                if (lse) lse[bt * H + h] = -INFINITY;
                continue;
            }
            for (i = 0; i < nv; ++i) {
                double acc = 0.0;
                for (c = 0; c < D; ++c) acc += bf16_value(qr[c]) * kh[(int64_t)i * D + c];
                z[i] = sm_scale * acc;
                if (z[i] > m) m = z[i];
            }
            for (i = 0; i < nv; ++i) sum += exp(z[i] - m);
            l = m + log(sum);
            for (i = 0; i < nv; ++i) {
                double p = exp(z[i] - l);
                for (c = 0; c < dv; ++c) o[c] += p * kh[(int64_t)i * D + c];
            }
            if (lse) lse[bt * H + h] = l;
        }
    }
    free(kh);
    free(z);
    return bad;
}

/*
 * Sliding-window branch with FP8 KV, merged with the sparse branch by
 * log-sum-exp.  "DeepSeek-V4.1-Flash：把 KV Cache 压缩到极限的百万上下文 MoE",
 * 效率组件四件 item 4 (SWA KV stays FP8) and "DeepSeek-V4.1-Flash: Pushing the
 * Limits of KV Cache Compression" (every layer also has a sliding window).
 * READINGS (the pages give neither the window size nor the FP8 layout): the
 * window KV is E4M3 rows [B, W, D] without a scale (like the indexer keys),
 * K = all D channels and V = the first dv (MLA-style, as the sparse branch);
 * query row (b, t) attends to the first swa_len[b*T+t] (<= W) rows of b's
 * window, all visible; the two branches cover disjoint entries, so the merge
 * is the softmax over their union:
 *     M = max(lse_w, lse_s),  a = e^(lse_w - M),  c = e^(lse_s - M),
 *     out = (a o_w + c o_s) / (a + c),  lse = M + log(a + c).
 * o_sparse / lse_sparse NULL: the window branch alone.  Empty window and
 * lse_s = -inf both: out = 0, lse = -inf.
 */
ORC_EXPORT int orc_swa_attn_merge(int B, int T, int H, int D, int dv, const uint16_t *q, const uint8_t *kv, int W,
                                  const int32_t *swa_len, double sm_scale, const double *o_sparse,
                                  const double *lse_sparse, double *out, double *lse)
{
    double *z = (double *)malloc((size_t)(W > 0 ? W : 1) * sizeof(double));
    double *ow = (double *)malloc((size_t)(dv > 0 ? dv : 1) * sizeof(double));
    int64_t bt;
    if (!z || !ow) { free(z); free(ow); return -1; }
    for (bt = 0; bt < (int64_t)B * T; ++bt) {
        const int64_t b = bt / T;
        int n = swa_len[bt] < W ? swa_len[bt] : W, h, c, i;
        if (n < 0) n = 0;
        for (h = 0; h < H; ++h) {
            const uint16_t *qr = q + (bt * H + h) * (int64_t)D;
            double *o = out + (bt * H + h) * (int64_t)dv;
            double m = -INFINITY, sum = 0.0, lw = -INFINITY, ls, M;
            for (c = 0; c < dv; ++c) ow[c] = 0.0;
            for (i = 0; i < n; ++i) {
                const uint8_t *kr = kv + (b * W + i) * (int64_t)D;
                double acc = 0.0;
                for (c = 0; c < D; ++c) acc += bf16_value(qr[c]) * orc_e4m3_value(kr[c]);
                z[i] = sm_scale * acc;
                if (z[i] > m) m = z[i];
            }
            if (n > 0) {
                for (i = 0; i < n; ++i) sum += exp(z[i] - m);
                lw = m + log(sum);
                for (i = 0; i < n; ++i) {
                    const uint8_t *kr = kv + (b * W + i) * (int64_t)D;
                    const double p = exp(z[i] - lw);
                    for (c = 0; c < dv; ++c) ow[c] += p * orc_e4m3_value(kr[c]);
                }
            }
            ls = lse_sparse ? lse_sparse[bt * H + h] : -INFINITY;
            M = lw > ls ? lw : ls;
            if (M == -INFINITY) {
                for (c = 0; c < dv; ++c) o[c] = 0.0;
                if (lse) lse[bt * H + h] = -INFINITY;
                continue;
            }
            {
                const double a = exp(lw - M), cs = exp(ls - M);
                for (c = 0; c < dv; ++c) {
                    const double os = o_sparse ? o_sparse[(bt * H + h) * (int64_t)dv + c] : 0.0;
                    o[c] = (a * ow[c] + cs * os) / (a + cs);
                }
                if (lse) lse[bt * H + h] = M + log(a + cs);
            }
        }
    }
    free(z);
    free(ow);
    return 0;
}
