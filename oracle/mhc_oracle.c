/*
 * CPU oracle of the mHC layer boundary (n_hc = 4): TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
 * arm may load this library. The CUDA path never calls it, and it shares no
 * code, header, table or helper with the CUDA path.
 *
 * Plain, slow, single-threaded C. Every step follows the per-token math of
 * two pages, in their order and at their rounding points:
 *   [B] "vllm.models.deepseek_v41.nvidia.ops.mhc_boundary" (DeepSeek-V4.1
 *       shifted mHC boundary), functions residual_update, lagged_collapse,
 *       prepare_boundary_weight, MhcBoundaryKernel.coefficients / sinkhorn /
 *       col_normalize / layer_input_words, sigmoid and rcp.
 *   [P] "The Hyper Connection Preprocessing GPU Kernel Study" (FlashInfer
 *       mhc_pre_big_fuse), sections "square sum and RMSNorm", "computing A_l",
 *       "computing C_l", "computing B_l" and "computing layer_input".
 * Where the pages leave an accumulation order open (the 4H-long sum of
 * squares, the 24 x 4H mixer contraction, the H-long sum of squares of the
 * collapse) the oracle sums in double, so that it stands for the exact value
 * rounded once. Build with -ffp-contract=off and without -ffast-math: every
 * fused multiply-add below is an explicit fmaf(), every other operation is
 * rounded on its own.
 *
 * Parity status per function is stated in tests/test_oracle_pins.py; every
 * function here has at least one pin there.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>

#define NHC 4
#define MIXES 24

typedef struct {
    float hc_norm_eps;   /* eps of the 4H RMS (rstd) */
    float hc_pre_eps;    /* floor added to pre */
    float hc_post_mult;  /* post multiplier (2) */
    float sinkhorn_eps;  /* eps of softmax floor and Sinkhorn denominators */
    float norm_eps;      /* eps of the layer RMSNorm of the collapse */
    int sinkhorn_iters;  /* >= 1 */
} oracle_params;

/* ---- scalar helpers (bit-level definitions) ---------------------------- */

static uint32_t bits_of(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float float_of(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* bf16 -> fp32 is exact: the bf16 pattern is the top half of the fp32 one. */
static float bf16_to_f32(uint16_t h) { return float_of((uint32_t)h << 16); }

/* fp32 -> bf16, round to nearest, ties to even (NaN inputs are excluded). */
static uint16_t f32_to_bf16(float f)
{
    uint32_t u = bits_of(f);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* Flush-to-zero of one value: subnormal -> zero of the same sign. */
static float ftz(float f)
{
    if (f != 0.0f && fabsf(f) < 0x1p-126f) return copysignf(0.0f, f);
    return f;
}

/* TF32 rounding of [B] prepare_boundary_weight: add half an ulp of the
 * 10-bit mantissa to the bit pattern and clear the 13 low bits, i.e. round
 * to nearest with ties away from zero on the magnitude. */
static float tf32_round(float w)
{
    return float_of((bits_of(w) + 0x1000u) & 0xFFFFE000u);
}

/* [B] rcp: the IEEE round-to-nearest reciprocal of a normal input. */
static float rcp(float x) { return 1.0f / x; }

/* [B] sigmoid: 1 / min(1 + exp(-v), 2^126). */
static float sigmoid(float v)
{
    return rcp(fminf(1.0f + expf(-v), 0x1p126f));
}

/* ---- weight preparation ----------------------------------------------- */

/* TF32 round and exact BF16 hi/lo split of n weights ([B]
 * prepare_boundary_weight): r = tf32(w), hi = bf16(r), lo = bf16(r - hi). */
void oracle_tf32_split(const float *w, int64_t n, float *rounded,
                       uint16_t *hi, uint16_t *lo)
{
    for (int64_t i = 0; i < n; ++i) {
        float r = tf32_round(w[i]);
        uint16_t h = f32_to_bf16(r);
        float rest = r - bf16_to_f32(h);
        if (rounded) rounded[i] = r;
        if (hi) hi[i] = h;
        if (lo) lo[i] = f32_to_bf16(rest);
    }
}

/* The library's prepared-weight layout, written out as nested loops from
 * its definition in include/mhc.h: for hidden chunk c (32 wide), stream s,
 * stacked row r (0-23 the hi parts of mixes 0-23, 24-47 their lo parts) and
 * element e of the chunk, the bf16 value of column k = s*H + 32c + e sits at
 *   ((c*4 + s)*48 + r)*32 + 8*((e/8) ^ ((r/2) % 4)) + e%8
 * (uint16 units): 64-byte rows with the 64-byte swizzle applied.
 * fn is [24][4H] fp32, out has 48*4H uint16 entries. */
void oracle_weight_tiles(const float *fn, int H, uint16_t *out)
{
    const int64_t K = (int64_t)NHC * H;
    for (int c = 0; c < H / 32; ++c)
        for (int s = 0; s < NHC; ++s)
            for (int r = 0; r < 2 * MIXES; ++r)
                for (int e = 0; e < 32; ++e) {
                    int n = r % MIXES;
                    int64_t k = (int64_t)s * H + 32 * c + e;
                    float rr = tf32_round(fn[n * K + k]);
                    uint16_t h = f32_to_bf16(rr);
                    uint16_t v = (r < MIXES) ? h
                                             : f32_to_bf16(rr - bf16_to_f32(h));
                    int64_t at = ((int64_t)(c * NHC + s) * 2 * MIXES + r) * 32
                                 + 8 * ((e / 8) ^ ((r / 2) % 4)) + e % 8;
                    out[at] = v;
                }
}

/* ---- residual update (post) -------------------------------------------- */

/* [B] residual_update for one token: for stream s and hidden h,
 *   cur[s][h] = bf16( ftz chain: post[s]*x[h], then + comb[j][s]*res[j][h]
 *                     for j = 0..3 as fused multiply-adds ),
 * every input and result of the chain flushed to zero when subnormal. */
static void residual_update_token(const uint16_t *x, const uint16_t *res,
                                  const float *post, const float *comb, int H,
                                  uint16_t *cur)
{
    for (int s = 0; s < NHC; ++s) {
        float ps = ftz(post[s]);
        for (int h = 0; h < H; ++h) {
            float nu = ftz(ps * ftz(bf16_to_f32(x[h])));
            for (int j = 0; j < NHC; ++j) {
                float c = ftz(comb[j * NHC + s]);
                float r = ftz(bf16_to_f32(res[(int64_t)j * H + h]));
                nu = ftz(fmaf(c, r, nu));
            }
            cur[(int64_t)s * H + h] = f32_to_bf16(nu);
        }
    }
}

void oracle_post(const uint16_t *x, const uint16_t *residual, const float *post,
                 const float *comb, int64_t T, int H, uint16_t *residual_out)
{
    for (int64_t t = 0; t < T; ++t)
        residual_update_token(x + t * H, residual + t * NHC * H, post + t * NHC,
                              comb + t * NHC * NHC, H,
                              residual_out + t * NHC * H);
}

/* ---- coefficients ------------------------------------------------------ */

/* [B] col_normalize: column sums (c0k + c1k) + (c2k + c3k), plus eps, and a
 * multiply by the reciprocal. */
static void col_normalize(float *c, float eps)
{
    for (int k = 0; k < NHC; ++k) {
        float inv = rcp(((c[k] + c[4 + k]) + (c[8 + k] + c[12 + k])) + eps);
        for (int i = 0; i < NHC; ++i) c[4 * i + k] = c[4 * i + k] * inv;
    }
}

/* [B] sinkhorn: one column normalisation, then iters - 1 times a row
 * normalisation (((c0 + c1) + c2) + c3 + eps) followed by a column one. */
static void sinkhorn(float *c, int iters, float eps)
{
    col_normalize(c, eps);
    for (int it = 1; it < iters; ++it) {
        for (int i = 0; i < NHC; ++i) {
            float rinv = rcp((((c[4 * i] + c[4 * i + 1]) + c[4 * i + 2])
                              + c[4 * i + 3]) + eps);
            for (int k = 0; k < NHC; ++k) c[4 * i + k] = c[4 * i + k] * rinv;
        }
        col_normalize(c, eps);
    }
}

/* [B] MhcBoundaryKernel.coefficients (same order as [P] "computing A_l",
 * "computing C_l", "computing B_l"): from the 24 mixes and rstd,
 *   pre[i]  = sigmoid(fma(mix[i]*rstd, scale[0], base[i])) + hc_pre_eps
 *   post[i] = sigmoid(fma(mix[4+i]*rstd, scale[1], base[4+i])) * post_mult
 *   comb    = sinkhorn(row softmax of fma(mix[8+4i+k]*rstd, scale[2], base)
 *                      with fma(e, rcp(sum e), eps)). */
static void coefficients(const float *mix, float rstd, const float *scale,
                         const float *base, const oracle_params *p,
                         float *pre, float *post, float *comb)
{
    for (int i = 0; i < NHC; ++i) {
        float v = fmaf(mix[i] * rstd, scale[0], base[i]);
        pre[i] = sigmoid(v) + p->hc_pre_eps;
    }
    for (int i = 0; i < NHC; ++i) {
        float v = fmaf(mix[NHC + i] * rstd, scale[1], base[NHC + i]);
        post[i] = sigmoid(v) * p->hc_post_mult;
    }
    float c[NHC * NHC];
    for (int i = 0; i < NHC; ++i) {
        float l[NHC];
        for (int k = 0; k < NHC; ++k) {
            int n = 2 * NHC + NHC * i + k;
            l[k] = fmaf(mix[n] * rstd, scale[2], base[n]);
        }
        float m = fmaxf(fmaxf(l[0], l[1]), fmaxf(l[2], l[3]));
        float e[NHC];
        for (int k = 0; k < NHC; ++k) e[k] = expf(l[k] - m);
        float inv = rcp(((e[0] + e[1]) + e[2]) + e[3]);
        for (int k = 0; k < NHC; ++k)
            c[NHC * i + k] = fmaf(e[k], inv, p->sinkhorn_eps);
    }
    sinkhorn(c, p->sinkhorn_iters, p->sinkhorn_eps);
    memcpy(comb, c, sizeof c);
}

/* ---- collapse and layer RMSNorm ------------------------------------------ */

/* One token: li[h] = bf16(fma chain over j from 0 of pc[j] * cur[j][h]), not
 * flushed ([B] lagged_collapse; [P] "computing layer_input"), then the RMSNorm
 * over H ([B] layer_input_words): out = bf16((li * rstd_li) * norm_w), or li
 * itself without norm_w. Returns rstd_li. li is scratch of H values. */
static float collapse_norm(const uint16_t *cur, const float *pc, const void *norm_w,
                           int nw_bf16, const oracle_params *p, int H, uint16_t *li,
                           uint16_t *out)
{
    for (int h = 0; h < H; ++h) {
        float acc = 0.0f;
        for (int j = 0; j < NHC; ++j)
            acc = fmaf(pc[j], bf16_to_f32(cur[(int64_t)j * H + h]), acc);
        li[h] = f32_to_bf16(acc);
    }
    double ssq_li = 0.0;
    for (int h = 0; h < H; ++h) {
        double v = bf16_to_f32(li[h]);
        ssq_li += v * v;
    }
    float rstd_li = (float)(1.0 / sqrt(ssq_li / (double)H + (double)p->norm_eps));
    if (out) {
        for (int h = 0; h < H; ++h) {
            if (!norm_w) { out[h] = li[h]; continue; }
            float w = nw_bf16 ? bf16_to_f32(((const uint16_t *)norm_w)[h])
                              : ((const float *)norm_w)[h];
            float a = bf16_to_f32(li[h]) * rstd_li;
            out[h] = f32_to_bf16(a * w);
        }
    }
    return rstd_li;
}

/* ---- the boundary ------------------------------------------------------- */

enum { ORACLE_PRE_ONLY = 0, ORACLE_FUSED_UNSHIFTED = 1, ORACLE_FUSED_SHIFTED = 2 };

/*
 * One boundary over T tokens.
 *   mode 0 (pre only, [P] mhc_pre_big_fuse with prenorm): the residual is the
 *          stream; no update, no x/post/comb/pre_lag.
 *   mode 1 (fused, unshifted): update, then this boundary's own pre collapses.
 *   mode 2 (fused, shifted, [B] mhc_shifted_post_pre_boundary): update, and
 *          the collapse uses the previous boundary's pre (pre_lag).
 * fn is the fp32 mixer [24][4H]; norm_w is NULL (layer input = collapse) or
 * [H] of fp32 (nw_bf16 = 0) or bf16 (nw_bf16 = 1).
 * Outputs (any may be NULL): residual_out [T][4][H] (modes 1, 2),
 * layer_input [T][H], pre/post [T][4], comb [T][4][4]; diagnostics mix
 * [T][24], mix_scale [T][24] = sqrt(sum_k (w_k x_k)^2), rstd [T], rstd_li [T].
 */
void oracle_boundary(int mode, const uint16_t *x, const uint16_t *residual,
                     const float *post_in, const float *comb_in,
                     const float *pre_lag, const float *fn, const float *scale,
                     const float *base, const void *norm_w, int nw_bf16,
                     const oracle_params *p, int64_t T, int H,
                     uint16_t *residual_out, uint16_t *layer_input,
                     float *pre_out, float *post_out, float *comb_out,
                     float *mix_out, float *mix_scale_out, float *rstd_out,
                     float *rstd_li_out)
{
    const int64_t K = (int64_t)NHC * H;
    float *r = (float *)malloc(sizeof(float) * MIXES * K);
    uint16_t *cur = (uint16_t *)malloc(sizeof(uint16_t) * K);
    uint16_t *li = (uint16_t *)malloc(sizeof(uint16_t) * H);
    if (!r || !cur || !li) { free(r); free(cur); free(li); return; }
    /* the mixer as the tensor cores see it: TF32-rounded ([B]
     * prepare_boundary_weight); hi + lo reproduces r exactly */
    for (int64_t i = 0; i < MIXES * K; ++i) r[i] = tf32_round(fn[i]);

    for (int64_t t = 0; t < T; ++t) {
        /* 1. updated residual ([B] residual_update), or the residual itself */
        if (mode == ORACLE_PRE_ONLY)
            memcpy(cur, residual + t * K, sizeof(uint16_t) * K);
        else
            residual_update_token(x + t * H, residual + t * K, post_in + t * NHC,
                                  comb_in + t * NHC * NHC, H, cur);
        if (residual_out && mode != ORACLE_PRE_ONLY)
            memcpy(residual_out + t * K, cur, sizeof(uint16_t) * K);

        /* 2. sum of squares over the flattened 4H and rstd ([P] "square sum
         *    and RMSNorm"; [B] coefficients) */
        double ssq = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double v = bf16_to_f32(cur[k]);
            ssq += v * v;
        }
        float rstd = (float)(1.0 / sqrt(ssq / (double)K + (double)p->hc_norm_eps));

        /* 3. mixer contraction mix[n] = sum_k tf32(fn[n][k]) * cur_flat[k],
         *    cur_flat[s*H + h] = cur[s][h]; every product is exact in double */
        float mix[MIXES];
        for (int n = 0; n < MIXES; ++n) {
            double acc = 0.0, sq = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double term = (double)r[n * K + k] * (double)bf16_to_f32(cur[k]);
                acc += term;
                sq += term * term;
            }
            mix[n] = (float)acc;
            if (mix_out) mix_out[t * MIXES + n] = mix[n];
            if (mix_scale_out) mix_scale_out[t * MIXES + n] = (float)sqrt(sq);
        }
        if (rstd_out) rstd_out[t] = rstd;

        /* 4-6. pre, post, softmax + Sinkhorn comb */
        float pre[NHC], post[NHC], comb[NHC * NHC];
        coefficients(mix, rstd, scale, base, p, pre, post, comb);
        if (pre_out) memcpy(pre_out + t * NHC, pre, sizeof pre);
        if (post_out) memcpy(post_out + t * NHC, post, sizeof post);
        if (comb_out) memcpy(comb_out + t * NHC * NHC, comb, sizeof comb);

        /* 7-8. collapse and layer RMSNorm */
        const float *pc = (mode == ORACLE_FUSED_SHIFTED) ? pre_lag + t * NHC : pre;
        float rstd_li = collapse_norm(cur, pc, norm_w, nw_bf16, p, H, li,
                                      layer_input ? layer_input + t * H : NULL);
        if (rstd_li_out) rstd_li_out[t] = rstd_li;
    }
    free(r);
    free(cur);
    free(li);
}

/*
 * Pre from split-K mixes ([P] "square sum and RMSNorm", path 1 with split-K,
 * and "explaining split-K"): the previous GEMM split the 4H-long contraction
 * into S parts and left its partial mixes dot_mix [S][T][24] and partial sums
 * of squares of the flattened residual sqrsum [S][T]. Here
 *   mix[t][n] = sum over s of dot_mix[s][t][n]   (summed in double, rounded once)
 *   ssq[t]    = sum over s of sqrsum[s][t]       (in double)
 * and rstd, pre / post / comb, the collapse of the residual with this pre and
 * the layer RMSNorm follow exactly as in oracle_boundary mode 0.
 */
void oracle_pre_split_k(const uint16_t *residual, const float *dot_mix, const float *sqrsum,
                        int S, const float *scale, const float *base, const void *norm_w,
                        int nw_bf16, const oracle_params *p, int64_t T, int H,
                        uint16_t *layer_input, float *pre_out, float *post_out,
                        float *comb_out)
{
    const int64_t K = (int64_t)NHC * H;
    uint16_t *li = (uint16_t *)malloc(sizeof(uint16_t) * H);
    if (!li) return;
    for (int64_t t = 0; t < T; ++t) {
        float mix[MIXES];
        for (int n = 0; n < MIXES; ++n) {
            double acc = 0.0;
            for (int s = 0; s < S; ++s) acc += (double)dot_mix[((int64_t)s * T + t) * MIXES + n];
            mix[n] = (float)acc;
        }
        double ssq = 0.0;
        for (int s = 0; s < S; ++s) ssq += (double)sqrsum[(int64_t)s * T + t];
        float rstd = (float)(1.0 / sqrt(ssq / (double)K + (double)p->hc_norm_eps));
        float pre[NHC], post[NHC], comb[NHC * NHC];
        coefficients(mix, rstd, scale, base, p, pre, post, comb);
        if (pre_out) memcpy(pre_out + t * NHC, pre, sizeof pre);
        if (post_out) memcpy(post_out + t * NHC, post, sizeof post);
        if (comb_out) memcpy(comb_out + t * NHC * NHC, comb, sizeof comb);
        collapse_norm(residual + t * K, pre, norm_w, nw_bf16, p, H, li,
                      layer_input ? layer_input + t * H : NULL);
    }
    free(li);
}

/* Coefficients alone, for pins that start from given mixes and rstd. */
void oracle_coefficients(const float *mix, const float *rstd, const float *scale,
                         const float *base, const oracle_params *p, int64_t T,
                         float *pre, float *post, float *comb)
{
    for (int64_t t = 0; t < T; ++t)
        coefficients(mix + t * MIXES, rstd[t], scale, base, p, pre + t * NHC,
                     post + t * NHC, comb + t * NHC * NHC);
}

/* Scalar conversions, exported for the bit-level pins. */
void oracle_f32_to_bf16(const float *f, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16(f[i]);
}

void oracle_tf32_round(const float *w, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = tf32_round(w[i]);
}

void oracle_sigmoid(const float *v, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = sigmoid(v[i]);
}

void oracle_sinkhorn(float *c16, int64_t T, int iters, float eps)
{
    for (int64_t t = 0; t < T; ++t) sinkhorn(c16 + t * 16, iters, eps);
}
