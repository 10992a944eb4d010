// Per-token coefficient math of the boundary and the RMSNorm of the collapse,
// shared by the streaming and finishing kernels.
#pragma once
#include "mhc_internal.h"
#include "ptx.cuh"

namespace mhc {

// ------------------------------------------------------------ coefficients
// Reciprocal of a positive normal x whose reciprocal is also normal, as the
// "mhc_boundary" page's rcp: the hardware approximation y0 refined by one
// Newton-Raphson step in fused multiply-add form, y0 + y0 * (1 - x * y0)
// (Markstein); 1 - x * y0 is exact. The library checks on the GPU that this
// equals the correctly rounded reciprocal for every such x.
static __device__ __forceinline__ float rcp_nr(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return fmaf(y, fmaf(-x, y, 1.0f), y);
}

static __device__ __forceinline__ float sigmoid_clamped(float v) {
    // 1 / min(1 + exp(-v), 2^126) ("mhc_boundary" page, sigmoid)
    return rcp_nr(fminf(1.0f + expf(-v), 0x1p126f));
}

// Coefficients of token t formed by one thread from the token's reduced
// values v[i * stride]: i = 0..23 the mixes, 24 the 4H sum of squares; writes
// pre / post / comb. Order of operations as in the "mhc_boundary" page
// (coefficients, sinkhorn, col_normalize): pre = sigmoid(m0 * s0 + b) + eps,
// post = sigmoid(m1 * s1 + b) * post_mult, comb = row softmax (multiplied by
// the reciprocal of the row sum, plus eps), one column normalisation, then
// iters - 1 times a row and a column normalisation; column sums pair rows
// (0, 1) and (2, 3).
// sb: scale[0..2] then base[0..23], staged in shared memory by the caller.
static __device__ __forceinline__ void coefficients_thread(const float *v, int stride,
                                                           const float *sb, const CoefArgs &c,
                                                           int H, long long t, float *pre_out,
                                                           float *post_out, float *comb_out) {
    const float rstd =
        rsqrtf(__fdiv_rn(v[24 * stride], static_cast<float>(4 * H)) + c.hc_norm_eps);
    const float s0 = sb[0], s1 = sb[1], s2 = sb[2];
    const float *bs = sb + 3;
    float pp[4], po[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        pp[i] = sigmoid_clamped(fmaf(v[i * stride] * rstd, s0, bs[i])) + c.hc_pre_eps;
        po[i] = sigmoid_clamped(fmaf(v[(4 + i) * stride] * rstd, s1, bs[4 + i])) * c.hc_post_mult;
    }
    reinterpret_cast<float4 *>(pre_out)[t] = make_float4(pp[0], pp[1], pp[2], pp[3]);
    reinterpret_cast<float4 *>(post_out)[t] = make_float4(po[0], po[1], po[2], po[3]);
    const float eps = c.sinkhorn_eps;
    float x[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        float l[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            l[k] = fmaf(v[(8 + 4 * r + k) * stride] * rstd, s2, bs[8 + 4 * r + k]);
        const float mx = fmaxf(fmaxf(l[0], l[1]), fmaxf(l[2], l[3]));
        float e[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) e[k] = expf(l[k] - mx);
        const float inv = rcp_nr(((e[0] + e[1]) + e[2]) + e[3]);
#pragma unroll
        for (int k = 0; k < 4; ++k) x[r][k] = fmaf(e[k], inv, eps);
    }
    auto col_normalize = [&]() {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float r = rcp_nr(((x[0][k] + x[1][k]) + (x[2][k] + x[3][k])) + eps);
#pragma unroll
            for (int i = 0; i < 4; ++i) x[i][k] = x[i][k] * r;
        }
    };
    col_normalize();
    for (int it = 1; it < c.sinkhorn_iters; ++it) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float r = rcp_nr((((x[i][0] + x[i][1]) + x[i][2]) + x[i][3]) + eps);
#pragma unroll
            for (int k = 0; k < 4; ++k) x[i][k] = x[i][k] * r;
        }
        col_normalize();
    }
    float4 *cb = reinterpret_cast<float4 *>(comb_out) + t * 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) cb[i] = make_float4(x[i][0], x[i][1], x[i][2], x[i][3]);
}

// The same coefficients formed by 16 lanes of a warp, lane l holding comb
// entry (l / 4, l % 4): row and column sums gather their four terms by
// shuffle and add them in the order of coefficients_thread, and every other
// operation is the same, so the outputs are bitwise those of
// coefficients_thread, with about a quarter of its instructions per lane
// (the Sinkhorn steps run on the 16 entries at once): for latency, when few
// tokens wait on it. Called by all 32 lanes of a warp: lanes 0-15 form token
// t_lo (if valid_lo), lanes 16-31 token t_hi (if valid_hi); v_lo / v_hi as
// in coefficients_thread.
static __device__ __forceinline__ void coefficients_16lanes(const float *v_lo, const float *v_hi,
                                                            int stride, const float *sb,
                                                            const CoefArgs &c, int H, long long t_lo,
                                                            long long t_hi, bool valid_lo,
                                                            bool valid_hi, float *pre_out,
                                                            float *post_out, float *comb_out) {
    const int lane = threadIdx.x & 31;
    const int l = lane & 15, g0 = lane & 16;          // entry, first lane of this token's group
    const bool hi = lane >= 16;
    const float *v = hi ? v_hi : v_lo;
    const long long t = hi ? t_hi : t_lo;
    const bool valid = hi ? valid_hi : valid_lo;
    const float rstd =
        rsqrtf(__fdiv_rn(v[24 * stride], static_cast<float>(4 * H)) + c.hc_norm_eps);
    const float *bs = sb + 3;
    if (l < 4) {
        const float p = sigmoid_clamped(fmaf(v[l * stride] * rstd, sb[0], bs[l])) + c.hc_pre_eps;
        if (valid) pre_out[t * 4 + l] = p;
    } else if (l < 8) {
        const float p =
            sigmoid_clamped(fmaf(v[l * stride] * rstd, sb[1], bs[l])) * c.hc_post_mult;
        if (valid) post_out[t * 4 + (l - 4)] = p;
    }
    const int r = l >> 2, k = l & 3;
    const float eps = c.sinkhorn_eps;
    auto at = [&](float x, int e) { return __shfl_sync(0xffffffffu, x, g0 + e); };
    // row softmax of the logits, multiplied by the reciprocal of the row sum, plus eps
    const float lg = fmaf(v[(8 + l) * stride] * rstd, sb[2], bs[8 + l]);
    const float l0 = at(lg, 4 * r), l1 = at(lg, 4 * r + 1), l2 = at(lg, 4 * r + 2),
                l3 = at(lg, 4 * r + 3);
    const float e = expf(lg - fmaxf(fmaxf(l0, l1), fmaxf(l2, l3)));
    const float e0 = at(e, 4 * r), e1 = at(e, 4 * r + 1), e2 = at(e, 4 * r + 2),
                e3 = at(e, 4 * r + 3);
    float x = fmaf(e, rcp_nr(((e0 + e1) + e2) + e3), eps);
    auto col_normalize = [&]() {
        const float c0 = at(x, k), c1 = at(x, 4 + k), c2 = at(x, 8 + k), c3 = at(x, 12 + k);
        x = x * rcp_nr(((c0 + c1) + (c2 + c3)) + eps);
    };
    col_normalize();
    for (int it = 1; it < c.sinkhorn_iters; ++it) {
        const float x0 = at(x, 4 * r), x1 = at(x, 4 * r + 1), x2 = at(x, 4 * r + 2),
                    x3 = at(x, 4 * r + 3);
        x = x * rcp_nr((((x0 + x1) + x2) + x3) + eps);
        col_normalize();
    }
    if (valid) comb_out[t * 16 + l] = x;
}

// Stages scale[0..2] and base[0..23] into sb[0..26] (threads 0..26 of the caller's group).
static __device__ __forceinline__ void stage_coef_consts(const CoefArgs &c, float *sb, int i) {
    if (i < 3) sb[i] = __ldg(c.scale + i);
    else if (i < 27) sb[i] = __ldg(c.base + i - 3);
}

// out = bf16((li * rstd_li) * norm_w) for 8 values
static __device__ __forceinline__ uint4 norm8(uint4 li, float rstd_li, const void *norm_w, int nw_bf16,
                                       long long h) {
    float w[8];
    if (nw_bf16) {
        const uint4 nv = ld_global_nc_v4(static_cast<const uint16_t *>(norm_w) + h);
        const uint32_t ws[4] = {nv.x, nv.y, nv.z, nv.w};
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            w[2 * p] = __uint_as_float(ws[p] << 16);
            w[2 * p + 1] = __uint_as_float(ws[p] & 0xFFFF0000u);
        }
    } else {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(norm_w) + h));
        const float4 b =
            __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(norm_w) + h) + 1);
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
        w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
    }
    const uint32_t ls[4] = {li.x, li.y, li.z, li.w};
    uint32_t o[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const float lo = __fmul_rn(__fmul_rn(__uint_as_float(ls[p] << 16), rstd_li), w[2 * p]);
        const float hi =
            __fmul_rn(__fmul_rn(__uint_as_float(ls[p] & 0xFFFF0000u), rstd_li), w[2 * p + 1]);
        o[p] = bf2_pack_rn(f2_pack(lo, hi));
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace mhc
