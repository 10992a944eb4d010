// Per-token coefficient math of the boundary and the RMSNorm of the collapse,
// shared by the streaming and finishing kernels.
#pragma once
#include "mhc_internal.h"
#include "ptx.cuh"

namespace mhc {

// ------------------------------------------------------------ coefficients
static __device__ __forceinline__ float sigmoid_clamped(float v) {
    // 1 / min(1 + exp(-v), 2^126) ("mhc_boundary" page, sigmoid)
    return __frcp_rn(fminf(1.0f + expf(-v), 0x1p126f));
}

// Lane map of one token's warp: lanes 0-3 pre (mix 0-3), 4-7 post (mix 4-7),
// lane 8 the 4H sum of squares, lane 9 the collapse's sum of squares, lanes
// 16-31 comb (mix 8-23, lane 16 + 4i + k = row i, column k).
static __device__ __forceinline__ int lane_slot(int lane) {
    if (lane < 8) return lane;
    if (lane == 8) return 24;
    if (lane == 9) return 25;
    if (lane >= 16) return lane - 8;
    return -1;
}

// Sum of one token's slice partials in slice order (fixed, deterministic).
static __device__ __forceinline__ float reduce_slices(const float *__restrict__ partials, int n_slices,
                                               long long T, long long t, int slot) {
    float v = 0.f;
    if (slot >= 0) {
        // independent loads, added in slice order
        const float *p = partials + t * kPartStride + slot;
        const long long step = T * kPartStride;
        int s = 0;
        for (; s + 8 <= n_slices; s += 8) {
            float w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) w[i] = __ldg(p + (s + i) * step);
#pragma unroll
            for (int i = 0; i < 8; ++i) v += w[i];
        }
        for (; s < n_slices; ++s) v += __ldg(p + s * step);
    }
    return v;
}

// Coefficients of token t from its reduced value v (lane map above); writes
// pre / post / comb. Returns pre[lane & 3] in lanes 0-3 (undefined elsewhere).
// Order of operations as in the "mhc_boundary" page (coefficients, sinkhorn,
// col_normalize); the Sinkhorn runs on 16 lanes with shuffles.
static __device__ __forceinline__ float coefficients_warp(float v, int lane, const CoefArgs &c, int H, long long t,
                                   float *pre_out, float *post_out, float *comb_out) {
    const unsigned full = 0xffffffffu;
    const float ssq = __shfl_sync(full, v, 8);
    const float rstd = rsqrtf(__fdiv_rn(ssq, static_cast<float>(4 * H)) + c.hc_norm_eps);
    const int slot = lane_slot(lane);
    const float m = v * rstd;
    float pre = 0.f;
    if (lane < 4) {
        pre = sigmoid_clamped(fmaf(m, __ldg(c.scale + 0), __ldg(c.base + slot))) + c.hc_pre_eps;
        pre_out[t * 4 + lane] = pre;
    } else if (lane < 8) {
        const float p = sigmoid_clamped(fmaf(m, __ldg(c.scale + 1), __ldg(c.base + slot)));
        post_out[t * 4 + lane - 4] = p * c.hc_post_mult;
    }
    // comb lanes 16..31; the other lanes follow the shuffles on dummy values
    const bool comb_lane = lane >= 16;
    const float l = comb_lane ? fmaf(m, __ldg(c.scale + 2), __ldg(c.base + slot)) : 0.f;
    const int rb = lane & ~3;   // first lane of this row
    float mx = fmaxf(l, __shfl_xor_sync(full, l, 1));
    mx = fmaxf(mx, __shfl_xor_sync(full, mx, 2));
    const float e = comb_lane ? expf(l - mx) : 1.f;
    const float e0 = __shfl_sync(full, e, rb), e1 = __shfl_sync(full, e, rb + 1);
    const float e2 = __shfl_sync(full, e, rb + 2), e3 = __shfl_sync(full, e, rb + 3);
    const float inv = __frcp_rn(((e0 + e1) + e2) + e3);
    const float eps = c.sinkhorn_eps;
    float x = fmaf(e, inv, eps);
    // column normalisation: (c0k + c1k) + (c2k + c3k), plus eps
    float cs = x + __shfl_xor_sync(full, x, 4);
    cs = cs + __shfl_xor_sync(full, cs, 8);
    x = x * __frcp_rn(cs + eps);
    for (int it = 1; it < c.sinkhorn_iters; ++it) {
        const float c0 = __shfl_sync(full, x, rb), c1 = __shfl_sync(full, x, rb + 1);
        const float c2 = __shfl_sync(full, x, rb + 2), c3 = __shfl_sync(full, x, rb + 3);
        x = x * __frcp_rn((((c0 + c1) + c2) + c3) + eps);
        cs = x + __shfl_xor_sync(full, x, 4);
        cs = cs + __shfl_xor_sync(full, cs, 8);
        x = x * __frcp_rn(cs + eps);
    }
    if (comb_lane) comb_out[t * 16 + (lane - 16)] = x;
    return pre;
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
