// Per-token elementwise chains of the boundary on packed fp32 pairs, shared
// by the streaming and the cluster kernels: the residual update ("mhc_boundary"
// page, residual_update: the flush-to-zero FMA chain post[s]*x, then
// comb[j][s]*residual[j] for j = 0..3, rounded to bf16), the lagged collapse
// (lagged_collapse: fma chain of pre[j]*cur[j] from zero, rounded to bf16) and
// the sums of squares of bf16 values.
#pragma once
#include "ptx.cuh"

namespace mhc {

struct Coefs {
    uint64_t post2[4];       // (post[s], post[s])
    uint64_t comb2[4][4];    // [j][s] -> (comb[j][s], comb[j][s])
    uint64_t pre2[4];        // (pre_lag[j], pre_lag[j])
};

// Residual update of 8 hidden values of every stream: r[j] holds stream j,
// xw holds x. Chain per value: ftz(post*x), then ftz(fma(comb[j][s], r[j], .)).
static __device__ __forceinline__ void update8(const uint4 (&r)[4], const uint4 &xw, const Coefs &c,
                                        uint4 (&cur)[4]) {
    const uint32_t xs[4] = {xw.x, xw.y, xw.z, xw.w};
    uint32_t rs[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        rs[j][0] = r[j].x; rs[j][1] = r[j].y; rs[j][2] = r[j].z; rs[j][3] = r[j].w;
    }
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        uint32_t w[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            uint64_t nu = mul2_ftz(c.post2[s], bf2_unpack(xs[p]));
#pragma unroll
            for (int j = 0; j < 4; ++j) nu = fma2_ftz(c.comb2[j][s], bf2_unpack(rs[j][p]), nu);
            w[p] = bf2_pack_rn(nu);
        }
        cur[s] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// The same update for 4 hidden values (2 bf16 pairs) of every stream.
static __device__ __forceinline__ void update4(const uint2 (&r)[4], const uint2 &xw, const Coefs &c,
                                        uint2 (&cur)[4]) {
    const uint32_t xs[2] = {xw.x, xw.y};
    uint32_t rs[4][2];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        rs[j][0] = r[j].x; rs[j][1] = r[j].y;
    }
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        uint32_t w[2];
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            uint64_t nu = mul2_ftz(c.post2[s], bf2_unpack(xs[p]));
#pragma unroll
            for (int j = 0; j < 4; ++j) nu = fma2_ftz(c.comb2[j][s], bf2_unpack(rs[j][p]), nu);
            w[p] = bf2_pack_rn(nu);
        }
        cur[s] = make_uint2(w[0], w[1]);
    }
}

static __device__ __forceinline__ void sq_accum2(const uint2 &v, uint64_t &acc) {
    uint64_t a = bf2_unpack(v.x); acc = fma2(a, a, acc);
    a = bf2_unpack(v.y); acc = fma2(a, a, acc);
}

// Lagged collapse of 4 hidden values.
static __device__ __forceinline__ uint2 collapse4(const uint2 (&cur)[4], const Coefs &c) {
    const uint32_t cs[4][2] = {{cur[0].x, cur[0].y}, {cur[1].x, cur[1].y}, {cur[2].x, cur[2].y},
                               {cur[3].x, cur[3].y}};
    uint32_t w[2];
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        uint64_t acc = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) acc = fma2(c.pre2[j], bf2_unpack(cs[j][p]), acc);
        w[p] = bf2_pack_rn(acc);
    }
    return make_uint2(w[0], w[1]);
}

// Coefs of one token from its post, comb and lagged pre.
static __device__ __forceinline__ Coefs coefs_of(const float4 &pv, const float4 (&cv)[4], const float4 &lv) {
    Coefs c;
    const float ps[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
    for (int s = 0; s < 4; ++s) c.post2[s] = f2_pack(ps[s], ps[s]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float cs[4] = {cv[j].x, cv[j].y, cv[j].z, cv[j].w};
#pragma unroll
        for (int s = 0; s < 4; ++s) c.comb2[j][s] = f2_pack(cs[s], cs[s]);
    }
    const float ls[4] = {lv.x, lv.y, lv.z, lv.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) c.pre2[j] = f2_pack(ls[j], ls[j]);
    return c;
}

static __device__ __forceinline__ void sq_accum(const uint4 &v, uint64_t &acc) {
    uint64_t a = bf2_unpack(v.x); acc = fma2(a, a, acc);
    a = bf2_unpack(v.y); acc = fma2(a, a, acc);
    a = bf2_unpack(v.z); acc = fma2(a, a, acc);
    a = bf2_unpack(v.w); acc = fma2(a, a, acc);
}

// Lagged collapse of 8 hidden values: li = bf16(fma chain over j from 0).
static __device__ __forceinline__ uint4 collapse8(const uint4 (&cur)[4], const Coefs &c) {
    uint32_t cs[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        cs[j][0] = cur[j].x; cs[j][1] = cur[j].y; cs[j][2] = cur[j].z; cs[j][3] = cur[j].w;
    }
    uint32_t w[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        uint64_t acc = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) acc = fma2(c.pre2[j], bf2_unpack(cs[j][p]), acc);
        w[p] = bf2_pack_rn(acc);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace mhc
