// Streaming pass of the mHC boundary: one CTA per (hidden slice, 128-token
// tile). Per 32-wide hidden chunk of its slice the CTA
//   1. TMA-loads the residual tile [4 streams][128 tokens][32] and the x tile
//      [128][32] (bf16, 64-byte swizzled rows) and the chunk's prepared
//      weight tile [4][48][32] (bulk copy, already in swizzled order);
//   2. updates the residual in shared memory (post: the flush-to-zero FMA
//      chain of the "mhc_boundary" page's residual_update), folds the squares
//      of the updated values into per-token sums, and for the shifted form
//      writes the collapse with the lagged pre (lagged_collapse) over x;
//   3. TMA-stores the updated residual (and the unnormalised collapse);
//   4. issues 8 tcgen05 MMAs (M=128 tokens, N=48 stacked hi/lo weight rows,
//      K=16) accumulating the mixer contraction in TMEM.
// At the end each token's 24 partial mixes (hi + lo) and its partial sums of
// squares go to the workspace; a finishing kernel reduces the slices in a
// fixed order. Warp roles: warp 0 TMA producer and TMEM owner, warp 1 MMA
// issuer, warps 2-9 elementwise workers (token = 32*(warp%4) + lane, so that
// a worker reads the TMEM lanes of its own tokens).
#include "mhc_internal.h"
#include "ptx.cuh"

namespace mhc {
namespace {

constexpr int kBarOff(int stages) { return stages * kStageBytes; }
constexpr int kSsqOff(int stages) { return kBarOff(stages) + 256; }
constexpr int kMiscOff(int stages) { return kSsqOff(stages) + 2 * kTileT * 4; }
constexpr int kSmemUsed(int stages) { return kMiscOff(stages) + 64; }

// Wait-site ids recorded with a timeout.
enum : int { SITE_PROD_READY = 1, SITE_PROD_MMA = 2, SITE_MMA_FULL = 3, SITE_MMA_READY = 4,
             SITE_WORK_FULL = 5, SITE_EPI_MMA = 6, SITE_DRAIN = 7 };

struct Coefs {
    uint64_t post2[4];       // (post[s], post[s])
    uint64_t comb2[4][4];    // [j][s] -> (comb[j][s], comb[j][s])
    uint64_t pre2[4];        // (pre_lag[j], pre_lag[j])
};

// Residual update of 8 hidden values of every stream: r[j] holds stream j,
// xw holds x. Chain per value: ftz(post*x), then ftz(fma(comb[j][s], r[j], .)).
__device__ __forceinline__ void update8(const uint4 (&r)[4], const uint4 &xw, const Coefs &c,
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

__device__ __forceinline__ void sq_accum(const uint4 &v, uint64_t &acc) {
    uint64_t a = bf2_unpack(v.x); acc = fma2(a, a, acc);
    a = bf2_unpack(v.y); acc = fma2(a, a, acc);
    a = bf2_unpack(v.z); acc = fma2(a, a, acc);
    a = bf2_unpack(v.w); acc = fma2(a, a, acc);
}

// Lagged collapse of 8 hidden values: li = bf16(fma chain over j from 0).
__device__ __forceinline__ uint4 collapse8(const uint4 (&cur)[4], const Coefs &c) {
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

__device__ __forceinline__ void named_bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Bounded wait that ignores the abort flag (used to drain copies in flight
// before the CTA exits after an abort).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                           unsigned int *status) {
    int local = 0;
    mbar_wait(bar, parity, &local, timeout_ns, status, SITE_DRAIN);
}

template <int MODE, int STAGES>
__global__ void __launch_bounds__(kStreamThreads, 1)
stream_kernel(const __grid_constant__ CUtensorMap tm_res, const __grid_constant__ CUtensorMap tm_x,
              const __grid_constant__ CUtensorMap tm_rout, const __grid_constant__ CUtensorMap tm_li,
              const StreamArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t bars = base + kBarOff(STAGES);
    auto full = [&](int st) { return bars + 8u * st; };
    auto ready = [&](int st) { return bars + 8u * (STAGES + st); };
    auto mma_done = [&](int st) { return bars + 8u * (2 * STAGES + st); };
    float *ssq_x = reinterpret_cast<float *>(gbase + kSsqOff(STAGES));
    float *ssql_x = ssq_x + kTileT;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + kMiscOff(STAGES));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + kMiscOff(STAGES) + 16);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int slice = blockIdx.x;
    const int h0 = slice * a.slice_w;
    const long long t0 = static_cast<long long>(blockIdx.y) * kTileT;
    const int n = a.slice_w / kChunk;
    const uint64_t tmo = a.timeout_ns;

    if (tid == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(full(i), 1);
            mbar_init(ready(i), 8);
            mbar_init(mma_done(i), 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (tid == 32) {
        tma_prefetch_desc(&tm_res);
        if (MODE != PRE_ONLY) { tma_prefetch_desc(&tm_x); tma_prefetch_desc(&tm_rout); }
        if (MODE == FUSED_SHIFTED) tma_prefetch_desc(&tm_li);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_d = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            const uint64_t pol_stream = policy_evict_first();
            const uint64_t pol_w = policy_evict_last();
            constexpr uint32_t kLoadBytes =
                kResBytes + kWBytes + (MODE != PRE_ONLY ? kXBytes : 0);
            auto issue_load = [&](int c) {
                const int st = c % STAGES;
                const uint32_t sb = base + st * kStageBytes;
                const int hc = h0 + c * kChunk;
                mbar_arrive_expect_tx(full(st), kLoadBytes);
                tma_load_3d(sb, &tm_res, hc, static_cast<int>(t0), 0, full(st), pol_stream);
                if (MODE != PRE_ONLY)
                    tma_load_2d(sb + kResBytes, &tm_x, hc, static_cast<int>(t0), full(st),
                                pol_stream);
                bulk_load(sb + kResBytes + kXBytes,
                          a.weight + static_cast<size_t>(hc / kChunk) * kWBytes, kWBytes,
                          full(st), pol_w);
            };
            int loaded = 0;
            for (; loaded < n && loaded < STAGES; ++loaded) issue_load(loaded);
            int j = 0;
            for (; j < n; ++j) {
                const int st = j % STAGES;
                const uint32_t ph = (j / STAGES) & 1;
                if (!mbar_wait(ready(st), ph, abort_flag, tmo, a.status, SITE_PROD_READY)) break;
                const uint32_t sb = base + st * kStageBytes;
                if (MODE != PRE_ONLY) {
                    tma_store_3d(&tm_rout, h0 + j * kChunk, static_cast<int>(t0), 0, sb,
                                 pol_stream);
                    if (MODE == FUSED_SHIFTED)
                        tma_store_2d(&tm_li, h0 + j * kChunk, static_cast<int>(t0),
                                     sb + kResBytes, pol_stream);
                    bulk_commit();
                }
                if (loaded < n) {
                    if (MODE != PRE_ONLY) bulk_wait_read_all();
                    if (!mbar_wait(mma_done(st), ph, abort_flag, tmo, a.status, SITE_PROD_MMA))
                        break;
                    issue_load(loaded);
                    ++loaded;
                }
            }
            bulk_wait_all();
            if (j < n) {  // aborted: let the loads in flight land before exiting
                for (int c = j; c < loaded; ++c)
                    drain_wait(full(c % STAGES), (c / STAGES) & 1, tmo, a.status);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            constexpr uint32_t kIdesc = idesc_bf16_f32(kTileT, kWRows);
            int issued = 0;
            for (int j = 0; j < n; ++j) {
                const int st = j % STAGES;
                const uint32_t ph = (j / STAGES) & 1;
                if (!mbar_wait(full(st), ph, abort_flag, tmo, a.status, SITE_MMA_FULL)) break;
                if (!mbar_wait(ready(st), ph, abort_flag, tmo, a.status, SITE_MMA_READY)) break;
                tc_fence_after();
                const uint32_t sb = base + st * kStageBytes;
#pragma unroll
                for (int s = 0; s < 4; ++s) {
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const uint64_t ad =
                            smem_desc_sw64(sb + s * kTileT * kRowBytes + k * 32, 8 * kRowBytes);
                        const uint64_t bd = smem_desc_sw64(
                            sb + kResBytes + kXBytes + s * kWRows * kRowBytes + k * 32,
                            8 * kRowBytes);
                        tc_mma_bf16(tmem_d, ad, bd, kIdesc, (j | s | k) != 0);
                    }
                }
                tc_commit(mma_done(st));
                issued = j + 1;
            }
            if (issued > 0 && issued < n) {  // aborted: let the issued MMAs finish
                const int c = issued - 1;
                drain_wait(mma_done(c % STAGES), (c / STAGES) & 1, tmo, a.status);
            }
        }
    } else {
        // ---------------------------------------------------- elementwise workers
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        const int t = q * 32 + lane;
        const long long gt = t0 + t;
        const bool valid = gt < a.T;
        Coefs cf;
        if (MODE != PRE_ONLY) {
            float4 pv = make_float4(0.f, 0.f, 0.f, 0.f);
            float4 cv[4] = {pv, pv, pv, pv};
            if (valid) {
                pv = __ldg(reinterpret_cast<const float4 *>(a.post) + gt);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    cv[j] = __ldg(reinterpret_cast<const float4 *>(a.comb) + gt * 4 + j);
            }
            const float ps[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
            for (int s = 0; s < 4; ++s) cf.post2[s] = f2_pack(ps[s], ps[s]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float cs[4] = {cv[j].x, cv[j].y, cv[j].z, cv[j].w};
#pragma unroll
                for (int s = 0; s < 4; ++s) cf.comb2[j][s] = f2_pack(cs[s], cs[s]);
            }
        }
        if (MODE == FUSED_SHIFTED) {
            float4 lv = make_float4(0.f, 0.f, 0.f, 0.f);
            if (valid) lv = __ldg(reinterpret_cast<const float4 *>(a.pre_lag) + gt);
            const float ls[4] = {lv.x, lv.y, lv.z, lv.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) cf.pre2[j] = f2_pack(ls[j], ls[j]);
        }
        uint64_t ssq2 = 0, ssql2 = 0;
        const uint32_t swz = (t >> 1) & 3;
        for (int j = 0; j < n; ++j) {
            const int st = j % STAGES;
            const uint32_t ph = (j / STAGES) & 1;
            if (!mbar_wait(full(st), ph, abort_flag, tmo, a.status, SITE_WORK_FULL)) break;
            const uint32_t sb = base + st * kStageBytes;
            if (valid) {
#pragma unroll
                for (int uu = 0; uu < 2; ++uu) {
                    const int u = 2 * half + uu;
                    const uint32_t off = t * kRowBytes + 16u * (u ^ swz);
                    uint4 r[4];
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        r[s] = ld_shared_v4(sb + s * kTileT * kRowBytes + off);
                    if (MODE == PRE_ONLY) {
#pragma unroll
                        for (int s = 0; s < 4; ++s) sq_accum(r[s], ssq2);
                    } else {
                        const uint4 xw = ld_shared_v4(sb + kResBytes + off);
                        uint4 cur[4];
                        update8(r, xw, cf, cur);
#pragma unroll
                        for (int s = 0; s < 4; ++s) {
                            st_shared_v4(sb + s * kTileT * kRowBytes + off, cur[s]);
                            sq_accum(cur[s], ssq2);
                        }
                        if (MODE == FUSED_SHIFTED) {
                            const uint4 li = collapse8(cur, cf);
                            st_shared_v4(sb + kResBytes + off, li);
                            sq_accum(li, ssql2);
                        }
                    }
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(ready(st));
        }
        // ---- epilogue: sums of squares (half 0 + half 1), mixes from TMEM
        const float ssq = f2_lo(ssq2) + f2_hi(ssq2);
        const float ssql = f2_lo(ssql2) + f2_hi(ssql2);
        if (half == 1) {
            ssq_x[t] = ssq;
            ssql_x[t] = ssql;
        }
        named_bar_sync(1, 256);
        if (half == 0) {
            const int c = n - 1;
            const bool ok = mbar_wait(mma_done(c % STAGES), (c / STAGES) & 1, abort_flag, tmo,
                                      a.status, SITE_EPI_MMA);
            tc_fence_after();
            uint32_t v[48];
            const uint32_t row = tmem_d + (static_cast<uint32_t>(q * 32) << 16);
            tmem_ld16(row + 0, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
            tmem_ld16(row + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
            tmem_ld16(row + 32, *reinterpret_cast<uint32_t(*)[16]>(&v[32]));
            tmem_ld_wait();
            tc_fence_before();
            if (valid && ok) {
                float out[kPartStride];
#pragma unroll
                for (int i = 0; i < 24; ++i)
                    out[i] = __uint_as_float(v[i]) + __uint_as_float(v[24 + i]);
                out[24] = ssq + ssq_x[t];
                out[25] = ssql + ssql_x[t];
                out[26] = 0.f;
                out[27] = 0.f;
                float4 *dst = reinterpret_cast<float4 *>(
                    a.partials + (static_cast<size_t>(slice) * a.T + gt) * kPartStride);
#pragma unroll
                for (int i = 0; i < kPartStride / 4; ++i)
                    dst[i] = make_float4(out[4 * i], out[4 * i + 1], out[4 * i + 2],
                                         out[4 * i + 3]);
            }
        }
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_d, kTmemCols);
    }
}

template <int MODE, int STAGES>
cudaError_t launch_t(const CUtensorMap &res, const CUtensorMap &x, const CUtensorMap &rout,
                     const CUtensorMap &li, const StreamArgs &a, int n_slices, int n_tiles,
                     cudaStream_t s) {
    constexpr int smem = kSmemUsed(STAGES) + 1024;
    auto kern = stream_kernel<MODE, STAGES>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(n_slices, n_tiles), kStreamThreads, smem, s>>>(res, x, rout, li, a);
    return cudaGetLastError();
}

}  // namespace

size_t stream_smem_bytes(int stages) { return kSmemUsed(stages) + 1024; }

cudaError_t launch_stream(int mode, int stages, const CUtensorMap &res, const CUtensorMap &x,
                          const CUtensorMap &rout, const CUtensorMap &li, const StreamArgs &a,
                          int n_slices, int n_tiles, cudaStream_t s) {
    if (stages != 2) return cudaErrorInvalidValue;
    switch (mode) {
        case PRE_ONLY: return launch_t<PRE_ONLY, 2>(res, x, rout, li, a, n_slices, n_tiles, s);
        case FUSED_UNSHIFTED:
            return launch_t<FUSED_UNSHIFTED, 2>(res, x, rout, li, a, n_slices, n_tiles, s);
        case FUSED_SHIFTED:
            return launch_t<FUSED_SHIFTED, 2>(res, x, rout, li, a, n_slices, n_tiles, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mhc
