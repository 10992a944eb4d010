// Streaming pass of the mHC boundary, persistent: one CTA per SM walks a
// static list of work items (a 128-token tile x a hidden slice) and runs one
// continuous chunk pipeline across them. Per 32-wide hidden chunk:
//   1. TMA-load the residual tile [4 streams][128 tokens][32] and the x tile
//      [128][32] (bf16, 64-byte swizzled rows) and bulk-load the chunk's
//      prepared weight tile [4][48][32] (already in swizzled order);
//   2. workers update the residual in shared memory (post: the flush-to-zero
//      FMA chain of the "mhc_boundary" page's residual_update), fold squares
//      of the updated values into per-token sums, and for the shifted form
//      write the collapse with the lagged pre (lagged_collapse) over x;
//   3. TMA-store the updated residual (and the unnormalised collapse);
//   4. one thread issues 8 tcgen05 MMAs (M=128 tokens, N=48 stacked hi/lo
//      weight rows, K=16) accumulating the mixer contraction in TMEM.
// Each item accumulates into one of two TMEM buffers; its epilogue (24
// partial mixes hi + lo and the partial sums of squares per token, written
// to the workspace) runs in the workers after they have handled the first
// chunk of the next item, so neither the MMA nor the stream drains between
// items. A finishing kernel reduces the slices in a fixed order.
// Warp roles: warp 0 TMA producer and TMEM owner, warp 1 MMA issuer, warps
// 2-9 workers (token = 32*(warp%4) + lane: a worker reads the TMEM lanes of
// its own tokens; warps 2-5 and 6-9 each take two of the four 8-wide units).
#include "mhc_internal.h"
#include "ptx.cuh"

namespace mhc {
namespace {

constexpr int kStages = 4;
constexpr int kBarOff = kStages * kStageBytes;
constexpr int kNumBars = 3 * kStages + 8;
constexpr int kSsqOff = kBarOff + 256;                 // [2 buffers][2 sums][128] fp32
constexpr int kMiscOff = kSsqOff + 2 * 2 * kTileT * 4;
constexpr int kSmemUsed = kMiscOff + 64;
constexpr int kAccCols = 64;                           // one accumulator buffer (48 used)
static_assert(kNumBars * 8 <= 256, "barrier area");

// Wait-site ids recorded with a timeout.
enum : int { SITE_PROD_READY = 1, SITE_PROD_MMA = 2, SITE_MMA_FULL = 3, SITE_MMA_READY = 4,
             SITE_WORK_FULL = 5, SITE_EPI_ACC = 6, SITE_DRAIN = 7, SITE_MMA_ACC = 8,
             SITE_EPI_SSQ = 9, SITE_EPI_SSQ_FREE = 10 };

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

// Bounded wait that ignores the abort flag (drains copies in flight before
// the CTA exits after an abort).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                           unsigned int *status) {
    int local = 0;
    mbar_wait(bar, parity, &local, timeout_ns, status, SITE_DRAIN);
}

// Work item k of this CTA -> (tile, slice). Consecutive CTAs take the
// slices of one tile, so they stream the same rows at the same time.
struct Item {
    int tile, slice;
};
__device__ __forceinline__ Item item_of(int k, int n_slices) {
    const int i = blockIdx.x + k * gridDim.x;
    return {i / n_slices, i % n_slices};
}

// First hidden index of chunk c of a slice. Slices interleave chunk by chunk
// (slice s owns chunks s, s + S, s + 2S, ...), so the CTAs working on one tile
// read adjacent 64-byte pieces of every row together: DRAM pages are opened
// once for all of them instead of once per CTA.
__device__ __forceinline__ int chunk_hidden(int slice, int c, int n_slices) {
    return (c * n_slices + slice) * kChunk;
}

template <int MODE>
__global__ void __launch_bounds__(kStreamThreads, 1)
stream_kernel(const __grid_constant__ CUtensorMap tm_res, const __grid_constant__ CUtensorMap tm_x,
              const __grid_constant__ CUtensorMap tm_rout, const __grid_constant__ CUtensorMap tm_li,
              const StreamArgs a, int n_slices, int n_items) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t bars = base + kBarOff;
    auto full = [&](int st) { return bars + 8u * st; };
    auto ready = [&](int st) { return bars + 8u * (kStages + st); };
    auto mma_done = [&](int st) { return bars + 8u * (2 * kStages + st); };
    auto acc_full = [&](int b) { return bars + 8u * (3 * kStages + b); };
    auto acc_empty = [&](int b) { return bars + 8u * (3 * kStages + 2 + b); };
    auto ssq_full = [&](int b) { return bars + 8u * (3 * kStages + 4 + b); };
    auto ssq_empty = [&](int b) { return bars + 8u * (3 * kStages + 6 + b); };
    float *ssq_x = reinterpret_cast<float *>(gbase + kSsqOff);   // [b][0: ssq, 1: ssql][t]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + kMiscOff + 16);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int d = a.slice_w / kChunk;                               // chunks per item
    const int n_local = (n_items - static_cast<int>(blockIdx.x) + gridDim.x - 1) / gridDim.x;
    const int total = n_local * d;                                   // chunks of this CTA
    const uint64_t tmo = a.timeout_ns;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(full(i), 1);
            mbar_init(ready(i), 8);
            mbar_init(mma_done(i), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full(b), 1);
            mbar_init(acc_empty(b), 4);
            mbar_init(ssq_full(b), 4);
            mbar_init(ssq_empty(b), 4);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_addr(tmem_slot), 2 * kAccCols);
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
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            const uint64_t pol_stream = policy_evict_first();
            const uint64_t pol_keep = policy_evict_last();
            constexpr uint32_t kLoadBytes =
                kResBytes + kWBytes + (MODE != PRE_ONLY ? kXBytes : 0);
            auto issue_load = [&](int g) {
                const int st = g % kStages;
                const uint32_t sb = base + st * kStageBytes;
                const Item it = item_of(g / d, n_slices);
                const int hc = chunk_hidden(it.slice, g % d, n_slices);
                const int t0 = it.tile * kTileT;
                mbar_arrive_expect_tx(full(st), kLoadBytes);
                tma_load_3d(sb, &tm_res, hc, t0, 0, full(st), pol_stream);
                if (MODE != PRE_ONLY) tma_load_2d(sb + kResBytes, &tm_x, hc, t0, full(st), pol_stream);
                bulk_load(sb + kResBytes + kXBytes,
                          a.weight + static_cast<size_t>(hc / kChunk) * kWBytes, kWBytes,
                          full(st), pol_keep);
            };
            int loaded = 0;
            for (; loaded < total && loaded < kStages; ++loaded) issue_load(loaded);
            int g = 0;
            for (; g < total; ++g) {
                const int st = g % kStages;
                const uint32_t ph = (g / kStages) & 1;
                if (!mbar_wait(ready(st), ph, abort_flag, tmo, a.status, SITE_PROD_READY)) break;
                if (MODE != PRE_ONLY) {
                    const uint32_t sb = base + st * kStageBytes;
                    const Item it = item_of(g / d, n_slices);
                    const int hc = chunk_hidden(it.slice, g % d, n_slices);
                    const int t0 = it.tile * kTileT;
                    tma_store_3d(&tm_rout, hc, t0, 0, sb, pol_stream);
                    // the collapse is re-read by the finishing kernel: keep it in L2
                    if (MODE == FUSED_SHIFTED) tma_store_2d(&tm_li, hc, t0, sb + kResBytes, pol_keep);
                    bulk_commit();
                }
                // refill the stage of the previous chunk: its stores have had a
                // whole chunk to read shared memory
                if (g >= 1 && loaded < total) {
                    const int gp = g - 1;
                    if (MODE != PRE_ONLY) bulk_wait_read_allbut1();
                    if (!mbar_wait(mma_done(gp % kStages), (gp / kStages) & 1, abort_flag, tmo,
                                   a.status, SITE_PROD_MMA))
                        break;
                    issue_load(loaded);
                    ++loaded;
                }
            }
            bulk_wait_all();
            if (g < total) {  // aborted: let the loads in flight land before exiting
                for (int c = g; c < loaded; ++c)
                    drain_wait(full(c % kStages), (c / kStages) & 1, tmo, a.status);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            constexpr uint32_t kIdesc = idesc_bf16_f32(kTileT, kWRows);
            int issued = 0;
            for (int g = 0; g < total; ++g) {
                const int st = g % kStages;
                const uint32_t ph = (g / kStages) & 1;
                const int k = g / d, c = g % d, b = k & 1;
                if (c == 0 && k >= 2 &&
                    !mbar_wait(acc_empty(b), ((k >> 1) + 1) & 1, abort_flag, tmo, a.status,
                               SITE_MMA_ACC))
                    break;
                if (!mbar_wait(full(st), ph, abort_flag, tmo, a.status, SITE_MMA_FULL)) break;
                if (!mbar_wait(ready(st), ph, abort_flag, tmo, a.status, SITE_MMA_READY)) break;
                tc_fence_after();
                const uint32_t sb = base + st * kStageBytes;
                const uint32_t dcol = tmem_base + b * kAccCols;
#pragma unroll
                for (int s = 0; s < 4; ++s) {
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        const uint64_t ad =
                            smem_desc_sw64(sb + s * kTileT * kRowBytes + kk * 32, 8 * kRowBytes);
                        const uint64_t bd = smem_desc_sw64(
                            sb + kResBytes + kXBytes + s * kWRows * kRowBytes + kk * 32,
                            8 * kRowBytes);
                        tc_mma_bf16(dcol, ad, bd, kIdesc, (c | s | kk) != 0);
                    }
                }
                tc_commit(mma_done(st));
                if (c == d - 1) tc_commit(acc_full(b));
                issued = g + 1;
            }
            if (issued > 0 && issued < total) {  // aborted: let the issued MMAs finish
                const int c = issued - 1;
                drain_wait(mma_done(c % kStages), (c / kStages) & 1, tmo, a.status);
            }
        }
    } else {
        // ---------------------------------------------------- elementwise workers
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        const int t = q * 32 + lane;
        const uint32_t swz = (t >> 1) & 3;
        Coefs cf;
        bool valid = false;
        uint64_t ssq2 = 0, ssql2 = 0;
        float pend_ssq = 0.f, pend_ssql = 0.f;
        int pend_k = -1;
        bool aborted = false;

        // epilogue of item kp: 24 partial mixes (hi + lo) and the two partial
        // sums of squares per token, to the workspace; frees its accumulator.
        // Half 1 hands its sums to half 0 through shared memory buffer kp & 1,
        // guarded by mbarriers (bounded waits only, so an abort cannot strand
        // a warp at a barrier).
        auto epilogue = [&](int kp) {
            const int b = kp & 1;
            float *sx = ssq_x + b * 2 * kTileT;
            if (half == 1) {
                const bool free_ok = kp < 2 || mbar_wait(ssq_empty(b), ((kp >> 1) + 1) & 1,
                                                         abort_flag, tmo, a.status,
                                                         SITE_EPI_SSQ_FREE);
                if (free_ok) {
                    sx[t] = pend_ssq;
                    sx[kTileT + t] = pend_ssql;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(ssq_full(b));
                return;
            }
            const Item it = item_of(kp, n_slices);
            const long long gt = static_cast<long long>(it.tile) * kTileT + t;
            const bool got_ssq = mbar_wait(ssq_full(b), (kp >> 1) & 1, abort_flag, tmo, a.status,
                                           SITE_EPI_SSQ);
            const float ssq_other = sx[t], ssql_other = sx[kTileT + t];
            __syncwarp();
            if (lane == 0) mbar_arrive(ssq_empty(b));
            const bool ok = !aborted && got_ssq &&
                            mbar_wait(acc_full(b), (kp >> 1) & 1, abort_flag, tmo, a.status,
                                      SITE_EPI_ACC);
            tc_fence_after();
            uint32_t v[48];
            const uint32_t row = tmem_base + b * kAccCols + (static_cast<uint32_t>(q * 32) << 16);
            tmem_ld16(row + 0, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
            tmem_ld16(row + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
            tmem_ld16(row + 32, *reinterpret_cast<uint32_t(*)[16]>(&v[32]));
            tmem_ld_wait();
            tc_fence_before();
            if (gt < a.T && ok) {
                float out[kPartStride];
#pragma unroll
                for (int i = 0; i < 24; ++i)
                    out[i] = __uint_as_float(v[i]) + __uint_as_float(v[24 + i]);
                out[24] = pend_ssq + ssq_other;
                out[25] = pend_ssql + ssql_other;
                out[26] = 0.f;
                out[27] = 0.f;
                float4 *dst = reinterpret_cast<float4 *>(
                    a.partials + (static_cast<size_t>(it.slice) * a.T + gt) * kPartStride);
#pragma unroll
                for (int i = 0; i < kPartStride / 4; ++i)
                    dst[i] = make_float4(out[4 * i], out[4 * i + 1], out[4 * i + 2], out[4 * i + 3]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(b));
        };

        for (int g = 0; g < total; ++g) {
            const int st = g % kStages;
            const uint32_t ph = (g / kStages) & 1;
            const int k = g / d, c = g % d;
            if (c == 0) {
                // new item: park the previous item's sums, load this tile's coefficients
                if (k > 0) {
                    pend_ssq = f2_lo(ssq2) + f2_hi(ssq2);
                    pend_ssql = f2_lo(ssql2) + f2_hi(ssql2);
                    pend_k = k - 1;
                }
                ssq2 = 0;
                ssql2 = 0;
                const Item it = item_of(k, n_slices);
                const long long gt = static_cast<long long>(it.tile) * kTileT + t;
                valid = gt < a.T;
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
            }
            if (!mbar_wait(full(st), ph, abort_flag, tmo, a.status, SITE_WORK_FULL)) {
                aborted = true;
                break;
            }
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
            if (c == 0 && pend_k >= 0) {
                epilogue(pend_k);
                pend_k = -1;
            }
        }
        // the last item's epilogue (after an abort it only frees the warps)
        pend_ssq = f2_lo(ssq2) + f2_hi(ssq2);
        pend_ssql = f2_lo(ssql2) + f2_hi(ssql2);
        if (pend_k >= 0) epilogue(pend_k);   // aborted before the deferred point
        epilogue(n_local - 1);
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 2 * kAccCols);
    }
}

template <int MODE>
cudaError_t launch_t(const CUtensorMap &res, const CUtensorMap &x, const CUtensorMap &rout,
                     const CUtensorMap &li, const StreamArgs &a, int n_slices, int n_items,
                     int grid, cudaStream_t s) {
    constexpr int smem = kSmemUsed + 1024;
    auto kern = stream_kernel<MODE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kStreamThreads, smem, s>>>(res, x, rout, li, a, n_slices, n_items);
    return cudaGetLastError();
}

}  // namespace

size_t stream_smem_bytes() { return kSmemUsed + 1024; }

cudaError_t launch_stream(int mode, const CUtensorMap &res, const CUtensorMap &x,
                          const CUtensorMap &rout, const CUtensorMap &li, const StreamArgs &a,
                          int n_slices, int n_items, int grid, cudaStream_t s) {
    switch (mode) {
        case PRE_ONLY: return launch_t<PRE_ONLY>(res, x, rout, li, a, n_slices, n_items, grid, s);
        case FUSED_UNSHIFTED:
            return launch_t<FUSED_UNSHIFTED>(res, x, rout, li, a, n_slices, n_items, grid, s);
        case FUSED_SHIFTED:
            return launch_t<FUSED_SHIFTED>(res, x, rout, li, a, n_slices, n_items, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mhc
