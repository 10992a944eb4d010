// Shifted boundary of a decode batch (at most 64 tokens, one tile) on one
// thread-block cluster, the hidden dimension sliced across its CTAs and the
// slices' partial results exchanged through distributed shared memory
// ("mhc_boundary" page, MhcBoundaryKernel: hidden slices of one token tile in
// one cluster, partial mixes and sums of squares pushed to an owner CTA and
// summed in rank order). No workspace, no global flags: one kernel per call.
//
// CTA r of a cluster of C owns hidden chunks r, r + C, r + 2C, ... (nch chunks
// of 32). Per chunk, as in the streaming kernel: TMA-load the residual box
// [4 streams][rows][32] and the x box (rows = T rounded up to 8) and
// bulk-load the chunk's 12 KB prepared weight tile; a worker warp updates the
// residual in shared memory (the flush-to-zero FMA chain), folds the squares
// into per-token sums and writes the lagged collapse into a buffer of the CTA
// that outlives the stages; the producer TMA-stores the updated residual;
// four threads (one per stream, in four warps) issue the chunk's 8 tcgen05
// MMAs (M = 128 rows, of which the first T are tokens, N = 48 hi/lo weight
// rows) into four TMEM accumulators, one per stream, added at the end. The stages are
// packed by token rows (4 residual boxes, the x box, the weight tile), so at
// up to 8 tokens every chunk of a 14-chunk slice is resident at once and the
// producer sends every load during the set-up.
//
// Exchange: once the accumulator is complete each finisher thread (one per
// token) pushes its token's 24 partial mixes and partial 4H sum of squares to
// the token's owner CTA (token t belongs to rank t % C) with st.async, which
// completes bytes on the owner's mbarrier, and pushes its partial sum of
// squares of the collapse to every CTA. The owner adds the C records of each
// of its tokens in rank order and forms pre / post / comb (16 lanes per
// token); every CTA adds the C collapse sums of each token in rank order (the
// same order everywhere, so the same rstd_li) and writes its slice of the
// layer input. All reductions run in a fixed order: results are deterministic.
//
// Warps: 0 TMA producer and TMEM owner, 1-3 idle, 4-11 workers
// (worker warp w takes the chunks of stages w, w + 8, ... or, above 32
// tokens, token half w % 2 of the chunks of stages w / 2, w / 2 + 4, ...),
// 12-15 MMA issuers (stream warp % 4), then finishers (token 32 (warp % 4) +
// lane, the TMEM lane quarter of the warp). Every wait on a barrier is
// bounded; the two cluster barriers (after barrier initialisation, and before
// exit so that no CTA leaves while a peer may still write into its shared
// memory) are reached by every thread without any wait before them that is
// not bounded.
#include <atomic>

#include "coef.cuh"
#include "elementwise.cuh"
#include "mhc_internal.h"
#include "ptx.cuh"

namespace mhc {
namespace {

constexpr int kThreads = 512;
constexpr int kWorkThreads = 256;
constexpr int kFinThreads = 128;
constexpr int kFinBarrier = 1;
constexpr int kWorkBarrier = 2;
// One TMEM accumulator per residual stream (kAccCols columns each, 48 used),
// each fed by its own issuing warp (two MMAs per chunk); no fp32 accumulation
// chain is longer than 2 MMAs per chunk (1024 products at the most chunks);
// the finishers add the four in a fixed order.
constexpr int kAccs = 4;
constexpr int kEarlyLoads = 2;          // chunks whose loads go out during the set-up
constexpr int kAccCols = 64;
constexpr uint32_t kTmemCols = kAccs * kAccCols;
constexpr int kRegsProducer = 40, kRegsWorker = 184, kRegsFinisher = 96;
static_assert(128 * (kRegsProducer + kRegsFinisher) + 256 * kRegsWorker <= kThreads * 128,
              "register split exceeds the CTA's allocation (512 threads x 128 at launch)");

// Wait-site ids recorded with a timeout (distinct from the streaming kernel's).
enum : int { SITE_C_PROD_READY = 31, SITE_C_PROD_MMA = 32, SITE_C_MMA = 33, SITE_C_WORK_FULL = 34,
             SITE_C_FIN = 35, SITE_C_PART = 36, SITE_C_SQL = 37, SITE_C_DRAIN = 38 };

// ------------------------------------------------------------ cluster PTX
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The address of this CTA's shared-memory location `addr` in CTA `rank`'s
// shared memory (the cluster's shared window).
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(addr), "r"(rank));
    return d;
}
// Asynchronous store of 16 / 4 bytes into a peer's shared memory, completing
// that many bytes on the peer's mbarrier `rbar` once they have landed.
__device__ __forceinline__ void st_async_v4(uint32_t raddr, const uint4 &v, uint32_t rbar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
        ::"r"(raddr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(rbar) : "memory");
}
__device__ __forceinline__ void st_async_b32(uint32_t raddr, uint32_t v, uint32_t rbar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
                 ::"r"(raddr), "r"(v), "r"(rbar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
// Bounded wait for bytes pushed by peers (acquire at cluster scope).
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  volatile int *abort_flag, uint64_t timeout_ns,
                                                  unsigned int *status, int site) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > timeout_ns) {
            record_failure(status, 7, site);
            *abort_flag = 1;
            return false;
        }
    }
}

__device__ __forceinline__ void regs_dec_producer() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsProducer));
}
__device__ __forceinline__ void regs_inc_worker() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsWorker));
}
__device__ __forceinline__ void regs_dec_finisher() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsFinisher));
}

// Tokens of rank r among T tokens dealt round-robin to C ranks.
__device__ __forceinline__ int owned_tokens(int T, int C, int r) {
    return T > r ? (T - 1 - r) / C + 1 : 0;
}

__global__ void __launch_bounds__(kThreads, 1)
cluster_kernel(const __grid_constant__ CUtensorMap tm_res, const __grid_constant__ CUtensorMap tm_x,
               const __grid_constant__ CUtensorMap tm_rout, const ClusterArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int C = a.ctas, nch = a.nch, R = a.rows, NS = a.stages, T = a.T;
    const uint32_t rank = cluster_rank();
    const uint32_t SB = a.stage_bytes;
    const uint32_t res_bytes = 4u * R * kRowBytes;      // the four residual boxes
    const uint32_t x_bytes = static_cast<uint32_t>(R) * kRowBytes;
    const uint64_t tmo = a.timeout_ns;

    const uint32_t bars = base + a.bar_off;
    auto full = [&](int st) { return bars + 8u * st; };
    auto ready = [&](int st) { return bars + 8u * (kClusterMaxStages + st); };
    auto mma_done = [&](int st) { return bars + 8u * (2 * kClusterMaxStages + st); };
    const uint32_t acc_full = bars + 8u * (3 * kClusterMaxStages);
    const uint32_t sums_full = acc_full + 8u;
    const uint32_t part_bar = acc_full + 16u;          // owned tokens' records have landed
    const uint32_t sql_bar = acc_full + 24u;           // every CTA's collapse sums have landed
    const uint32_t exit_bar = acc_full + 32u;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + a.bar_off + 8 * (3 * kClusterMaxStages + 5));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 2);
    float *sums = reinterpret_cast<float *>(gbase + a.sums_off);     // [8][2][64]
    float *part = reinterpret_cast<float *>(gbase + a.part_off);     // [owned][C][28]
    float *sql = reinterpret_cast<float *>(gbase + a.sql_off);       // [C][T]
    float *red = reinterpret_cast<float *>(gbase + a.red_off);       // [16][25]
    float *consts = red + 16 * kPartVals;                             // [32]
    float *rstd_sh = consts + 32;                                     // [64]
    const int n_own = owned_tokens(T, C, static_cast<int>(rank));

    const uint64_t pol_load = policy_evict_normal();
    const uint64_t pol_keep = policy_evict_last();
    const uint32_t load_bytes = 5u * R * kRowBytes + kWBytes;
    auto hidden_of = [&](int c) { return (c * C + static_cast<int>(rank)) * kChunk; };
    auto issue_load = [&](int g) {
        const int st = g % NS;
        const uint32_t sb = base + st * SB;
        const int hc = hidden_of(g);
        mbar_arrive_expect_tx(full(st), load_bytes);
        // one box of [4 streams][R rows][32] lands as the four packed boxes
        tma_load_3d(sb, &tm_res, hc, 0, 0, full(st), pol_load);
        tma_load_2d(sb + res_bytes, &tm_x, hc, 0, full(st), pol_load);
        bulk_load(sb + res_bytes + x_bytes, a.weight + static_cast<size_t>(hc / kChunk) * kWBytes,
                  kWBytes, full(st), pol_keep);
    };

    // ---- set-up: thread 32 initialises the barriers, posts the bytes this
    // CTA will receive from its peers and sends the first loads while warp 0
    // allocates TMEM; the first 27 threads stage scale and base.
    if (tid == 32) {
        tma_prefetch_desc(&tm_res);
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_rout);
        for (int i = 0; i < NS; ++i) {
            mbar_init(full(i), 1);
            mbar_init(ready(i), T > 32 ? 2 : 1);    // the worker warps of the chunk
            mbar_init(mma_done(i), kAccs);           // one commit per issuing warp
        }
        mbar_init(acc_full, kAccs);
        mbar_init(sums_full, 8);
        mbar_init(part_bar, 1);
        mbar_init(sql_bar, 1);
        mbar_init(exit_bar, kThreads / 32);
        *abort_flag = 0;
        fence_mbar_init();
        // expected before any peer can push (the cluster barrier below)
        mbar_arrive_expect_tx(part_bar, static_cast<uint32_t>(n_own * C * kClusterRecFloats * 4));
        mbar_arrive_expect_tx(sql_bar, static_cast<uint32_t>(C * T * 4));
        // Launched as a programmatic dependent, the kernel may start while
        // the previous kernel on the stream still runs: until
        // griddepcontrol.wait nothing here reads global memory that kernel
        // might write, but the first chunks' weight tiles are prefetched
        // into L2 (a prefetch reads nothing into the CTA).
        for (int g = 0; g < nch && g < NS; ++g)
            bulk_prefetch_l2(a.weight + static_cast<size_t>(hidden_of(g) / kChunk) * kWBytes, kWBytes);
        griddep_wait();
        // the first two chunks' loads now; the producer sends the others
        // once the set-up is done (one thread issuing every copy held the
        // whole CTA's set-up back by ~2.5 us at 14 chunks)
        for (int g = 0; g < nch && g < kEarlyLoads; ++g) issue_load(g);
    }
    if (tid == 0) griddep_launch_dependents();
    // every global read below may depend on the previous kernel
    griddep_wait();
    if (tid < 27) stage_coef_consts(a.coef, consts, tid);
    __syncwarp();
    if (warp == 0) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    // worker lanes: the token they update and its coefficients (loaded now,
    // while the set-up runs). Up to 8 tokens four lanes share a token (one
    // 8-wide unit each), up to 16 two lanes (two units each), above that one
    // lane (four units); above 32 tokens the worker warps split by token half.
    const int ntg = T > 32 ? 2 : 1;
    const int wq = warp - 4;
    const int tg = ntg == 2 ? (wq & 1) : 0;
    const int lpt = T <= 8 ? 4 : (T <= 16 ? 2 : 1);    // lanes per token
    const int tpp = 32 / lpt;                          // tokens per warp
    const int upt = 4 / lpt;                           // units per lane
    const int wt_tok = 32 * tg + (lane % tpp);
    const int u0 = (lane / tpp) * upt;
    float4 pv = make_float4(0.f, 0.f, 0.f, 0.f), lv = pv;
    float4 cv[4] = {pv, pv, pv, pv};
    if (warp >= 4 && warp < 12 && wt_tok < T) {
        pv = __ldg(reinterpret_cast<const float4 *>(a.post) + wt_tok);
#pragma unroll
        for (int j = 0; j < 4; ++j) cv[j] = __ldg(reinterpret_cast<const float4 *>(a.comb) + wt_tok * 4 + j);
        lv = __ldg(reinterpret_cast<const float4 *>(a.pre_lag) + wt_tok);
    }
    cluster_arrive();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_wait();      // every CTA's barriers are initialised: peers may push
    const uint32_t tmem_base = *tmem_slot;

    if (warp < 4) {
        regs_dec_producer();
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------ TMA producer
            const uint64_t pol_out = policy_evict_first();
            const int first = nch < NS ? nch : NS;
            for (int g0 = kEarlyLoads; g0 < first; ++g0) issue_load(g0);
            int loaded = first;
            int g = 0;
            for (; g < nch; ++g) {
                const int st = g % NS;
                if (!mbar_wait(ready(st), (g / NS) & 1, abort_flag, tmo, a.status, SITE_C_PROD_READY))
                    break;
                const uint32_t sb = base + st * SB;
                tma_store_3d(&tm_rout, hidden_of(g), 0, 0, sb, pol_out);
                bulk_commit();
                // refill the stage of the previous chunk once its store has
                // read shared memory and its MMAs are done
                if (g >= 1 && loaded < nch) {
                    const int gp = g - 1;
                    bulk_wait_read_allbut1();
                    if (!mbar_wait(mma_done(gp % NS), (gp / NS) & 1, abort_flag, tmo, a.status,
                                   SITE_C_PROD_MMA))
                        break;
                    issue_load(loaded);
                    ++loaded;
                }
            }
            bulk_wait_all();
            if (g < nch)       // aborted: let the loads in flight land before exiting
                for (int c = g; c < loaded; ++c) {
                    int local = 0;
                    mbar_wait(full(c % NS), (c / NS) & 1, &local, tmo, a.status, SITE_C_DRAIN);
                }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(exit_bar);
        if (warp == 0) {
            int local = 0;
            mbar_wait(exit_bar, 0, &local, tmo, a.status, SITE_C_DRAIN);
            tc_fence_after();
            tmem_dealloc(tmem_base, kTmemCols);
        }
    } else if (warp < 12) {
        // ---------------------------------------------------- elementwise workers
        regs_inc_worker();
        const Coefs cf = coefs_of(pv, cv, lv);
        // a warp (a pair of warps, one per token half, above 32 tokens) owns
        // whole stages: stage st belongs to group st % groups, and a group
        // visits the chunks of its stages in increasing order, so that it
        // waits for the phases of each stage's barrier one after another
        // (a parity wait must never run two phases ahead)
        const int groups = 8 / ntg;
        const int grp = ntg == 2 ? (wq >> 1) : wq;
        const bool active = wt_tok < T;
        const uint32_t swz = (wt_tok >> 1) & 3;
        const uint32_t li_base = base + a.li_off;
        uint64_t sq = 0, sql2 = 0;
        bool ok = true;
        for (int c = 0; c < nch; ++c) {
            const int st = c % NS;
            if (st % groups != grp) continue;
            if (!mbar_wait(full(st), (c / NS) & 1, abort_flag, tmo, a.status, SITE_C_WORK_FULL)) {
                ok = false;
                break;
            }
            const uint32_t sb = base + st * SB;
            if (active) {
#pragma unroll 1
                for (int uu = 0; uu < upt; ++uu) {
                    const int u = u0 + uu;
                    const uint32_t off = wt_tok * kRowBytes + 16u * (u ^ swz);
                    uint4 r[4], cur[4];
#pragma unroll
                    for (int s = 0; s < 4; ++s) r[s] = ld_shared_v4(sb + s * R * kRowBytes + off);
                    update8(r, ld_shared_v4(sb + res_bytes + off), cf, cur);
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        st_shared_v4(sb + s * R * kRowBytes + off, cur[s]);
                        sq_accum(cur[s], sq);
                    }
                    const uint4 li = collapse8(cur, cf);
                    sq_accum(li, sql2);
                    // the collapse, unswizzled: [chunk][token][32]
                    st_shared_v4(li_base + (c * R + wt_tok) * kRowBytes + 16u * u, li);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(ready(st));
        }
        // per-token sums of this warp: the lanes of a token add theirs in a
        // fixed order, then [warp][0 ssq / 1 ssql][64 tokens] (zeros for
        // tokens this warp does not handle)
        float s0 = f2_lo(sq) + f2_hi(sq), s1 = f2_lo(sql2) + f2_hi(sql2);
        for (int m = tpp; m < 32; m <<= 1) {
            s0 += __shfl_xor_sync(0xffffffffu, s0, m);
            s1 += __shfl_xor_sync(0xffffffffu, s1, m);
        }
        const bool rep = lane < tpp;
        float *sw = sums + wq * 2 * kClusterMaxTokens;
        sw[lane] = tg == 0 && rep ? s0 : 0.f;
        sw[32 + lane] = tg == 1 && rep ? s0 : 0.f;
        sw[kClusterMaxTokens + lane] = tg == 0 && rep ? s1 : 0.f;
        sw[kClusterMaxTokens + 32 + lane] = tg == 1 && rep ? s1 : 0.f;
        __syncwarp();
        if (lane == 0) mbar_arrive(sums_full);

        // ---- coefficients of the tokens this CTA owns (t = rank + C j): the
        // C records of each are added in rank order, then 16 lanes per token
        // form pre / post / comb. Rounds of up to 16 tokens; every worker warp
        // takes part in each barrier.
        const int wt = tid - 4 * 32;
        ok = __all_sync(0xffffffffu, ok);
        if (n_own > 0)
            ok = __all_sync(0xffffffffu, mbar_wait_cluster(part_bar, 0, abort_flag, tmo, a.status,
                                                           SITE_C_PART) && ok);
        for (int j0 = 0; j0 < n_own; j0 += 16) {
            const int n = n_own - j0 < 16 ? n_own - j0 : 16;
            for (int p = wt; p < n * kPartVals; p += kWorkThreads) {
                const int j = p / kPartVals, m = p - j * kPartVals;
                const float *rec = part + static_cast<size_t>(j0 + j) * C * kClusterRecFloats + m;
                float acc = 0.f;
                for (int src = 0; src < C; ++src) acc += rec[src * kClusterRecFloats];
                red[p] = acc;
                // the token's reduced values, kept in the caller's scratch
                if (a.mix_out != nullptr)
                    a.mix_out[(static_cast<long long>(rank) + static_cast<long long>(C) * (j0 + j)) *
                                  kClusterRecFloats + m] = acc;
            }
            named_barrier_sync(kWorkBarrier, kWorkThreads);
            const int jl = 2 * wq;
            if (ok && jl < n) {
                const long long t_lo = static_cast<long long>(rank) + static_cast<long long>(C) * (j0 + jl);
                coefficients_16lanes(red + jl * kPartVals, red + (jl + 1) * kPartVals, 1, consts, a.coef,
                                     a.H, t_lo, t_lo + C, true, jl + 1 < n, a.pre_out, a.post_out,
                                     a.comb_out);
            }
            named_barrier_sync(kWorkBarrier, kWorkThreads);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(exit_bar);
    } else {
        // ---------------------------------------------------- finishers
        regs_dec_finisher();
        const int q = warp & 3;
        const int t = q * 32 + lane;
        const int ft = tid - 12 * 32;                  // 0..127 among the finishers
        // ---- MMA issue: lane 0 of finisher warp q issues stream q's two
        // MMAs of every chunk into accumulator q. One thread issues a
        // tcgen05.mma about every 80 ns whatever its shape, while several
        // warps issue concurrently, so the four streams go out in parallel.
        if (lane == 0) {
            constexpr uint32_t kIdesc = idesc_bf16_f32(kTileT, kWRows);
            const uint32_t dcol = tmem_base + q * kAccCols;
            int issued = 0;
            for (int g = 0; g < nch; ++g) {
                const int st = g % NS;
                const uint32_t ph = (g / NS) & 1;
                if (!mbar_wait(full(st), ph, abort_flag, tmo, a.status, SITE_C_MMA)) break;
                if (!mbar_wait(ready(st), ph, abort_flag, tmo, a.status, SITE_C_MMA)) break;
                tc_fence_after();
                const uint32_t sb = base + st * SB;
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    // A: 128 rows from stream q's box (rows past T are other
                    // data of the stage: their accumulator rows are never
                    // read); B: the stream's 48 weight rows
                    const uint64_t ad = smem_desc_sw64(sb + q * R * kRowBytes + kk * 32, 8 * kRowBytes);
                    const uint64_t bd = smem_desc_sw64(
                        sb + res_bytes + x_bytes + q * kWRows * kRowBytes + kk * 32, 8 * kRowBytes);
                    tc_mma_bf16(dcol, ad, bd, kIdesc, g | kk);
                }
                tc_commit(mma_done(st));
                if (g == nch - 1) tc_commit(acc_full);
                issued = g + 1;
            }
            if (issued > 0 && issued < nch) {
                int local = 0;
                const int c = issued - 1;
                mbar_wait(mma_done(c % NS), (c / NS) & 1, &local, tmo, a.status, SITE_C_DRAIN);
            }
        }
        __syncwarp();
        bool ok = mbar_wait(sums_full, 0, abort_flag, tmo, a.status, SITE_C_FIN);
        ok = mbar_wait(acc_full, 0, abort_flag, tmo, a.status, SITE_C_FIN) && ok;
        tc_fence_after();
        float ssq = 0.f, ssql = 0.f;
        if (t < kClusterMaxTokens) {
            for (int w2 = 0; w2 < 8; ++w2) {
                ssq += sums[w2 * 2 * kClusterMaxTokens + t];
                ssql += sums[(w2 * 2 + 1) * kClusterMaxTokens + t];
            }
        }
        // the four streams' accumulators, added as ((a0 + a1) + a2) + a3
        constexpr int nacc = kAccs;
        uint32_t v[48];
        const uint32_t acc = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll
        for (int b = 0; b < 3; ++b) {
            uint32_t w[16];
            tmem_ld16(acc + 16 * b, *reinterpret_cast<uint32_t(*)[16]>(&v[16 * b]));
            tmem_ld_wait();
#pragma unroll
            for (int k = 1; k < nacc; ++k) {
                tmem_ld16(acc + k * kAccCols + 16 * b, w);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    v[16 * b + i] = __float_as_uint(__uint_as_float(v[16 * b + i]) + __uint_as_float(w[i]));
            }
        }
        tc_fence_before();
        ok = __all_sync(0xffffffffu, ok);
        if (ok && t < T) {
            // the token's record to its owner: 24 partial mixes (hi + lo) and
            // the partial 4H sum of squares, at [t / C][this rank]
            // in place: v[0..23] = hi + lo, then v[24] = the sum of squares
            uint32_t *o = v;
#pragma unroll
            for (int i = 0; i < 24; ++i) o[i] = __float_as_uint(__uint_as_float(v[i]) + __uint_as_float(v[24 + i]));
            o[24] = __float_as_uint(ssq);
            o[25] = o[26] = o[27] = 0u;
            const uint32_t owner = static_cast<uint32_t>(t % C);
            const uint32_t dst = map_to_rank(
                base + a.part_off + ((t / C) * C + rank) * (kClusterRecFloats * 4), owner);
            const uint32_t rb = map_to_rank(part_bar, owner);
#pragma unroll
            for (int i = 0; i < kClusterRecFloats / 4; ++i)
                st_async_v4(dst + 16 * i, make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]), rb);
            // the collapse's partial sum of squares to every CTA, at [rank][t]
            const uint32_t loc = base + a.sql_off + (rank * T + t) * 4;
            for (int r2 = 0; r2 < C; ++r2)
                st_async_b32(map_to_rank(loc, r2), __float_as_uint(ssql), map_to_rank(sql_bar, r2));
        }
        // every CTA's collapse sums: rstd_li of each token (rank order)
        ok = __all_sync(0xffffffffu, mbar_wait_cluster(sql_bar, 0, abort_flag, tmo, a.status, SITE_C_SQL) && ok);
        if (ft < T) {
            float sl = 0.f;
            for (int r2 = 0; r2 < C; ++r2) sl += sql[r2 * T + ft];
            rstd_sh[ft] = rsqrtf(__fdiv_rn(sl, static_cast<float>(a.H)) + a.coef.norm_eps);
        }
        named_barrier_sync(kFinBarrier, kFinThreads);
        // the layer input of this CTA's slice: per (chunk, token, 16-wide half)
        const int per_chunk = 2 * T;
        const uint64_t pol_out = policy_evict_first();
        for (int idx = ft; ok && idx < nch * per_chunk; idx += kFinThreads) {
            const int c = idx / per_chunk, rem = idx - c * per_chunk;
            const int tk = rem >> 1, hh = rem & 1;
            const long long h0 = hidden_of(c) + 16 * hh;
            const uint32_t src = base + a.li_off + (c * R + tk) * kRowBytes + 32u * hh;
            const uint4 l0 = ld_shared_v4(src), l1 = ld_shared_v4(src + 16);
            const uint32_t w16[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
            uint32_t o[8];
            if (a.norm_w != nullptr) {
                const float r = rstd_sh[tk];
                float wv[16];
                if (a.nw_bf16) {
                    const uint16_t *wp = static_cast<const uint16_t *>(a.norm_w) + h0;
                    const uint4 a0 = ld_global_nc_v4(wp), a1 = ld_global_nc_v4(wp + 8);
                    const uint32_t ws[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                    for (int p = 0; p < 8; ++p) {
                        wv[2 * p] = __uint_as_float(ws[p] << 16);
                        wv[2 * p + 1] = __uint_as_float(ws[p] & 0xFFFF0000u);
                    }
                } else {
                    const float4 *wp = reinterpret_cast<const float4 *>(static_cast<const float *>(a.norm_w) + h0);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float4 w4 = __ldg(wp + j);
                        wv[4 * j] = w4.x; wv[4 * j + 1] = w4.y; wv[4 * j + 2] = w4.z; wv[4 * j + 3] = w4.w;
                    }
                }
#pragma unroll
                for (int p = 0; p < 8; ++p) {
                    const float lo = __fmul_rn(__fmul_rn(__uint_as_float(w16[p] << 16), r), wv[2 * p]);
                    const float hi = __fmul_rn(__fmul_rn(__uint_as_float(w16[p] & 0xFFFF0000u), r), wv[2 * p + 1]);
                    o[p] = bf2_pack_rn(f2_pack(lo, hi));
                }
            } else {
#pragma unroll
                for (int p = 0; p < 8; ++p) o[p] = w16[p];
            }
            uint16_t *dst = a.layer_input + static_cast<long long>(tk) * a.H + h0;
            const uint4 o0 = make_uint4(o[0], o[1], o[2], o[3]), o1 = make_uint4(o[4], o[5], o[6], o[7]);
            if (a.out32) {
                st_global_v8(dst, o0, o1, pol_out);
            } else {
                st_global_v4(dst, o0, pol_out);
                st_global_v4(dst + 8, o1, pol_out);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(exit_bar);
    }
    // no CTA leaves while a peer may still push into its shared memory
    __syncwarp();
    cluster_arrive();
    cluster_wait();
}

// The kernel's launch attributes (the largest dynamic shared memory, clusters
// of more than 8 CTAs) are set once per device.
bool set_attributes_once() {
    static std::atomic<unsigned long long> done{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    const unsigned long long bit = 1ull << dev;
    if (done.load(std::memory_order_acquire) & bit) return true;
    auto kern = cluster_kernel;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kClusterSmemMax) !=
            cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    done.fetch_or(bit, std::memory_order_release);
    return true;
}

}  // namespace

bool cluster_fits(int ctas, uint32_t smem) {
    // per device and cluster size: one bit per 4 KB step of shared memory for
    // "checked", one for "fits"
    static std::atomic<unsigned long long> checked[64][kClusterMaxCtas + 1];
    static std::atomic<unsigned long long> fits[64][kClusterMaxCtas + 1];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (ctas < 1 || ctas > kClusterMaxCtas || smem > static_cast<uint32_t>(kClusterSmemMax)) return false;
    const unsigned bucket = (smem + 4095u) / 4096u;         // at most 57 steps
    const unsigned long long bit = 1ull << bucket;
    if (checked[dev][ctas].load(std::memory_order_acquire) & bit)
        return (fits[dev][ctas].load(std::memory_order_acquire) & bit) != 0;
    if (!set_attributes_once()) return false;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(kThreads);
    const uint32_t rounded = bucket * 4096u;
    cfg.dynamicSmemBytes = rounded < static_cast<uint32_t>(kClusterSmemMax) ? rounded : kClusterSmemMax;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ctas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, cluster_kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    if (n >= 1) fits[dev][ctas].fetch_or(bit, std::memory_order_release);
    checked[dev][ctas].fetch_or(bit, std::memory_order_release);
    return n >= 1;
}

cudaError_t launch_cluster(const CUtensorMap &res, const CUtensorMap &x, const CUtensorMap &rout,
                           const ClusterArgs &a, cudaStream_t s) {
    auto kern = cluster_kernel;
    if (!set_attributes_once()) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.ctas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = a.smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = a.ctas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    int n = 1;
    // a programmatic dependent of the previous kernel on the stream (the
    // kernel waits for it before any read of global memory)
    if (a.pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, res, x, rout, a);
}

}  // namespace mhc
