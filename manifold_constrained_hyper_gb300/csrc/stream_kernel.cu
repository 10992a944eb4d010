// Streaming pass of the mHC boundary, persistent: one CTA per SM walks a
// static list of work items (a 128-token tile x a hidden slice) and runs one
// continuous chunk pipeline across them. Per 32-wide hidden chunk:
//   1. TMA-load the residual tile [4 streams][128 tokens][32] and the x tile
//      [128][32] (bf16, 64-byte swizzled rows) and bulk-load the chunk's
//      prepared weight tile [4][48][32] (already in swizzled order);
//   2. workers update the residual in shared memory (post: the flush-to-zero
//      FMA chain of the "mhc_boundary" page's residual_update) and fold the
//      squares of the updated values into per-token sums;
//   3. TMA-store the updated residual;
//   4. one thread issues 8 tcgen05 MMAs (M=128 tokens, N=48 stacked hi/lo
//      weight rows, K=16) accumulating the mixer contraction in TMEM.
// Slices interleave chunk by chunk and consecutive CTAs take the slices of
// one tile, so the CTAs of a tile read adjacent pieces of every row together
// (DRAM row locality). Each item accumulates into one of two TMEM buffers.
//
// Finisher warps take every item off the workers' path: they read its
// accumulator from TMEM and write the 24 partial mixes (hi + lo) and the
// partial sums of squares of each token to the workspace. In the shifted
// form ("mhc_boundary" page, lagged_collapse and layer_input_words) the
// workers also collapse the updated residual with the lagged pre into TMEM;
// the finishers publish the item with a per-call flag, wait until every
// slice of the tile has published, and write the layer input
// bf16((li * rsqrt(sum li^2 / H + eps)) * norm_w) from TMEM. The shifted form
// also forms the coefficients in this kernel, by its worker warps: when every
// CTA has a single item (a decode batch) as soon as the tile has published;
// otherwise once the CTA has streamed its last chunk, from partial records
// that bulk copies land in the then idle stage buffers (nothing of it runs
// while the CTA streams). The other forms leave the coefficients to a small
// kernel that reduces the partials.
//
// Warps: 0 TMA producer and TMEM owner, 1 MMA issuer, 2-3 idle (but warp 2
// of CTA 0, which advances a captured call's flag value), 4-11 workers
// (token 32*(warp%4) + lane, so a warp's tokens are its TMEM lane quarter;
// warps 4-7 take hidden 0-15 of a chunk, 8-11 hidden 16-31), 12-15
// finishers (token 32*(warp%4) + lane). Registers are redistributed per
// warpgroup with setmaxnreg: 40 + 184 + 184 + 96 per thread, 64,512 of the
// 65,536 the CTA is launched with (the workers measured 2 % slower at 168,
// the finishers 3 % at 88).
#include <atomic>

#include "coef.cuh"
#include "elementwise.cuh"
#include "mhc_internal.h"
#include "ptx.cuh"

namespace mhc {
namespace {

constexpr int kThreads = 512;
constexpr int kStages = kStreamStages;
// Template values of the decode variants (the decode worker mapping, chosen
// by the host through StreamArgs::decode_map) of the two fused forms: up to
// 32 tokens (quarter units) and 33 to kDecodeMaxTokens tokens (whole units).
// (The pre-only form has no update to spread: with the mapping its decode
// calls measured 0.1-0.35 us slower at hidden 7168, 1 to 64 tokens.)
constexpr int kShiftedDecode = 3;
constexpr int kShiftedDecodeHalf = 4;
constexpr int kUnshiftedDecode = 5;
constexpr int kUnshiftedDecodeHalf = 6;
constexpr int kBarOff = kStages * kStageBytes;
constexpr int kAccBufs = 2;                            // accumulator / sums buffers
constexpr int kLiBufs = 3;                             // shifted: collapse buffers
constexpr int kNumBars = 3 * kStages + 4 * kAccBufs + 3 + 1 + 1 + 4;
constexpr int kBarBytes = 256;
constexpr int kSumsOff = kBarOff + kBarBytes;          // [buffers][2 halves][2 sums][128] fp32
constexpr int kMiscOff = kSumsOff + kAccBufs * 2 * 2 * kTileT * 4;
// scratch: the workers' coefficient reduction [256] + [128], the finishers'
// collapse sums [128], the coefficient constants [32], each finisher warp's
// copy of its item's layer norm weights [4][8 chunks][32] (fp32)
constexpr int kRedOff = kMiscOff + 64;
constexpr int kWorkThreads = 256;
constexpr int kFinThreads = 128;
constexpr int kFinBarrier = 1;                         // named barrier of the finisher warps
constexpr int kWorkBarrier = 2;                        // named barrier of the worker warps
constexpr int kRsumOff = kWorkThreads + kFinThreads;   // float offsets within the scratch
constexpr int kConstOff = kRsumOff + kFinThreads;
constexpr int kNwOff = kConstOff + 32;
constexpr int kSmemUsed = kRedOff + (kNwOff + 4 * 8 * 32) * 4;
// shifted, several items per CTA: the coefficients are formed after the
// CTA's last item, from token groups' partial records [4][S][32] fp32 landed
// by bulk copies in the (then free) stage buffers
constexpr int kCoefGroup = 4;                          // tokens per group
constexpr int kCoefPairs = kCoefGroup * kPartVals;     // (token, value) pairs of a group
constexpr int kEndGroups = kWorkThreads / kCoefGroup;  // token groups per round at most
static_assert(8 * 2 * kDecodeMaxTokens <= kAccBufs * 2 * 2 * kTileT, "decode sums in the sums area");
static_assert(kRoundTok * kPartVals <= kFinThreads, "one combined value per thread");
static_assert(kSmemUsed + 1024 <= 227 * 1024, "shared memory per CTA");
constexpr int kAccCols = 64;                           // one accumulator buffer (48 used)
constexpr int kLiCol = kAccBufs * kAccCols;            // shifted: collapse buffers
constexpr int kLiCols = 128;                           // 8 chunks x 16 columns
constexpr int kRegsProducer = 40, kRegsWorker = 184, kRegsFinisher = 96;
static_assert(kNumBars * 8 <= kBarBytes, "barrier area");
static_assert(128 * (kRegsProducer + kRegsFinisher) + 256 * kRegsWorker <= kThreads * 128,
              "register split exceeds the CTA's allocation (512 threads x 128 at launch)");

// Wait-site ids recorded with a timeout.
enum : int { SITE_PROD_READY = 1, SITE_PROD_MMA = 2, SITE_MMA_FULL = 3, SITE_MMA_READY = 4,
             SITE_WORK_FULL = 5, SITE_FIN_ACC = 6, SITE_DRAIN = 7, SITE_MMA_ACC = 8,
             SITE_FIN_SUMS = 9, SITE_WORK_SUMS = 10, SITE_TILE_FLAGS = 11, SITE_WORK_LI = 12,
             SITE_WORK_COEF = 14, SITE_EPOCH = 15 };

// AND of `v` over the 256 worker threads (named barrier kWorkBarrier = 2);
// every worker warp must call it.
__device__ __forceinline__ bool workers_and(bool v) {
    uint32_t r;
    __syncwarp();
    asm volatile(
        "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.and.pred q, 2, 256, p;\n"
        "selp.u32 %0, 1, 0, q;\n}"
        : "=r"(r) : "r"(static_cast<uint32_t>(v)) : "memory");
    return r != 0;
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

// Bounded wait that ignores the abort flag (drains copies in flight before
// the CTA exits after an abort).
__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                           unsigned int *status) {
    int local = 0;
    return mbar_wait(bar, parity, &local, timeout_ns, status, SITE_DRAIN);
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
__global__ void __launch_bounds__(kThreads, 1)
stream_kernel(const __grid_constant__ CUtensorMap tm_res, const __grid_constant__ CUtensorMap tm_x,
              const __grid_constant__ CUtensorMap tm_rout, const StreamArgs a, int n_slices,
              int n_items) {
    constexpr bool kDecodeMap = MODE >= kShiftedDecode;
    // the form (PRE_ONLY, FUSED_UNSHIFTED or FUSED_SHIFTED) and, for the decode
    // variants, whether tokens 33 to 64 are mapped (whole units per lane)
    constexpr int kBase = !kDecodeMap ? MODE : (MODE <= kShiftedDecodeHalf ? FUSED_SHIFTED : FUSED_UNSHIFTED);
    constexpr bool kHalfMap = MODE == kShiftedDecodeHalf || MODE == kUnshiftedDecodeHalf;
    constexpr bool kShifted = kBase == FUSED_SHIFTED;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t bars = base + kBarOff;
    auto full = [&](int st) { return bars + 8u * st; };
    auto ready = [&](int st) { return bars + 8u * (kStages + st); };
    auto mma_done = [&](int st) { return bars + 8u * (2 * kStages + st); };
    auto acc_full = [&](int b) { return bars + 8u * (3 * kStages + b); };
    auto acc_empty = [&](int b) { return bars + 8u * (3 * kStages + kAccBufs + b); };
    auto sums_full = [&](int b) { return bars + 8u * (3 * kStages + 2 * kAccBufs + b); };
    auto sums_empty = [&](int b) { return bars + 8u * (3 * kStages + 3 * kAccBufs + b); };
    auto li_empty = [&](int b) { return bars + 8u * (3 * kStages + 4 * kAccBufs + b); };
    const uint32_t exit_bar = bars + 8u * (3 * kStages + 4 * kAccBufs + kLiBufs);   // every warp is done
    const uint32_t coef_go = exit_bar + 8u;   // single wave: the tile's partials are all published
    // several items: the producer's copies have left the stage buffers;
    // every finisher warp has seen the tiles of the CTA's items
    // 0..n_early-1 (prev_go) and of its last item (end_go) published; a
    // round's partial records have landed (end_full)
    const uint32_t stages_free = coef_go + 8u;
    const uint32_t prev_go = stages_free + 8u;
    const uint32_t end_go = prev_go + 8u;
    const uint32_t end_full = end_go + 8u;
    // per-token sums of squares handed from workers to finishers: [b][half][ssq, ssql][t]
    float *sums = reinterpret_cast<float *>(gbase + kSumsOff);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + kMiscOff + 16);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int d = a.slice_w / kChunk;                               // chunks per item
    const int n_local = (n_items - static_cast<int>(blockIdx.x) + gridDim.x - 1) / gridDim.x;
    const int total = n_local * d;                                   // chunks of this CTA
    const uint64_t tmo = a.timeout_ns;

    // Loads of chunk g into its stage: residual and x with evict_normal
    // (measured: evict_first on these loads cost 14 % of the call at
    // 8192 x 7168, with the same DRAM bytes), the weight tile kept in L2.
    const uint64_t pol_load = policy_evict_normal();
    const uint64_t pol_keep = policy_evict_last();
    constexpr uint32_t kLoadBytes = kResBytes + kWBytes + (kBase != PRE_ONLY ? kXBytes : 0);
    // A call of one tile (box_rows != 0) loads only the first box_rows token
    // rows of each stream, one box per stream into the same place of the
    // stage: the copy engine spends time on every row of a box, filled or
    // not, and a decode batch has few tokens. Rows past box_rows keep stale
    // contents; they belong to tokens >= T, whose results are never used.
    const int box_rows = a.box_rows;
    const uint32_t load_bytes =
        box_rows == 0 ? kLoadBytes
                      : kWBytes + (kBase != PRE_ONLY ? 5u : 4u) * static_cast<uint32_t>(box_rows) * kRowBytes;
    auto issue_load = [&](int g) {
        const int st = g % kStages;
        const uint32_t sb = base + st * kStageBytes;
        const Item it = item_of(g / d, n_slices);
        const int hc = chunk_hidden(it.slice, g % d, n_slices);
        const int t0 = it.tile * kTileT;
        mbar_arrive_expect_tx(full(st), load_bytes);
        if (box_rows == 0) {
            tma_load_3d(sb, &tm_res, hc, t0, 0, full(st), pol_load);
        } else {
#pragma unroll
            for (int s = 0; s < 4; ++s)
                tma_load_3d(sb + s * kTileT * kRowBytes, &tm_res, hc, t0, s, full(st), pol_load);
        }
        if (kBase != PRE_ONLY) tma_load_2d(sb + kResBytes, &tm_x, hc, t0, full(st), pol_load);
        bulk_load(sb + kResBytes + kXBytes, a.weight + static_cast<size_t>(hc / kChunk) * kWBytes,
                  kWBytes, full(st), pol_keep);
    };

    // Set-up: lane 0 of warp 1 (the MMA issuer, idle until then) fetches the
    // tensor maps, initialises the barriers and, in a single wave, sends the
    // first loads, while warp 0 allocates TMEM (done in series on one warp,
    // the two took 1.2 us of a decode call).
    if (tid == 32) {
        tma_prefetch_desc(&tm_res);
        if (kBase != PRE_ONLY) { tma_prefetch_desc(&tm_x); tma_prefetch_desc(&tm_rout); }
        for (int i = 0; i < kStages; ++i) {
            mbar_init(full(i), 1);
            mbar_init(ready(i), 8);
            mbar_init(mma_done(i), kDecodeMap ? 4 : 1);   // decode: one commit per stream's issuer
        }
        for (int b = 0; b < kAccBufs; ++b) {
            mbar_init(acc_full(b), kDecodeMap ? 4 : 1);
            mbar_init(acc_empty(b), 4);
            mbar_init(sums_full(b), 8);
            mbar_init(sums_empty(b), 4);
        }
        for (int b = 0; b < kLiBufs; ++b) mbar_init(li_empty(b), 4);
        mbar_init(exit_bar, kThreads / 32);
        mbar_init(coef_go, 4);
        mbar_init(stages_free, 1);
        mbar_init(prev_go, 4);
        mbar_init(end_go, 4);
        mbar_init(end_full, 1);
        *abort_flag = 0;
        fence_mbar_init();
        // Launched as a programmatic dependent, the kernel may start while
        // the previous kernel on the stream still runs: until
        // griddepcontrol.wait nothing here reads global memory that kernel
        // might write, but when the CTA's chunks all fit the stages (a
        // single wave) their weight tiles are prefetched into L2 (a prefetch
        // reads nothing into the CTA). Longer calls skip it: it held the
        // first loads back by ~0.9 us at 8192 tokens, hidden 7168.
        for (int g = 0; total <= kStages && g < total; ++g) {
            const Item it = item_of(g / d, n_slices);
            bulk_prefetch_l2(a.weight + static_cast<size_t>(chunk_hidden(it.slice, g % d, n_slices) / kChunk) *
                                            kWBytes,
                             kWBytes);
        }
        griddep_wait();
        // the shifted form sends its first loads before the rest of the
        // set-up (the first stage landed ~3.5 us after the kernel started;
        // 0.4-0.9 us less from 768 to 8192 tokens at hidden 7168); the
        // unshifted forms keep them in the producer (their register
        // allocation spilled otherwise)
        if (kShifted)
            for (int g = 0; g < total && g < kStages; ++g) issue_load(g);
    }
    // decode variants: one accumulator per residual stream (4 x kAccCols)
    constexpr uint32_t kTmemCols = kShifted && !kDecodeMap ? 512 : (kDecodeMap ? 4 : kAccBufs) * kAccCols;
    static_assert(kAccBufs * kAccCols + kLiBufs * kLiCols <= 512, "TMEM columns");
    if (warp == 0) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    // the kernel launched after this one may start its blocks as soon as
    // SMs free up; it waits for this grid's completion itself
    if (tid == 0) griddep_launch_dependents();
    // every global read below may depend on the previous kernel
    griddep_wait();
    // the worker threads load the first item's coefficients of the previous
    // boundary now, while the set-up runs (at the start of the item their
    // latency delayed a decode call's first chunk by ~0.5 us)
    // (the decode mapping: token lane of the one tile)
    float4 pv0 = make_float4(0.f, 0.f, 0.f, 0.f), lv0 = pv0;
    float4 cv0[4] = {pv0, pv0, pv0, pv0};
    if (kBase != PRE_ONLY && warp >= 4 && warp < 12 && n_local > 0) {
        const long long gt0 = static_cast<long long>(item_of(0, n_slices).tile) * kTileT +
                              (kDecodeMap ? (kHalfMap ? ((warp - 4) & 1) * 32 : 0)
                                          : (warp & 3) * 32) + lane;
        if (gt0 < a.T) {
            pv0 = __ldg(reinterpret_cast<const float4 *>(a.post) + gt0);
#pragma unroll
            for (int j = 0; j < 4; ++j) cv0[j] = __ldg(reinterpret_cast<const float4 *>(a.comb) + gt0 * 4 + j);
            if (kShifted) lv0 = __ldg(reinterpret_cast<const float4 *>(a.pre_lag) + gt0);
        }
    }
    // the finishers' scale / base constants and (one thread) this call's
    // flag value, loaded now so that their latency passes during the set-up
    // (the decode variants' finisher warps issue the MMAs before they stage
    // them)
    float fin_const = 0.f;
    unsigned long long fin_epoch = 0;
    if (warp >= 12) {
        const int i = tid - 12 * 32;
        if (i < 3) fin_const = __ldg(a.coef.scale + i);
        else if (i < 27) fin_const = __ldg(a.coef.base + i - 3);
        if (tid == 12 * 32)
            fin_epoch = a.epoch_cell != nullptr
                            ? *reinterpret_cast<volatile const unsigned long long *>(a.epoch_cell) + 1
                            : a.epoch;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp < 4) {
        regs_dec_producer();
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------ TMA producer
            // (in the shifted form the first kStages loads went out right
            // after the barriers were initialised)
            const uint64_t pol_stream = policy_evict_first();
            int loaded = 0;
            if (kShifted)
                loaded = total < kStages ? total : kStages;
            else
                for (; loaded < total && loaded < kStages; ++loaded) issue_load(loaded);
            int g = 0;
            for (; g < total; ++g) {
                const int st = g % kStages;
                const uint32_t ph = (g / kStages) & 1;
                if (!mbar_wait(ready(st), ph, abort_flag, tmo, a.status, SITE_PROD_READY)) break;
                if (kBase != PRE_ONLY) {
                    const uint32_t sb = base + st * kStageBytes;
                    const Item it = item_of(g / d, n_slices);
                    const int hc = chunk_hidden(it.slice, g % d, n_slices);
                    if (box_rows == 0) {
                        tma_store_3d(&tm_rout, hc, it.tile * kTileT, 0, sb, pol_stream);
                    } else {
#pragma unroll
                        for (int s = 0; s < 4; ++s)
                            tma_store_3d(&tm_rout, hc, it.tile * kTileT, s, sb + s * kTileT * kRowBytes,
                                         pol_stream);
                    }
                    bulk_commit();
                }
                // refill the stage of the previous chunk: its store has had a
                // whole chunk to read shared memory
                if (g >= 1 && loaded < total) {
                    const int gp = g - 1;
                    if (kBase != PRE_ONLY) bulk_wait_read_allbut1();
                    if (!mbar_wait(mma_done(gp % kStages), (gp / kStages) & 1, abort_flag, tmo,
                                   a.status, SITE_PROD_MMA))
                        break;
                    issue_load(loaded);
                    ++loaded;
                }
            }
            bulk_wait_read_all();
            if (g < total) {  // aborted: let the loads in flight land before exiting
                for (int c = g; c < loaded; ++c)
                    drain_wait(full(c % kStages), (c / kStages) & 1, tmo, a.status);
            }
            // the stage buffers are free of this CTA's copies (the stores
            // have read them; their writes complete below)
            if (kShifted && a.coef_end) mbar_arrive(stages_free);
            bulk_wait_all();
        } else if (warp == 1 && lane == 0 && !kDecodeMap) {
            // ------------------------------------------------ MMA issuer
            constexpr uint32_t kIdesc = idesc_bf16_f32(kTileT, kWRows);
            int issued = 0;
            for (int g = 0; g < total; ++g) {
                const int st = g % kStages;
                const uint32_t ph = (g / kStages) & 1;
                const int k = g / d, c = g % d, b = k % kAccBufs;
                if (c == 0 && k >= kAccBufs &&
                    !mbar_wait(acc_empty(b), ((k / kAccBufs) + 1) & 1, abort_flag, tmo, a.status,
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
        if (warp == 2 && a.bump_poll && blockIdx.x == 0) {
            // ------------------------------------------------ epoch advance
            // A captured call of several tiles. CTA b's first item is item b,
            // and the flag of its first token quarter (word 4b) is written by
            // the thread that read the cell, with the value derived from it:
            // once every CTA's is seen, no CTA of this call reads the cell
            // again, and it is advanced for the next replay.
            const unsigned long long e =
                *reinterpret_cast<volatile const unsigned long long *>(a.epoch_cell) + 1;
            const int nb = static_cast<int>(gridDim.x);
            bool done = false;
            uint64_t t_start = 0;
            for (;;) {
                unsigned long long v[kGridCap / 32 + 1];
#pragma unroll
                for (int i = 0; i <= kGridCap / 32; ++i)
                    v[i] = lane + 32 * i < nb ? flag_relaxed(a.flags + 4LL * (lane + 32 * i)) : e;
                bool seen = true;
#pragma unroll
                for (int i = 0; i <= kGridCap / 32; ++i) seen = seen && v[i] == e;
                if (__all_sync(0xffffffffu, seen)) {
                    done = true;
                    break;
                }
                if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
                const uint64_t now = __shfl_sync(0xffffffffu, globaltimer_ns(), 0);
                if (t_start == 0) {
                    t_start = now;
                } else if (now - t_start > tmo) {
                    if (lane == 0) record_failure(a.status, 7, SITE_EPOCH);
                    break;
                }
                nanosleep_ns(1000);
            }
            // after a failure: past every value this call may have used
            if (lane == 0) *reinterpret_cast<volatile unsigned long long *>(a.epoch_cell) = done ? e : e + 1;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(exit_bar);
        if (warp == 0) {
            // no warp touches TMEM any more: release it
            drain_wait(exit_bar, 0, tmo, a.status);
            tc_fence_after();
            tmem_dealloc(tmem_base, kTmemCols);
        }
    } else if (warp < 12) {
        // ---------------------------------------------------- elementwise workers
        regs_inc_worker();
        const int q = warp & 3;
        const int half = (warp - 4) >> 2;
        const int t = q * 32 + lane;
        const uint32_t swz = (t >> 1) & 3;
        const uint32_t li_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + kLiCol + half * 8;
        Coefs cf;
        bool valid = false;
        uint64_t ssq2 = 0, ssql2 = 0;

        // hand item kp's per-token sums to the finishers (buffer kp % kAccBufs)
        auto hand_over = [&](int kp) {
            const int b = kp % kAccBufs;
            if (kp >= kAccBufs)
                mbar_wait(sums_empty(b), ((kp / kAccBufs) + 1) & 1, abort_flag, tmo, a.status,
                          SITE_WORK_SUMS);
            float *sx = sums + (b * 2 + half) * 2 * kTileT;
            sx[t] = f2_lo(ssq2) + f2_hi(ssq2);
            sx[kTileT + t] = f2_lo(ssql2) + f2_hi(ssql2);
            if (kShifted) {
                tmem_st_wait();      // the item's collapse is in TMEM
                tc_fence_before();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(sums_full(b));
        };

        int g = 0;
        // ---- decode mapping (one tile of at most kDecodeMaxTokens tokens, one
        // item of at most kStages chunks, so no stage is refilled): the
        // elementwise work of a chunk is instruction-bound per warp, and with
        // the usual mapping only the warps of the first token quarter or two
        // have tokens. Here worker warp w' = warp - 4 takes hidden unit w' / 2
        // of every chunk: of token lane, pairs 2 (w' % 2) and 2 (w' % 2) + 1
        // (up to 32 tokens: a quarter of the usual work per thread), or whole
        // for token lane + 32 (w' % 2) (33 to 64 tokens: half). The shifted
        // form's collapse goes into the chunk's x tile (consumed by then, and
        // read by neither the copy out nor the MMA) instead of TMEM, whose
        // lane quarters belong to fixed warps; the finishers read it there.
        // The per-token sums of squares are handed over per warp.
        constexpr bool dmap = kDecodeMap;
        if (dmap && total > 0) {
            // up to 32 tokens: warp w' takes unit w' / 2, pair-half w' % 2, of
            // token lane; 33 to 64: unit w' / 2 whole, of token lane + 32 (w' % 2)
            constexpr bool quarter = !kHalfMap;
            const int wq = warp - 4, un = wq >> 1, pq = wq & 1;
            const int tt = quarter ? lane : lane + 32 * pq;
            const Coefs cd = coefs_of(pv0, cv0, lv0);      // token tt's, loaded in the set-up
            uint64_t sq = 0, sql = 0;
            for (; g < total; ++g) {
                const uint32_t sb = base + g * kStageBytes;
                if (!mbar_wait(full(g), 0, abort_flag, tmo, a.status, SITE_WORK_FULL)) break;
                if (tt < a.T) {
                    const uint32_t unit = tt * kRowBytes + 16u * (un ^ ((tt >> 1) & 3));
                    if (quarter) {
                        const uint32_t off = unit + 8u * pq;
                        uint2 r[4], cur[4];
#pragma unroll
                        for (int s2 = 0; s2 < 4; ++s2) r[s2] = ld_shared_v2(sb + s2 * kTileT * kRowBytes + off);
                        update4(r, ld_shared_v2(sb + kResBytes + off), cd, cur);
#pragma unroll
                        for (int s2 = 0; s2 < 4; ++s2) {
                            st_shared_v2(sb + s2 * kTileT * kRowBytes + off, cur[s2]);
                            sq_accum2(cur[s2], sq);
                        }
                        if (kShifted) {
                            const uint2 li = collapse4(cur, cd);
                            st_shared_v2(sb + kResBytes + off, li);
                            sq_accum2(li, sql);
                        }
                    } else {
                        uint4 r[4], cur[4];
#pragma unroll
                        for (int s2 = 0; s2 < 4; ++s2) r[s2] = ld_shared_v4(sb + s2 * kTileT * kRowBytes + unit);
                        update8(r, ld_shared_v4(sb + kResBytes + unit), cd, cur);
#pragma unroll
                        for (int s2 = 0; s2 < 4; ++s2) {
                            st_shared_v4(sb + s2 * kTileT * kRowBytes + unit, cur[s2]);
                            sq_accum(cur[s2], sq);
                        }
                        if (kShifted) {
                            const uint4 li = collapse8(cur, cd);
                            st_shared_v4(sb + kResBytes + unit, li);
                            sq_accum(li, sql);
                        }
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(ready(g));
            }
            // sums of warp w' for token t at [w'][0 / 1][t] of the item's sums
            // buffer; a warp that has no share of token t leaves zeros there
            sums[(wq * 2 + 0) * kDecodeMaxTokens + tt] = f2_lo(sq) + f2_hi(sq);
            sums[(wq * 2 + 1) * kDecodeMaxTokens + tt] = f2_lo(sql) + f2_hi(sql);
            sums[(wq * 2 + 0) * kDecodeMaxTokens + (tt ^ 32)] = 0.f;
            sums[(wq * 2 + 1) * kDecodeMaxTokens + (tt ^ 32)] = 0.f;
            __syncwarp();
            if (lane == 0) mbar_arrive(sums_full(0));
        }
        for (; !dmap && g < total; ++g) {
            const int st = g % kStages;
            const uint32_t ph = (g / kStages) & 1;
            const int k = g / d, c = g % d;
            if (c == 0) {
                // new item: hand over the previous item's sums, load this tile's coefficients
                if (k > 0) hand_over(k - 1);
                ssq2 = 0;
                ssql2 = 0;
                const Item it = item_of(k, n_slices);
                const long long gt = static_cast<long long>(it.tile) * kTileT + t;
                valid = gt < a.T;
                if (kBase != PRE_ONLY) {
                    // item 0's were loaded during the set-up
                    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
                    float4 pv = k == 0 ? pv0 : z;
                    float4 cv[4] = {k == 0 ? cv0[0] : z, k == 0 ? cv0[1] : z, k == 0 ? cv0[2] : z,
                                    k == 0 ? cv0[3] : z};
                    if (valid && k > 0) {
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
                if (kShifted) {
                    float4 lv = k == 0 ? lv0 : make_float4(0.f, 0.f, 0.f, 0.f);
                    if (valid && k > 0) lv = __ldg(reinterpret_cast<const float4 *>(a.pre_lag) + gt);
                    const float ls[4] = {lv.x, lv.y, lv.z, lv.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) cf.pre2[j] = f2_pack(ls[j], ls[j]);
                    // the finishers are done with the collapse buffer this item reuses
                    if (k >= kLiBufs) {
                        mbar_wait(li_empty(k % kLiBufs), ((k / kLiBufs) + 1) & 1, abort_flag, tmo,
                                  a.status, SITE_WORK_LI);
                        tc_fence_after();
                    }
                }
            }
            if (!mbar_wait(full(st), ph, abort_flag, tmo, a.status, SITE_WORK_FULL)) break;
            const uint32_t sb = base + st * kStageBytes;
            const uint32_t li_chunk = li_lane + (k % kLiBufs) * kLiCols + c * 16;
#pragma unroll
            for (int uu = 0; uu < 2; ++uu) {
                const int u = 2 * half + uu;
                const uint32_t off = t * kRowBytes + 16u * (u ^ swz);
                uint4 li = make_uint4(0u, 0u, 0u, 0u);
                if (valid) {
                    uint4 r[4];
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        r[s] = ld_shared_v4(sb + s * kTileT * kRowBytes + off);
                    if (kBase == PRE_ONLY) {
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
                        if (kShifted) {
                            li = collapse8(cur, cf);
                            sq_accum(li, ssql2);
                        }
                    }
                }
                // this thread's 8 collapse values of the unit, kept in TMEM
                if (kShifted) tmem_st4(li_chunk + 4 * uu, li);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(ready(st));
        }
        // the last item (after an abort the finishers only get their barriers)
        if (!dmap && total > 0) hand_over(g < total ? g / d : n_local - 1);

        // ---- several items per CTA: the coefficients of every token of the
        // CTA's items, formed by the workers once they have streamed their
        // last chunk and the producer's stores have read the stage buffers
        // (free from then on). Nothing of this runs while the CTA streams.
        // Token groups of 4 (tokens 4gi..4gi+3 of an item's tile, gi = slice,
        // slice + S, ...) go in rounds of up to kEndGroups: one bulk copy per
        // group lands its partial records [4 tokens][S slices][32] (contiguous
        // in the workspace) in its slot of the stage area; a thread per
        // (group, token, value) sums over the slices in slice order (a running
        // sum from zero, as every other path) and leaves the sum in place;
        // then a thread per token forms pre / post / comb. The groups of
        // items 0..n_early-1 (all but the last two items, or but the last one
        // for two items), whose tiles the finishers have seen published by
        // then (prev_go), are copied at once; those of the later items are
        // laid out in the same round where they fit and copied as soon as the
        // last tiles have published (polled by the workers; end_go for two
        // items), while the first copies are in flight, so that one
        // coefficient step serves both (a separate round
        // for the last item, gated on item n-2, left two in series: 1.7 us
        // more at 8192 x 7168, 4.4 us at 2048). Worker thread 0 lays out each
        // round in shared memory, so every worker warp takes part in each
        // barrier, also after an abort.
        if (kShifted && a.coef_end) {
            const int wt = tid - 4 * 32;                   // 0..255 among the workers
            bool ok = g == total && mbar_wait(stages_free, 0, abort_flag, tmo, a.status, SITE_WORK_COEF);
            ok = __all_sync(0xffffffffu, ok);
            int *rdesc = reinterpret_cast<int *>(gbase + kRedOff);   // count, then (tile, group)
            const float *consts = reinterpret_cast<const float *>(gbase + kRedOff) + kConstOff;
            const uint32_t grp_bytes = kCoefGroup * n_slices * kRecFloats * 4;
            const uint32_t slot = (grp_bytes + 127u) & ~127u;
            int per_round = static_cast<int>((kStages * kStageBytes) / slot);
            if (per_round > kEndGroups) per_round = kEndGroups;
            const uint64_t pol_once = policy_evict_first();
            // items [0, n_early) wait for prev_go, the rest for end_go
            const int n_early = n_local >= 3 ? n_local - 2 : n_local - 1;
            if (n_early > 0)
                ok = ok && mbar_wait(prev_go, 0, abort_flag, tmo, a.status, SITE_WORK_COEF);
            ok = workers_and(ok);
            bool late_seen = false;                        // end_go waited for
            int ck = 0, cg = item_of(0, n_slices).slice;   // thread 0: next (item, group)
            uint32_t round = 0;
            {
                for (;; ++round) {
                    if (wt == 0) {
                        int n = 0, n_a = -1;
                        while (ok && n < per_round && ck < n_local) {
                            const Item it = item_of(ck, n_slices);
                            if (cg < kTileT / kCoefGroup &&
                                static_cast<long long>(it.tile) * kTileT + kCoefGroup * cg < a.T) {
                                if (ck >= n_early && n_a < 0) n_a = n;
                                rdesc[1 + 2 * n] = it.tile;
                                rdesc[2 + 2 * n] = cg;
                                ++n;
                                cg += n_slices;
                            } else if (++ck < n_local) {
                                cg = item_of(ck, n_slices).slice;
                            }
                        }
                        rdesc[0] = n;
                        rdesc[200] = n_a < 0 ? n : n_a;
                        if (n > 0) mbar_arrive_expect_tx(end_full, n * grp_bytes);
                    }
                    named_barrier_sync(kWorkBarrier, kWorkThreads);
                    const int n = rdesc[0], n_a = rdesc[200];
                    named_barrier_sync(kWorkBarrier, kWorkThreads);   // rdesc[0] read by all
                    if (n == 0) break;
                    // the records were written by other CTAs' generic stores,
                    // acquired through the finishers (prev_go, end_go) or the
                    // workers' own polls; the groups of the last items go out
                    // once their tiles have published, while the earlier
                    // groups' copies are in flight
                    auto copy_group = [&](int i) {
                        const long long t0 = static_cast<long long>(rdesc[1 + 2 * i]) * kTileT +
                                             kCoefGroup * rdesc[2 + 2 * i];
                        fence_proxy_async_global();
                        bulk_load(base + i * slot, a.partials + t0 * n_slices * kRecFloats, grp_bytes,
                                  end_full, pol_once);
                    };
                    if (wt < n_a) copy_group(wt);
                    if (n_a < n) {
                        if (!late_seen && n_local >= 3) {
                            // the last items' tiles: every slice's quarter
                            // flags, polled by the workers themselves (the
                            // finishers see them only after L(n-2): 1.5 us
                            // later at 8192 x 7168); the flag value came
                            // with prev_go. (Two items: end_go, measured
                            // 0.3 us faster at 1024 tokens.)
                            const unsigned long long ep =
                                *reinterpret_cast<volatile const unsigned long long *>(gbase + kMiscOff + 48);
                            const int per_tile = n_slices * 4;
                            const int nt = (n_local - n_early) * per_tile;
                            uint64_t t_start = 0;
                            for (;;) {
                                bool seen = true;
                                for (int i = wt; i < nt; i += kWorkThreads) {
                                    const Item itk = item_of(n_early + i / per_tile, n_slices);
                                    seen = seen && flag_acquire(a.flags + static_cast<long long>(itk.tile) * per_tile +
                                                                i % per_tile) == ep;
                                }
                                if (workers_and(seen)) break;
                                if (!workers_and(!*abort_flag)) { ok = false; break; }
                                const uint64_t now = globaltimer_ns();
                                if (t_start == 0) t_start = now;
                                if (!workers_and(now - t_start <= tmo)) {
                                    if (wt == 0) {
                                        record_failure(a.status, 7, SITE_WORK_COEF);
                                        *abort_flag = 1;
                                    }
                                    ok = false;
                                    break;
                                }
                                nanosleep_ns(200);
                            }
                            ok = workers_and(ok);
                            late_seen = true;
                        }
                        if (!late_seen) {
                            ok = workers_and(ok && mbar_wait(end_go, 0, abort_flag, tmo, a.status,
                                                             SITE_WORK_COEF));
                            late_seen = true;
                        }
                        // (after an abort too: the expected bytes must land)
                        if (wt >= n_a && wt < n) copy_group(wt);
                    }
                    // the copies must land before the buffers are read or the
                    // CTA exits: a bounded wait that ignores aborts
                    drain_wait(end_full, round & 1, tmo, a.status);
                    for (int pr = wt; pr < n * kCoefPairs; pr += kWorkThreads) {
                        const int i = pr / kCoefPairs, r = pr - i * kCoefPairs;
                        const int q = r / kPartVals, m = r - q * kPartVals;
                        float *v = reinterpret_cast<float *>(gbase + i * slot) + q * n_slices * kRecFloats + m;
                        float acc = 0.f;
                        for (int s2 = 0; s2 < n_slices; ++s2) acc += v[s2 * kRecFloats];
                        v[0] = acc;                        // the token's value m, in place
                    }
                    named_barrier_sync(kWorkBarrier, kWorkThreads);
                    if (ok && wt < n * kCoefGroup) {
                        const int i = wt / kCoefGroup, q = wt - i * kCoefGroup;
                        const long long tok = static_cast<long long>(rdesc[1 + 2 * i]) * kTileT +
                                              kCoefGroup * rdesc[2 + 2 * i] + q;
                        if (tok < a.T)
                            coefficients_thread(reinterpret_cast<const float *>(gbase + i * slot) +
                                                    q * n_slices * kRecFloats,
                                                1, consts, a.coef, a.H, tok, a.pre_out, a.post_out,
                                                a.comb_out);
                    }
                    named_barrier_sync(kWorkBarrier, kWorkThreads);
                }
            }
        }

        // ---- one item per CTA (a single wave): once the finishers have seen
        // every slice of the tile publish, the workers form the coefficients
        // of the tile's tokens slice + S * j while the finishers write the
        // layer input. In rounds of up to kRoundTok tokens the 256 worker
        // threads split the (token, value) pairs and, when there are fewer
        // than 256 pairs, the slices into G consecutive ranges; each thread
        // sums its range in slice order (loads through L2 only: other CTAs
        // wrote the partials in this kernel); one thread per pair adds the G
        // range sums in range order; then one thread per token forms
        // pre / post / comb. The rounds and barriers depend on the item only,
        // so all eight worker warps take part in each.
        if (a.fuse_coef && n_local > 0) {
            const int wt = tid - 4 * 32;                   // 0..255 among the workers
            const Item it = item_of(0, n_slices);
            bool ok = mbar_wait(coef_go, 0, abort_flag, tmo, a.status, SITE_WORK_COEF);
            ok = __all_sync(0xffffffffu, ok);
            float *red = reinterpret_cast<float *>(gbase + kRedOff);
            const float *consts = red + kConstOff;
            const int ntok = it.slice < kTileT ? (kTileT - 1 - it.slice) / n_slices + 1 : 0;
            const long long gbase_t = static_cast<long long>(it.tile) * kTileT + it.slice;
            for (int r0 = 0; r0 < ntok; r0 += kRoundTok) {
                int nr = ntok - r0 < kRoundTok ? ntok - r0 : kRoundTok;
                while (nr > 0 && gbase_t + static_cast<long long>(n_slices) * (r0 + nr - 1) >= a.T) --nr;
                const int pairs = nr * kPartVals;
                const int G = pairs > 0 ? kWorkThreads / pairs : 1;
                const int per = (n_slices + G - 1) / G;
                if (ok && wt < pairs * G) {
                    const int gi = wt / pairs, pr = wt - gi * pairs;
                    const int j = pr / kPartVals, m = pr - j * kPartVals;
                    const int tin = it.slice + n_slices * (r0 + j);
                    const float *pp = a.partials + static_cast<size_t>(it.tile) * n_slices * kItemFloats +
                                      tin * kTokStride + m;
                    const size_t step = kItemFloats;
                    const int s_end = (gi + 1) * per < n_slices ? (gi + 1) * per : n_slices;
                    float sum = 0.f;
                    for (int s2 = gi * per; s2 < s_end; s2 += 32) {
                        float vv[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) vv[i] = s2 + i < s_end ? __ldcg(pp + (s2 + i) * step) : 0.f;
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (s2 + i < s_end) sum += vv[i];
                    }
                    red[wt] = sum;
                }
                named_barrier_sync(kWorkBarrier, kWorkThreads);
                // one thread per (token, value) adds the G range sums in order
                if (ok && wt < pairs) {
                    float acc = 0.f;
                    for (int gi = 0; gi < G; ++gi) acc += red[gi * pairs + wt];
                    red[kWorkThreads + wt] = acc;
                }
                named_barrier_sync(kWorkBarrier, kWorkThreads);
                // 16 lanes per token (two tokens per worker warp): the end of a
                // decode call waits on this, and one thread per token would
                // take about twice as long
                const int j0 = 2 * (warp - 4);
                if (ok && j0 < nr) {
                    const float *v = red + kWorkThreads + j0 * kPartVals;
                    const long long t_lo = gbase_t + static_cast<long long>(n_slices) * (r0 + j0);
                    coefficients_16lanes(v, v + kPartVals, 1, consts, a.coef, a.H, t_lo,
                                         t_lo + n_slices, true, j0 + 1 < nr, a.pre_out, a.post_out,
                                         a.comb_out);
                }
                named_barrier_sync(kWorkBarrier, kWorkThreads);
            }
            // ---- unshifted forms, one kernel: the owner CTA writes the
            // layer input of each token whose coefficients it formed. Its
            // worker threads recompute the token's updated residual over the
            // whole hidden dimension from the inputs (the same chain as the
            // streaming pass, so bit for bit the stored residual; pre-only:
            // the residual itself), collapse it with this boundary's pre
            // (written above by this CTA), add the collapse's squares in a
            // fixed order (per thread, then a warp tree, then the warps in
            // order) and normalise. No second kernel, and no exchange
            // between CTAs beyond the coefficients'.
            if (!kShifted && a.collapse_in_kernel) {
                float *wsum = red;                               // [8] warp sums
                const int units = a.H / 8;
                ok = workers_and(ok);                            // one verdict for every worker warp
                for (int j = 0; j < ntok; ++j) {
                    const long long tok = gbase_t + static_cast<long long>(n_slices) * j;
                    if (!ok || tok >= a.T) break;                // the same for every worker
                    const float4 pv = reinterpret_cast<const float4 *>(a.pre_out)[tok];
                    Coefs c;
                    const float ps4[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) c.pre2[i] = f2_pack(ps4[i], ps4[i]);
                    if (kBase != PRE_ONLY) {
                        const float4 qv = __ldg(reinterpret_cast<const float4 *>(a.post) + tok);
                        float4 cq[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) cq[i] = __ldg(reinterpret_cast<const float4 *>(a.comb) + tok * 4 + i);
                        const Coefs u = coefs_of(qv, cq, pv);
#pragma unroll
                        for (int i = 0; i < 4; ++i) c.post2[i] = u.post2[i];
#pragma unroll
                        for (int i = 0; i < 4; ++i)
#pragma unroll
                            for (int k2 = 0; k2 < 4; ++k2) c.comb2[i][k2] = u.comb2[i][k2];
                    }
                    uint4 lis[4];
                    uint64_t sq = 0;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int u = wt + kWorkThreads * k;
                        lis[k] = make_uint4(0u, 0u, 0u, 0u);
                        if (u < units) {
                            const long long h0 = 8LL * u;
                            uint4 r[4], cur[4];
#pragma unroll
                            for (int s2 = 0; s2 < 4; ++s2) r[s2] = ld_global_nc_v4(a.res_in + (tok * 4 + s2) * a.H + h0);
                            if (kBase != PRE_ONLY) {
                                update8(r, ld_global_nc_v4(a.x_in + tok * a.H + h0), c, cur);
                            } else {
#pragma unroll
                                for (int s2 = 0; s2 < 4; ++s2) cur[s2] = r[s2];
                            }
                            lis[k] = collapse8(cur, c);
                            sq_accum(lis[k], sq);
                        }
                    }
                    float sw = f2_lo(sq) + f2_hi(sq);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) sw += __shfl_xor_sync(0xffffffffu, sw, o);
                    if (lane == 0) wsum[warp - 4] = sw;
                    named_barrier_sync(kWorkBarrier, kWorkThreads);
                    float tot = 0.f;
#pragma unroll
                    for (int w2 = 0; w2 < kWorkThreads / 32; ++w2) tot += wsum[w2];
                    const float rstd_li = rsqrtf(__fdiv_rn(tot, static_cast<float>(a.H)) + a.coef.norm_eps);
                    uint16_t *row = a.layer_input + tok * a.H;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int u = wt + kWorkThreads * k;
                        if (u < units) {
                            const uint4 o = a.norm_w == nullptr
                                                ? lis[k]
                                                : norm8(lis[k], rstd_li, a.norm_w, a.nw_bf16, 8LL * u);
                            *reinterpret_cast<uint4 *>(row + 8LL * u) = o;
                        }
                    }
                    named_barrier_sync(kWorkBarrier, kWorkThreads);   // wsum reused
                }
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(exit_bar);
    } else {
        // ---------------------------------------------------- finishers
        regs_dec_finisher();
        const int q = warp & 3;
        if (kDecodeMap && lane == 0) {
            // ---- decode variants: lane 0 of finisher warp q issues stream q's
            // two MMAs of every chunk of the item into accumulator q (one
            // thread issues a tcgen05.mma about every 80 ns whatever its
            // shape, and several warps issue concurrently: the four streams
            // go out in parallel instead of one after another)
            constexpr uint32_t kIdesc = idesc_bf16_f32(kTileT, kWRows);
            const uint32_t dcol = tmem_base + q * kAccCols;
            int issued = 0;
            for (int g = 0; g < total; ++g) {
                if (!mbar_wait(full(g), 0, abort_flag, tmo, a.status, SITE_MMA_FULL)) break;
                if (!mbar_wait(ready(g), 0, abort_flag, tmo, a.status, SITE_MMA_READY)) break;
                tc_fence_after();
                const uint32_t sb = base + g * kStageBytes;
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const uint64_t ad = smem_desc_sw64(sb + q * kTileT * kRowBytes + kk * 32, 8 * kRowBytes);
                    const uint64_t bd = smem_desc_sw64(
                        sb + kResBytes + kXBytes + q * kWRows * kRowBytes + kk * 32, 8 * kRowBytes);
                    tc_mma_bf16(dcol, ad, bd, kIdesc, g | kk);
                }
                tc_commit(mma_done(g));
                if (g == total - 1) tc_commit(acc_full(0));
                issued = g + 1;
            }
            if (issued > 0 && issued < total)
                drain_wait(mma_done(issued - 1), 0, tmo, a.status);
        }
        __syncwarp();
        // this call's flag value: from the host, or (a call captured into a
        // CUDA graph) one more than the workspace cell's, which the call then
        // advances itself. One thread reads the cell and hands the value to
        // the other finishers, so the first flag this CTA publishes (written
        // by that thread) shows that the CTA is done with the cell.
        volatile unsigned long long *epoch_sh =
            reinterpret_cast<volatile unsigned long long *>(gbase + kMiscOff + 48);
        if (tid == 12 * 32) *epoch_sh = fin_epoch;
        float *red = reinterpret_cast<float *>(gbase + kRedOff);
        float *rsum = red + kRsumOff;
        float *consts = red + kConstOff;
        if (tid - 12 * 32 < 27) consts[tid - 12 * 32] = fin_const;   // scale[0..2], base[0..23]
        named_barrier_sync(kFinBarrier, kFinThreads);
        const unsigned long long epoch = *epoch_sh;
        const int t = q * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        const uint64_t pol_out = policy_evict_first();
        // Steps: publish item k (P k) as soon as its accumulator is ready;
        // write its layer input (L k) once the tile's other slices have
        // published too. In the order P0 P1 L0 P2 L1 ... P(n-2) L(n-3), an
        // item's siblings have almost always published by the time of its
        // L step, so the polls rarely wait (polling right after each P cost
        // 10 % of a long run). With three or more items the tail runs
        // P(n-1) L(n-2) L(n-1): the layer-input steps take most of an item's
        // time in a long call, so L(n-2) could not overlap the last item's
        // streaming and held its publication ~5 us after its last chunk.
        // With two items it runs L0 P1 L1, so that L0 overlaps item 1's
        // streaming (measured 2.3 us faster at 1024 tokens). Every wait points at an earlier tile or
        // at items the same wave streams without this CTA, so there is no
        // cycle. Iteration j runs P(pk) (if pk >= 0), then L(lk) (if lk >= 0);
        // the decode variants (one item) run P0 L0 in one iteration.
        const int n_iter = kDecodeMap ? 1 : n_local + 1;
        for (int j = 0; j < n_iter; ++j) {
            const bool tail_p_first = n_local >= 3;
            const int pk = kDecodeMap ? 0
                                      : tail_p_first ? (j < n_local ? j : -1)
                                                     : j < n_local - 1 ? j : (j == n_local ? n_local - 1 : -1);
            const int lk = kDecodeMap ? 0 : tail_p_first ? j - 1 : j < n_local ? j - 1 : n_local - 1;
            if (pk >= 0) {
                const int k = pk;
                const int b = k % kAccBufs;
                const uint32_t ph = (k / kAccBufs) & 1;
                const Item it = item_of(k, n_slices);
                const long long gt = static_cast<long long>(it.tile) * kTileT + t;
                // partial mixes and sums of squares of the item
                bool ok = mbar_wait(sums_full(b), ph, abort_flag, tmo, a.status, SITE_FIN_SUMS);
                ok = mbar_wait(acc_full(b), ph, abort_flag, tmo, a.status, SITE_FIN_ACC) && ok;
                tc_fence_after();
                float ssq = 0.f, ssql = 0.f;
                if (kDecodeMap) {
                    // the eight worker warps' sums, in warp order
                    if (t < kDecodeMaxTokens) {
                        for (int w2 = 0; w2 < 8; ++w2) {
                            ssq += sums[(w2 * 2 + 0) * kDecodeMaxTokens + t];
                            ssql += sums[(w2 * 2 + 1) * kDecodeMaxTokens + t];
                        }
                    }
                } else {
                    const float *s0 = sums + (b * 2 + 0) * 2 * kTileT;
                    const float *s1 = sums + (b * 2 + 1) * 2 * kTileT;
                    ssq = s0[t] + s1[t];
                    ssql = s0[kTileT + t] + s1[kTileT + t];
                }
                uint32_t v[48];
                const uint32_t acc = tmem_base + b * kAccCols + lane_off;
                tmem_ld16(acc + 0, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                tmem_ld16(acc + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
                tmem_ld16(acc + 32, *reinterpret_cast<uint32_t(*)[16]>(&v[32]));
                tmem_ld_wait();
                if (kDecodeMap) {
                    // the four streams' accumulators, added as ((a0 + a1) + a2) + a3
#pragma unroll
                    for (int s2 = 1; s2 < 4; ++s2) {
#pragma unroll
                        for (int blk = 0; blk < 3; ++blk) {
                            uint32_t w[16];
                            tmem_ld16(acc + s2 * kAccCols + 16 * blk, w);
                            tmem_ld_wait();
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                v[16 * blk + i] =
                                    __float_as_uint(__uint_as_float(v[16 * blk + i]) + __uint_as_float(w[i]));
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(sums_empty(b));
                    mbar_arrive(acc_empty(b));
                }
                ok = __all_sync(0xffffffffu, ok);
                if (ok && gt < a.T) {
                    float *rec = a.partials +
                                 (static_cast<size_t>(it.tile) * n_slices + it.slice) * kItemFloats;
                    if (a.fuse_coef) {
                        // token-major [128][28]: the workers of this CTA and the
                        // tile's other CTAs read a token's 25 values as one run
                        float4 *dst = reinterpret_cast<float4 *>(rec + t * kTokStride);
                        float o[kTokStride];
#pragma unroll
                        for (int i = 0; i < 24; ++i) o[i] = __uint_as_float(v[i]) + __uint_as_float(v[24 + i]);
                        o[24] = ssq;
                        o[25] = o[26] = o[27] = 0.f;
#pragma unroll
                        for (int i = 0; i < kTokStride / 4; ++i)
                            dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                    } else if (kShifted) {
                        // the token's 128-byte record of this slice: four 32-byte
                        // stores of whole sectors, kept in L2 for the end of the
                        // kernel (where a token group's records of every slice
                        // are one contiguous run)
                        float *dst = a.partials + (gt * n_slices + it.slice) * kRecFloats;
                        uint32_t o[kRecFloats];
#pragma unroll
                        for (int i = 0; i < 24; ++i) o[i] = __float_as_uint(__uint_as_float(v[i]) + __uint_as_float(v[24 + i]));
                        o[24] = __float_as_uint(ssq);
#pragma unroll
                        for (int i = 25; i < kRecFloats; ++i) o[i] = 0u;
#pragma unroll
                        for (int i = 0; i < kRecFloats / 8; ++i)
                            st_global_v8(dst + 8 * i, make_uint4(o[8 * i], o[8 * i + 1], o[8 * i + 2], o[8 * i + 3]),
                                         make_uint4(o[8 * i + 4], o[8 * i + 5], o[8 * i + 6], o[8 * i + 7]),
                                         pol_keep);
                    } else {
                        // value-major [25][128], kept in L2 for the kernel that
                        // reduces them next: a warp writes 128-byte rows
                        float *dst = rec + t;
#pragma unroll
                        for (int i = 0; i < 24; ++i)
                            st_global_f32(dst + i * kTileT,
                                          __uint_as_float(v[i]) + __uint_as_float(v[24 + i]), pol_keep);
                        st_global_f32(dst + 24 * kTileT, ssq, pol_keep);
                    }
                    // kept in L2 for the tile's layer-input steps (with the
                    // default policy these loads missed L2 under the
                    // streaming load: 1.2 us of a call at 8192 x 7168)
                    if (kShifted)
                        st_global_f32(a.ssql + static_cast<size_t>(it.slice) * a.T + gt, ssql, pol_keep);
                }
                // publish this quarter of the item to the tile's other slices
                // (a single wave: the whole item at once, after the four
                // finisher warps have written, with one flag; the unshifted
                // forms publish only then, for the in-kernel coefficients)
                if (kShifted || a.fuse_coef) {
                    unsigned long long *flag =
                        a.flags + (static_cast<long long>(it.tile) * n_slices + it.slice) * 4;
                    if (a.fuse_coef) {
                        named_barrier_sync(kFinBarrier, kFinThreads);
                        if (q == 0 && lane == 0) flag_release(flag, epoch);
                    } else {
                        __syncwarp();
                        if (lane == 0) flag_release(flag + q, epoch);
                    }
                }
            }
            if (lk < 0 || (!kShifted && !a.fuse_coef)) continue;

            // ---- layer input of item kn = lk (the unshifted forms: only the
            // wait for the tile, which releases the workers' coefficients)
            const int kn = lk, lb = kn % kLiBufs;
            const Item it = item_of(kn, n_slices);
            const long long gt = static_cast<long long>(it.tile) * kTileT + t;
            bool ok = __all_sync(0xffffffffu, !*abort_flag);
            // 32 hidden per chunk; lane l fetches norm weight l of the chunk
            // (one coalesced load per warp)
            auto nw_lane = [&](int c) -> float {
                if (a.norm_w == nullptr) return 0.f;
                const long long h = chunk_hidden(it.slice, c, n_slices) + lane;
                if (a.nw_bf16)
                    return __uint_as_float(static_cast<uint32_t>(
                                               __ldg(static_cast<const uint16_t *>(a.norm_w) + h))
                                           << 16);
                return __ldg(static_cast<const float *>(a.norm_w) + h);
            };
            // every chunk's weights (at most 8 chunks) are requested before
            // the wait for the tile, so that they arrive during it (waiting
            // for them first cost ~1 us of each layer-input step, 1.7 us of a
            // call at 8192 x 7168), and are parked in this warp's shared copy
            // after it, so that no registers are held across the sums of
            // squares below; the lanes then read them back as broadcasts,
            // four at a time
            float *nws = red + kNwOff + q * (8 * kChunk);
            float nwv[8];
            if (kShifted) {
#pragma unroll
                for (int c = 0; c < 8; ++c) nwv[c] = c < d ? nw_lane(c) : 0.f;
            }
            // every slice of the tile published. The layer RMSNorm needs the
            // flags of this warp's token quarter only: one acquire read per
            // slice, spread over the lanes. Forming the coefficients here
            // needs every quarter's flags: relaxed reads, all in flight, then
            // one acquire fence once the warp has seen them all.
            if (ok && (a.norm_w != nullptr || a.fuse_coef || a.coef_end)) {
                const unsigned long long *fl = a.flags + static_cast<long long>(it.tile) * n_slices * 4;
                const int nf = n_slices;
                uint64_t t_start = 0;
                // a single wave: warp 0 alone polls (every flag of the tile),
                // then hands the result to the other finisher warps through a
                // named barrier (fewer loads on the tile's few flag lines)
                while (!a.fuse_coef || q == 0) {
                    bool seen = true;
                    if (a.fuse_coef) {
                        for (int f0 = lane; f0 < nf; f0 += 32 * 8) {
                            unsigned long long v[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                v[i] = f0 + 32 * i < nf ? flag_relaxed(fl + 4 * (f0 + 32 * i)) : epoch;
#pragma unroll
                            for (int i = 0; i < 8; ++i) seen = seen && v[i] == epoch;
                        }
                    } else {
                        for (int f = lane; f < nf; f += 32)
                            seen = seen && flag_acquire(fl + 4 * f + q) == epoch;
                    }
                    if (__all_sync(0xffffffffu, seen)) break;
                    if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
                    // lane 0's clock, so that the whole warp takes the same branch
                    const uint64_t now = __shfl_sync(0xffffffffu, globaltimer_ns(), 0);
                    if (t_start == 0) {
                        t_start = now;
                    } else if (now - t_start > tmo) {
                        if (lane == 0) {
                            record_failure(a.status, 7, SITE_TILE_FLAGS);
                            *abort_flag = 1;
                        }
                        ok = false;
                        break;
                    }
                    if (!a.fuse_coef) nanosleep_ns(256);
                }
                if (a.fuse_coef && q == 0) fence_acq_rel_gpu();
                __syncwarp();
                // the tiles of items 0..kn have all published in full (each
                // finisher warp saw its quarter of each): the workers may
                // copy those items' partial records (prev_go: items
                // 0..n_early-1; end_go: every item)
                if (a.coef_end && ok && lane == 0) {
                    const int n_early = n_local >= 3 ? n_local - 2 : n_local - 1;
                    if (kn == n_local - 1) mbar_arrive(end_go);
                    else if (kn == n_early - 1) mbar_arrive(prev_go);
                }
            }
            if (kShifted) {
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    if (c < d) nws[c * kChunk + lane] = nwv[c];
                __syncwarp();
            }
            // a captured call of one tile: every CTA has read the cell once this
            // one has seen them all publish; advance it for the next replay
            // (past every value this call may have used, after an abort)
            if (a.bump_cell && blockIdx.x == 0 && q == 0 && lane == 0)
                *reinterpret_cast<volatile unsigned long long *>(a.epoch_cell) = ok ? epoch : epoch + 1;
            if (a.fuse_coef) {
                // warp 0's verdict, and (through the barrier) what it acquired
                volatile int *fin_ok = reinterpret_cast<volatile int *>(gbase + kMiscOff + 32);
                if (q == 0 && lane == 0) *fin_ok = ok ? 1 : 0;
                named_barrier_sync(kFinBarrier, kFinThreads);
                ok = ok && *fin_ok != 0;
            }
            // the workers may form the coefficients now (also after an abort,
            // so that their wait ends)
            if (a.fuse_coef && lane == 0) mbar_arrive(coef_go);
            // the unshifted forms' layer input needs this boundary's pre: a
            // kernel after this one writes it
            if (!kShifted) continue;
            float rstd_li = 0.f;
            if (a.fuse_coef) {
                // single wave: the 128 finisher threads share the reduction.
                // The tile's valid tokens, rounded up to a power of two (tvp),
                // each get G = 128 / tvp threads; thread i takes token i % tvp
                // and the i / tvp-th of G consecutive slice ranges, summed in
                // slice order; each token adds its G range sums in range
                // order. (With one thread per token a decode batch of a few
                // tokens left almost every lane idle, and a token's loads went
                // out one after another: 2.3 us at one token.)
                const long long tvl = a.T - static_cast<long long>(it.tile) * kTileT;
                const int tv = tvl >= kTileT ? kTileT : static_cast<int>(tvl);
                int tvp = 1;
                while (tvp < tv) tvp <<= 1;
                const int G = kFinThreads / tvp;
                const int ft = q * 32 + lane;
                const int tk = ft % tvp, sg = ft / tvp;
                float part = 0.f;
                if (ok && a.norm_w != nullptr && tk < tv) {
                    const int per = (n_slices + G - 1) / G;
                    const int s_beg = sg * per;
                    const int s_end = s_beg + per < n_slices ? s_beg + per : n_slices;
                    const float *pp = a.ssql + static_cast<long long>(it.tile) * kTileT + tk;
                    const size_t step = static_cast<size_t>(a.T);
                    for (int s2 = s_beg; s2 < s_end; s2 += 32) {
                        float vv[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) vv[i] = s2 + i < s_end ? __ldcg(pp + (s2 + i) * step) : 0.f;
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (s2 + i < s_end) part += vv[i];
                    }
                }
                rsum[ft] = part;
                named_barrier_sync(kFinBarrier, kFinThreads);
                if (ok && gt < a.T && a.norm_w != nullptr) {
                    float sl = 0.f;
                    for (int g = 0; g < G; ++g) sl += rsum[g * tvp + t];
                    rstd_li = rsqrtf(__fdiv_rn(sl, static_cast<float>(a.H)) + a.coef.norm_eps);
                }
            } else if (ok && gt < a.T && a.norm_w != nullptr) {
                // independent loads, added in slice order
                const float *pp = a.ssql + gt;
                const size_t step = static_cast<size_t>(a.T);
                float sl = 0.f;
                for (int s2 = 0; s2 < n_slices; s2 += 32) {
                    float vv[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) vv[i] = s2 + i < n_slices ? __ldcg(pp + (s2 + i) * step) : 0.f;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (s2 + i < n_slices) sl += vv[i];
                }
                rstd_li = rsqrtf(__fdiv_rn(sl, static_cast<float>(a.H)) + a.coef.norm_eps);
            }
            const uint32_t li = tmem_base + lane_off + kLiCol + lb * kLiCols;
            for (int c = 0; c < d; ++c) {
                uint32_t w16[16];
                if (kDecodeMap) {
                    // the collapse of chunk c sits in its stage's x tile, row t
                    const uint32_t row = base + c * kStageBytes + kResBytes + (t & (kTileT - 1)) * kRowBytes;
                    const uint32_t swt = (t >> 1) & 3;
#pragma unroll
                    for (int u2 = 0; u2 < 4; ++u2) {
                        const uint4 q4 = ld_shared_v4(row + 16u * (u2 ^ swt));
                        w16[4 * u2] = q4.x; w16[4 * u2 + 1] = q4.y;
                        w16[4 * u2 + 2] = q4.z; w16[4 * u2 + 3] = q4.w;
                    }
                } else {
                    tmem_ld16(li + c * 16, w16);
                    tmem_ld_wait();
                }
                const long long h0 = chunk_hidden(it.slice, c, n_slices);
                uint16_t *dst = a.layer_input + gt * a.H + h0;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {            // the two 16-wide halves
                    uint32_t o[8];
                    // the half's 16 norm weights, broadcast from the warp's copy
                    float wv[16];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float4 w4 = *reinterpret_cast<const float4 *>(nws + c * kChunk + 16 * hh + 4 * j);
                        wv[4 * j] = w4.x;
                        wv[4 * j + 1] = w4.y;
                        wv[4 * j + 2] = w4.z;
                        wv[4 * j + 3] = w4.w;
                    }
#pragma unroll
                    for (int p = 0; p < 8; ++p) {
                        const uint32_t wd = w16[8 * hh + p];
                        const float w_lo = wv[2 * p], w_hi = wv[2 * p + 1];
                        if (a.norm_w != nullptr) {
                            const float lo = __fmul_rn(__fmul_rn(__uint_as_float(wd << 16), rstd_li), w_lo);
                            const float hi =
                                __fmul_rn(__fmul_rn(__uint_as_float(wd & 0xFFFF0000u), rstd_li), w_hi);
                            o[p] = bf2_pack_rn(f2_pack(lo, hi));
                        } else {
                            o[p] = wd;
                        }
                    }
                    if (ok && gt < a.T) {
                        const uint4 o0 = make_uint4(o[0], o[1], o[2], o[3]);
                        const uint4 o1 = make_uint4(o[4], o[5], o[6], o[7]);
                        if (a.out32) {
                            st_global_v8(dst + 16 * hh, o0, o1, pol_out);
                        } else {
                            st_global_v4(dst + 16 * hh, o0, pol_out);
                            st_global_v4(dst + 16 * hh + 8, o1, pol_out);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(li_empty(lb));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(exit_bar);
    }
}

template <int MODE>
cudaError_t launch_t(const CUtensorMap &res, const CUtensorMap &x, const CUtensorMap &rout,
                     const StreamArgs &a, int n_slices, int n_items, int grid, cudaStream_t s) {
    constexpr int smem = kSmemUsed + 1024;
    auto kern = stream_kernel<MODE>;
    // the shared-memory opt-in is per device: set it once for each
    static std::atomic<unsigned long long> opted{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(opted.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        opted.fetch_or(bit, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    // the shifted form's CTAs wait on one another (and the unshifted forms'
    // when they form the coefficients): launch them co-resident
    if (MODE == FUSED_SHIFTED || (MODE >= kShiftedDecode && MODE <= kShiftedDecodeHalf) || a.fuse_coef) {
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n].val.cooperative = 1;
        ++n;
    }
    // a programmatic dependent of the previous kernel on the stream: its
    // set-up overlaps that kernel's end (the kernel waits for it before any
    // read of global memory)
    if (a.pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, res, x, rout, a, n_slices, n_items);
}

}  // namespace

size_t stream_smem_bytes() { return kSmemUsed + 1024; }

cudaError_t launch_stream(int mode, const CUtensorMap &res, const CUtensorMap &x,
                          const CUtensorMap &rout, const StreamArgs &a, int n_slices, int n_items,
                          int grid, cudaStream_t s) {
    switch (mode) {
        case PRE_ONLY: return launch_t<PRE_ONLY>(res, x, rout, a, n_slices, n_items, grid, s);
        case FUSED_UNSHIFTED:
            if (a.decode_map == 1)
                return launch_t<kUnshiftedDecode>(res, x, rout, a, n_slices, n_items, grid, s);
            if (a.decode_map == 2)
                return launch_t<kUnshiftedDecodeHalf>(res, x, rout, a, n_slices, n_items, grid, s);
            return launch_t<FUSED_UNSHIFTED>(res, x, rout, a, n_slices, n_items, grid, s);
        case FUSED_SHIFTED:
            if (a.decode_map == 1)
                return launch_t<kShiftedDecode>(res, x, rout, a, n_slices, n_items, grid, s);
            if (a.decode_map == 2)
                return launch_t<kShiftedDecodeHalf>(res, x, rout, a, n_slices, n_items, grid, s);
            return launch_t<FUSED_SHIFTED>(res, x, rout, a, n_slices, n_items, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mhc
