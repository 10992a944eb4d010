// Weight preparation, the standalone residual update, the finishing kernels
// of the boundary (slice reduction and coefficients; for the unshifted form
// the collapse and its RMSNorm after them), the device status word and the
// wait-timeout probe.
#include <atomic>

#include <cuda_bf16.h>

#include "coef.cuh"
#include "mhc_internal.h"
#include "ptx.cuh"

namespace mhc {

__device__ unsigned int g_status_word;

namespace {

// ------------------------------------------------------------ weight prep
// One thread per (chunk c, stream s, stacked row r, 8-wide unit u): TF32
// rounding (half away from zero on the bit pattern), exact bf16 hi/lo split
// ("mhc_boundary" page, prepare_boundary_weight), written to the 64-byte
// swizzled position of the (c, s) tile.
__global__ void prepare_weight_kernel(const float *__restrict__ fn, int H,
                                      uint8_t *__restrict__ out) {
    const long long total = static_cast<long long>(H / kChunk) * 4 * kWRows * 4;
    const long long K = 4LL * H;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int u = static_cast<int>(i % 4);
        const int r = static_cast<int>((i / 4) % kWRows);
        const int s = static_cast<int>((i / (4 * kWRows)) % 4);
        const long long c = i / (4 * kWRows * 4);
        const int row = r % 24;
        const bool lo_part = r >= 24;
        const long long k0 = static_cast<long long>(s) * H + c * kChunk + 8 * u;
        const float4 *src = reinterpret_cast<const float4 *>(fn + row * K + k0);
        const float4 a = src[0], b = src[1];
        const float w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t h[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float rt = __uint_as_float((__float_as_uint(w[e]) + 0x1000u) & 0xFFFFE000u);
            const __nv_bfloat16 hi = __float2bfloat16_rn(rt);
            if (!lo_part) {
                h[e] = __bfloat16_as_ushort(hi);
            } else {
                const float rest = __fsub_rn(rt, __bfloat162float(hi));
                h[e] = __bfloat16_as_ushort(__float2bfloat16_rn(rest));
            }
        }
        const uint4 v = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                                   h[6] | (h[7] << 16));
        const long long tile = c * 4 + s;
        uint4 *dst = reinterpret_cast<uint4 *>(out + (tile * kWRows + r) * kRowBytes +
                                               16 * (u ^ ((r >> 1) & 3)));
        *dst = v;
    }
}

// ------------------------------------------------------------ residual update
// Standalone post ("mhc_boundary" page, residual_update): one thread per
// (token, 8-wide hidden unit), 16-byte loads and stores, coefficients through
// the read-only path.
__global__ void post_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ res,
                            const float *__restrict__ post, const float *__restrict__ comb,
                            uint16_t *out, long long T, int H) {
    const int units = H / 8;
    const long long total = T * units;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long t = i / units;
        const int u = static_cast<int>(i % units);
        const float4 pv = __ldg(reinterpret_cast<const float4 *>(post) + t);
        float4 cv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) cv[j] = __ldg(reinterpret_cast<const float4 *>(comb) + t * 4 + j);
        uint4 r[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            r[j] = ld_global_nc_v4(res + (t * 4 + j) * H + 8LL * u);
        const uint4 xw = ld_global_nc_v4(x + t * H + 8LL * u);
        const uint32_t xs[4] = {xw.x, xw.y, xw.z, xw.w};
        const float ps[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const float cs[4] = {(&cv[0].x)[s], (&cv[1].x)[s], (&cv[2].x)[s], (&cv[3].x)[s]};
            uint32_t w[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                uint64_t nu = mul2_ftz(f2_pack(ps[s], ps[s]), bf2_unpack(xs[p]));
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t rw = (&r[j].x)[p];
                    nu = fma2_ftz(f2_pack(cs[j], cs[j]), bf2_unpack(rw), nu);
                }
                w[p] = bf2_pack_rn(nu);
            }
            *reinterpret_cast<uint4 *>(out + (t * 4 + s) * H + 8LL * u) =
                make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// ------------------------------------------------------------ coefficients
// 32 tokens (a quarter of a tile) per block. Warp m (m < 25) sums value m of
// the block's tokens over the hidden slices, lane = token, in slice order with
// every load in flight at once (each load a 128-byte row of the item's
// value-major partials); then warp 0 forms the 32 tokens' pre / post / comb,
// one thread per token. Launched as a programmatic dependent of the streaming
// kernel: blocks may start early and wait here for its completion.
constexpr int kCoefTokens = 32;
constexpr int kCoefThreads = kPartVals * 32;

__global__ void __launch_bounds__(kCoefThreads, 2) coefficients_kernel(const FinishArgs a) {
    __shared__ float red[kPartVals][kCoefTokens];
    __shared__ float consts[32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    stage_coef_consts(a.coef, consts, threadIdx.x);
    const long long t0 = static_cast<long long>(blockIdx.x) * kCoefTokens;
    const long long t = t0 + lane;
    const long long tile = t0 / kTileT;
    const int tin = static_cast<int>(t0 % kTileT) + lane;
    griddep_wait();
    if (t < a.T) {
        const float *p = a.partials + tile * a.n_slices * kItemFloats + warp * kTileT + tin;
        const long long step = kItemFloats;
        float v = 0.f;
        for (int s = 0; s < a.n_slices; s += 32) {
            float w[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) w[i] = s + i < a.n_slices ? __ldg(p + (s + i) * step) : 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (s + i < a.n_slices) v += w[i];
        }
        red[warp][lane] = v;
    }
    __syncthreads();
    if (warp == 0 && t < a.T)
        coefficients_thread(&red[0][lane], kCoefTokens, consts, a.coef, a.H, t, a.pre_out,
                            a.post_out, a.comb_out);
    // a collapse kernel launched as this kernel's programmatic dependent may
    // start once every block has written its tokens' coefficients
    griddep_launch_dependents();
}

// ------------------------------------------------------------ coefficients (split-K)
// The pure pre path's inputs ("The Hyper Connection Preprocessing GPU Kernel
// Study", square sum and RMSNorm with split-K): partial mixes dot_mix
// [S][T][24] and partial sums of squares sqrsum [S][T]. 32 tokens per block;
// thread p < 768 owns flat value p of the block's 32 x 24 mixes (consecutive
// threads read consecutive floats), threads 768..799 the 32 sums of squares;
// each sums its value over the splits in split order. Then warp 0 forms the
// coefficients, one thread per token.
__global__ void __launch_bounds__(kCoefThreads, 2)
coefficients_split_k_kernel(const float *__restrict__ dot_mix, const float *__restrict__ sqrsum,
                            int n_splits, const FinishArgs a) {
    __shared__ float red[kPartVals][kCoefTokens];
    __shared__ float consts[32];
    const int p = threadIdx.x, warp = p >> 5, lane = p & 31;
    const long long t0 = static_cast<long long>(blockIdx.x) * kCoefTokens;
    stage_coef_consts(a.coef, consts, p);
    const int j = p < 24 * kCoefTokens ? p / 24 : p - 24 * kCoefTokens;
    const int m = p < 24 * kCoefTokens ? p - 24 * j : 24;
    if (t0 + j < a.T) {
        const float *src = m < 24 ? dot_mix + t0 * 24 + p : sqrsum + t0 + j;
        const long long step = m < 24 ? a.T * 24 : a.T;
        float v = 0.f;
        for (int s = 0; s < n_splits; s += 16) {
            float w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = s + i < n_splits ? __ldg(src + (s + i) * step) : 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (s + i < n_splits) v += w[i];
        }
        red[m][j] = v;
    }
    __syncthreads();
    if (warp == 0 && t0 + lane < a.T)
        coefficients_thread(&red[0][lane], kCoefTokens, consts, a.coef, a.H, t0 + lane, a.pre_out,
                            a.post_out, a.comb_out);
    // the collapse kernel after it (a programmatic dependent) may start once
    // every block has written its tokens' coefficients
    griddep_launch_dependents();
}

// ------------------------------------------------------------ split-K pre, one kernel
// One 128-thread block per token. Warp 0 sums the token's splits (lanes 0-23
// the mixes, lane 24 the sum of squares), forms rstd and pre (lanes 0-3) and
// hands pre to warps 1-3, which collapse the token's 4 streams with it and
// write the RMS-normed layer input ("computing pre_mix early" on the page:
// the collapse needs pre only); meanwhile lane 0 of warp 0 forms post and
// the Sinkhorn comb. The coefficients' arithmetic and order are the
// two-kernel form's; the collapse's sum of squares is reduced in this
// kernel's own fixed order. THREADS: 128, or 512 when every token has an SM
// to itself (the collapse's loads then come from 15 warps instead of 3:
// 6.75 -> 4.94 us at 128 tokens, hidden 7168; with more tokens than SMs the
// wide blocks measured slower, 10.6 against 8.3 us at 512 tokens).
template <int THREADS>
__global__ void __launch_bounds__(THREADS)
pre_split_k_kernel(const float *__restrict__ dot_mix, const float *__restrict__ sqrsum,
                   int n_splits, const FinishArgs a) {
    constexpr int kSkCollapse = THREADS - 32;
    extern __shared__ uint4 li_s[];            // [H/8]
    __shared__ float vals[kPartVals];
    __shared__ float consts[32];
    __shared__ float pre_s[4];
    __shared__ float red_s[kSkCollapse / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long t = blockIdx.x;
    if (warp == 0) {
        stage_coef_consts(a.coef, consts, lane);
        float v = 0.f;
        if (lane < kPartVals) {
            const float *src = lane < 24 ? dot_mix + t * 24 + lane : sqrsum + t;
            const long long step = lane < 24 ? a.T * 24 : a.T;
            for (int s = 0; s < n_splits; s += 16) {
                float w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) w[i] = s + i < n_splits ? __ldg(src + (s + i) * step) : 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    if (s + i < n_splits) v += w[i];
            }
            vals[lane] = v;
        }
        __syncwarp();
        if (lane < 4) {
            const float rstd =
                rsqrtf(__fdiv_rn(vals[24], static_cast<float>(4 * a.H)) + a.coef.hc_norm_eps);
            pre_s[lane] = sigmoid_clamped(fmaf(v * rstd, consts[0], consts[3 + lane])) +
                          a.coef.hc_pre_eps;
        }
    }
    __syncthreads();
    if (warp == 0) {
        if (lane == 0)
            coefficients_thread(vals, 1, consts, a.coef, a.H, t, a.pre_out, a.post_out,
                                a.comb_out);
        return;
    }
    const int ct = tid - 32;
    const uint64_t p2[4] = {f2_pack(pre_s[0], pre_s[0]), f2_pack(pre_s[1], pre_s[1]),
                            f2_pack(pre_s[2], pre_s[2]), f2_pack(pre_s[3], pre_s[3])};
    const int units = a.H / 8;
    uint64_t sq2 = 0;
    for (int u = ct; u < units; u += kSkCollapse) {
        uint32_t cs[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 r = ld_global_nc_v4(a.cur + (t * 4 + j) * a.H + 8LL * u);
            cs[j][0] = r.x; cs[j][1] = r.y; cs[j][2] = r.z; cs[j][3] = r.w;
        }
        uint32_t w[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            uint64_t acc = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) acc = fma2(p2[j], bf2_unpack(cs[j][p]), acc);
            w[p] = bf2_pack_rn(acc);
            const uint64_t lv = bf2_unpack(w[p]);
            sq2 = fma2(lv, lv, sq2);
        }
        li_s[u] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    uint16_t *row = a.layer_input + t * a.H;
    if (a.norm_w == nullptr) {
        for (int u = ct; u < units; u += kSkCollapse)
            *reinterpret_cast<uint4 *>(row + 8LL * u) = li_s[u];
        return;
    }
    float sq = f2_lo(sq2) + f2_hi(sq2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    if (lane == 0) red_s[warp - 1] = sq;
    named_barrier_sync(1, kSkCollapse);
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kSkCollapse / 32; ++w) tot += red_s[w];
    const float rstd_li = rsqrtf(__fdiv_rn(tot, static_cast<float>(a.H)) + a.coef.norm_eps);
    for (int u = ct; u < units; u += kSkCollapse)
        *reinterpret_cast<uint4 *>(row + 8LL * u) =
            norm8(li_s[u], rstd_li, a.norm_w, a.nw_bf16, 8LL * u);
}

// ------------------------------------------------------------ collapse (unshifted)
// One 128-thread block per token, after the coefficients: collapse the
// token's 4 updated streams with this boundary's pre into shared memory,
// reduce the collapse's sum of squares in a fixed order, and write the
// normalised layer input.
// THREADS: 128, or 512 when every token has an SM of its own (a few tokens
// after a single wave: the loads then come from 16 warps instead of 4).
template <int THREADS>
__global__ void __launch_bounds__(THREADS) collapse_unshifted_kernel(const FinishArgs a) {
    constexpr int kColThreads = THREADS;
    extern __shared__ uint4 li_s[];            // [H/8]
    __shared__ float red_s[kColThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // last tokens first: the streaming pass touched them last, so part of
    // their rows is still in L2
    const long long t = a.T - 1 - blockIdx.x;
    // (a no-op unless launched as a programmatic dependent)
    griddep_wait();
    const float4 pv = reinterpret_cast<const float4 *>(a.pre_out)[t];
    const uint64_t p2[4] = {f2_pack(pv.x, pv.x), f2_pack(pv.y, pv.y), f2_pack(pv.z, pv.z),
                            f2_pack(pv.w, pv.w)};
    const int units = a.H / 8;
    uint64_t sq2 = 0;
    for (int u = tid; u < units; u += kColThreads) {
        uint32_t cs[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 r = ld_global_nc_v4(a.cur + (t * 4 + j) * a.H + 8LL * u);
            cs[j][0] = r.x; cs[j][1] = r.y; cs[j][2] = r.z; cs[j][3] = r.w;
        }
        uint32_t w[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            uint64_t acc = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) acc = fma2(p2[j], bf2_unpack(cs[j][p]), acc);
            w[p] = bf2_pack_rn(acc);
            const uint64_t lv = bf2_unpack(w[p]);
            sq2 = fma2(lv, lv, sq2);
        }
        li_s[u] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    uint16_t *row = a.layer_input + t * a.H;
    if (a.norm_w == nullptr) {
        for (int u = tid; u < units; u += kColThreads)
            *reinterpret_cast<uint4 *>(row + 8LL * u) = li_s[u];
        return;
    }
    float sq = f2_lo(sq2) + f2_hi(sq2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    if (lane == 0) red_s[warp] = sq;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kColThreads / 32; ++w) tot += red_s[w];
    const float rstd_li = rsqrtf(__fdiv_rn(tot, static_cast<float>(a.H)) + a.coef.norm_eps);
    for (int u = tid; u < units; u += kColThreads)
        *reinterpret_cast<uint4 *>(row + 8LL * u) =
            norm8(li_s[u], rstd_li, a.norm_w, a.nw_bf16, 8LL * u);
}

// ------------------------------------------------------------ reciprocal check
// Counts the bit patterns in [first, first + count) whose rcp_nr differs from
// the correctly rounded reciprocal; out[0] += count, out[1] = min(pattern).
__global__ void rcp_check_kernel(uint32_t first, unsigned long long count,
                                 unsigned long long *out) {
    unsigned long long bad = 0, first_bad = ~0ull;
    const unsigned long long stride = static_cast<unsigned long long>(gridDim.x) * blockDim.x;
    for (unsigned long long i = blockIdx.x * static_cast<unsigned long long>(blockDim.x) + threadIdx.x;
         i < count; i += stride) {
        const uint32_t b = first + static_cast<uint32_t>(i);
        const float x = __uint_as_float(b);
        if (__float_as_uint(rcp_nr(x)) != __float_as_uint(__frcp_rn(x))) {
            ++bad;
            if (b < first_bad) first_bad = b;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        bad += __shfl_xor_sync(0xffffffffu, bad, o);
        const unsigned long long f = __shfl_xor_sync(0xffffffffu, first_bad, o);
        first_bad = f < first_bad ? f : first_bad;
    }
    if ((threadIdx.x & 31) == 0 && bad) {
        atomicAdd(out, bad);
        atomicMin(out + 1, first_bad);
    }
}

// ------------------------------------------------------------ timeout probe
__global__ void unarmed_wait_kernel(unsigned int *status, unsigned long long timeout_ns) {
    __shared__ alignas(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_addr(&bar), 1);
        fence_mbar_init();
        // Nothing ever arrives: the bounded wait must run out and return.
        mbar_wait(smem_addr(&bar), 0, &abort_flag, timeout_ns, status, 99);
    }
}

}  // namespace

// The dynamic shared-memory opt-in of a kernel, per device: raised to the
// largest size asked for so far (H * 2 bytes for the collapse kernels, up to
// 128 KB), so that a run of calls pays for it once.
struct SmemOptIn {
    std::atomic<int> bytes[64];
};

template <typename K>
cudaError_t ensure_dynamic_smem(K kernel, SmemOptIn &opt, size_t smem) {
    if (smem <= 48 * 1024) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::atomic<int> &cur = opt.bytes[dev & 63];
    if (cur.load(std::memory_order_acquire) >= static_cast<int>(smem)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int prev = cur.load();
    while (prev < static_cast<int>(smem) && !cur.compare_exchange_weak(prev, static_cast<int>(smem))) {
    }
    return cudaSuccess;
}

SmemOptIn g_optin_split_k, g_optin_split_k_wide, g_optin_collapse, g_optin_collapse_wide;

unsigned int *device_status_word() {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    return static_cast<unsigned int *>(p);
}

cudaError_t launch_prepare_weight(const float *fn, int H, uint8_t *out, cudaStream_t s) {
    const long long total = static_cast<long long>(H / kChunk) * 4 * kWRows * 4;
    const int threads = 256;
    const long long blocks = (total + threads - 1) / threads;
    prepare_weight_kernel<<<static_cast<int>(blocks < 4096 ? blocks : 4096), threads, 0, s>>>(fn, H, out);
    return cudaGetLastError();
}

cudaError_t launch_post(const uint16_t *x, const uint16_t *res, const float *post,
                        const float *comb, uint16_t *out, long long T, int H, cudaStream_t s) {
    const long long total = T * (H / 8);
    const int threads = 256;
    long long blocks = (total + threads - 1) / threads;
    const long long cap = 152LL * 8 * 4;
    if (blocks > cap) blocks = cap;
    post_kernel<<<static_cast<int>(blocks), threads, 0, s>>>(x, res, post, comb, out, T, H);
    return cudaGetLastError();
}

namespace {
// A producer for the programmatic-dependent-launch test: the next kernel on
// the stream may launch at once; this one then waits delay_ns on the global
// timer (bounded by the host at 1 ms) and only then writes dst, so that a
// dependent that read dst before waiting for this grid would see old data.
__global__ void delayed_copy_kernel(const uint16_t *__restrict__ src, uint16_t *__restrict__ dst,
                                    long long n, uint32_t delay_ns) {
    griddep_launch_dependents();
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < delay_ns) nanosleep_ns(200);
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        dst[i] = src[i];
}
}  // namespace

cudaError_t launch_delayed_copy(const uint16_t *src, uint16_t *dst, long long n, uint32_t delay_ns,
                                cudaStream_t s) {
    // few blocks, so that the dependent's CTAs find free SMs while it waits
    delayed_copy_kernel<<<4, 256, 0, s>>>(src, dst, n, delay_ns);
    return cudaGetLastError();
}

cudaError_t launch_coefficients(const FinishArgs &a, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((a.T + kCoefTokens - 1) / kCoefTokens));
    cfg.blockDim = dim3(kCoefThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, coefficients_kernel, a);
}

cudaError_t launch_coefficients_split_k(const float *dot_mix, const float *sqrsum, int n_splits,
                                        const FinishArgs &a, cudaStream_t s) {
    const unsigned blocks = static_cast<unsigned>((a.T + kCoefTokens - 1) / kCoefTokens);
    coefficients_split_k_kernel<<<blocks, kCoefThreads, 0, s>>>(dot_mix, sqrsum, n_splits, a);
    return cudaGetLastError();
}

cudaError_t launch_pre_split_k(const float *dot_mix, const float *sqrsum, int n_splits,
                               const FinishArgs &a, cudaStream_t s, bool wide) {
    const size_t smem = static_cast<size_t>(a.H) * 2;
    if (wide) {
        if (cudaError_t e = ensure_dynamic_smem(pre_split_k_kernel<512>, g_optin_split_k_wide, smem))
            return e;
        pre_split_k_kernel<512><<<static_cast<unsigned>(a.T), 512, smem, s>>>(dot_mix, sqrsum,
                                                                              n_splits, a);
    } else {
        if (cudaError_t e = ensure_dynamic_smem(pre_split_k_kernel<128>, g_optin_split_k, smem))
            return e;
        pre_split_k_kernel<128><<<static_cast<unsigned>(a.T), 128, smem, s>>>(dot_mix, sqrsum,
                                                                              n_splits, a);
    }
    return cudaGetLastError();
}

cudaError_t launch_collapse_unshifted(const FinishArgs &a, cudaStream_t s, bool pdl, bool wide) {
    const size_t smem = static_cast<size_t>(a.H) * 2;
    auto kern = wide ? collapse_unshifted_kernel<512> : collapse_unshifted_kernel<128>;
    if (cudaError_t e = ensure_dynamic_smem(kern, wide ? g_optin_collapse_wide : g_optin_collapse, smem))
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.T));
    cfg.blockDim = dim3(wide ? 512 : 128);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

// Test hook: the coefficients of n tokens from reduced values v [n][25],
// formed once by coefficients_thread (one thread per token) and once by
// coefficients_16lanes (16 lanes per token), into two sets of outputs
// [n][24] (pre 4, post 4, comb 16). 32 tokens per block of 32 threads.
__global__ void coef_check_kernel(const float *__restrict__ v, CoefArgs c, int H, long long n,
                                  float *out_thread, float *out_lanes) {
    __shared__ float sb[32];
    __shared__ float vs[32 * kPartVals];
    const int lane = threadIdx.x;
    const long long t0 = static_cast<long long>(blockIdx.x) * 32;
    stage_coef_consts(c, sb, lane);
    for (int i = lane; i < 32 * kPartVals; i += 32)
        vs[i] = t0 * kPartVals + i < n * kPartVals ? v[t0 * kPartVals + i] : 1.f;
    __syncwarp();
    const long long t = t0 + lane;
    if (t < n)
        coefficients_thread(vs + lane * kPartVals, 1, sb, c, H, 0, out_thread + t * 24,
                            out_thread + t * 24 + 4, out_thread + t * 24 + 8);
    for (int j = 0; j < 32; j += 2) {
        const long long ta = t0 + j, tb = t0 + j + 1;
        // each half writes its own token's 24-float record (token index 0 in it)
        float *rec = out_lanes + (lane < 16 ? ta : tb) * 24;
        coefficients_16lanes(vs + j * kPartVals, vs + (j + 1) * kPartVals, 1, sb, c, H, 0, 0,
                             ta < n && lane < 16, tb < n && lane >= 16, rec, rec + 4, rec + 8);
    }
}

cudaError_t launch_coef_check(const float *v, const CoefArgs &c, int H, long long n,
                              float *out_thread, float *out_lanes, cudaStream_t s) {
    const long long blocks = (n + 31) / 32;
    coef_check_kernel<<<static_cast<unsigned>(blocks), 32, 0, s>>>(v, c, H, n, out_thread, out_lanes);
    return cudaGetLastError();
}

cudaError_t launch_rcp_check(uint32_t first, unsigned long long count, unsigned long long *out,
                             cudaStream_t s) {
    rcp_check_kernel<<<152 * 8, 256, 0, s>>>(first, count, out);
    return cudaGetLastError();
}

cudaError_t launch_unarmed_wait(unsigned int *status, unsigned long long timeout_ns,
                                cudaStream_t s) {
    unarmed_wait_kernel<<<1, 32, 0, s>>>(status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace mhc
